// kda_tc.cu -- bf16 tensor-core path of the chunkwise KDA forward (K = V = 128, C = 64).
//
// kda_intra_tc: one CTA (8 warps, two CTAs per SM) per (chunk, head), fed by TMA.
//   a1  q, k, v (bf16) and g (fp32) tiles by TMA; rows past the sequence end count as
//       q = k = v = 0, g = 0, beta = 0 (an identity step, Tokamax design doc 9.1.7).
//   a2  G = log2(e) * cumsum(g) within the chunk (Tokamax design doc 9.1.3), held in
//       registers: each thread owns 4 rows x 8 key channels; a two-level scan joins them.
//   a3  Aqk and L by tcgen05 MMAs ("KDA Doesn't Care About the Future", "The rebasing
//       trick", "Sixteen keys, sixty-four queries"): for the 16-row block b of queries
//       the ratio 2^{G_i - G_j} is split at the block's first row G_{16b} into a query
//       factor 2^{G_i - G_{16b}} <= 1 and a key factor 2^{G_{16b} - G_j} <= 2^108 (gate
//       bound -5), so both stay finite and the reference depends on no later token.
//       Keys form the MMA's M side (R_b: 64 key rows rebased for query block b, two
//       blocks stacked to M = 128) and the block's 16 scaled query rows and 16
//       beta-scaled key rows the N side (N = 64 for two blocks); two rounds share one
//       operand buffer.
//   a4  (I + L)^{-1} by blocked forward substitution in fp32 (16 x 16 diagonal blocks,
//       then three levels of block products); [W | U] = (I + L)^{-1} [D_beta K+ | D_beta V]
//       by one M 128 x N 256 x K 64 MMA whose B operand is the k and v tiles rescaled in
//       place (token-major, read as an MN-major operand) (Tokamax design doc Eq. (6)-(7)).
//       Also K_bar = k 2^{G_C - G} and the gated, scaled query (9.1.5).
//   The results form one record per (chunk, head) (TcRecord), written as tensor-core
//   operand images.  Every product is computed from a thread's own rows and stored as
//   16-byte chunks; nothing is transposed through scalar stores.
//
// kda_h_o_tc: one CTA (4 warps) per (sequence, head, 64-column slice of V): the ordered
//   chunk recurrence (Eq. (8)) fused with the output (Eq. (9)).  Records are double-
//   buffered by bulk copies; the state slice lives in fp32 registers (thread d owns key
//   row d) and is written as a bf16 operand tile each chunk.  Per chunk:
//     MMA1  D1 = [W ; Qg] S                              (M 128, N 64, K 128)
//     ep1   V_new = U - W S                               (D1 rows 0-63)
//     MMA3  D3 = K_bar^T V_new                            (M 128 keys, N 64, K 64)
//     MMA2  D1 += [Qg rows ; Aqk] V_new                   (rows 64-127: O = Qg S + Aqk V_new)
//     ep2   S = Diag(gamma^C) S + D3.
//   MMA3 is issued before MMA2 so that the state update, the only step the next chunk
//   waits for, does not wait for the output product; D1 alternates between two TMEM
//   buffers and each chunk's output rows are read while the next chunk's MMA1 runs.
//   A fifth warp issues the record copies and every MMA; it meets the epilogue warps at
//   named barriers, so no epilogue thread is held up by MMA issue.  Records run through
//   a ring of three stages so each copy has two chunk steps to arrive.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {

namespace {

using namespace sm100;

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 p = __bfloat1622float2(h[i]);
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// 16-byte shared-memory accesses at a byte offset from the CTA's aligned dynamic
// shared base.  Plain C++ accesses, so the compiler may overlap independent ones;
// every synchronisation point (fences, barriers, mbarrier and tcgen05 operations) is
// an asm statement with a memory clobber, which keeps them ordered around it.
__device__ __forceinline__ void sts128(uint8_t* base, uint32_t off, uint4 v) {
    *reinterpret_cast<uint4*>(base + off) = v;
}
__device__ __forceinline__ uint4 lds128(const uint8_t* base, uint32_t off) {
    return *reinterpret_cast<const uint4*>(base + off);
}

// 8 consecutive floats of shared memory (32-byte aligned), read as two 16-byte halves
// in an order that spreads a warp's lanes over all banks when consecutive lanes read
// consecutive 32-byte groups.
__device__ __forceinline__ void ld8f(const float* p, int swap, float (&f)[8]) {
    const float4* q = reinterpret_cast<const float4*>(p);
    const float4 a = q[swap], b = q[swap ^ 1];
    const float4 lo = swap ? b : a, hi = swap ? a : b;
    f[0] = lo.x; f[1] = lo.y; f[2] = lo.z; f[3] = lo.w;
    f[4] = hi.x; f[5] = hi.y; f[6] = hi.z; f[7] = hi.w;
}

__device__ __forceinline__ void st8f(float* p, const float (&f)[8]) {
    float4* q = reinterpret_cast<float4*>(p);
    q[0] = make_float4(f[0], f[1], f[2], f[3]);
    q[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// index of the block pair (b, b'), b' < b, in the table of 2^{G_16b - G_16b'}
__device__ __forceinline__ int pair_index(int b, int bp) { return b * (b - 1) / 2 + bp; }

// ---------------------------------------------------------------------------
// intra-chunk kernel
// ---------------------------------------------------------------------------

constexpr int kIntraThreads = 256;

struct IntraMap {
    // relation B operand: group p (query blocks 2p, 2p+1), key panel P at (2p+P)*8K,
    // [64 rows][64]: rows 0-31 the chunk's q rows 32p..32p+31 (TMA), rescaled in place
    // to scale*q_i*2^{G_i-G_16b}; rows 32-63 beta_i*k_i*2^{G_i-G_16b} of the same rows
    static constexpr uint32_t RB = 0;
    static constexpr uint32_t KT = 32768;   // k (TMA), rescaled in place to D_beta K+
    static constexpr uint32_t VT = 49152;   // v (TMA), rescaled in place to D_beta V
    static constexpr uint32_t RA = 65536;   // g tile (TMA); then relation A: 2 panels [128][64]
    static constexpr uint32_t MISC = 98304;
    static constexpr uint32_t REFS = MISC;         // [5][128] G rows 0, 16, 32, 48, 63
    static constexpr uint32_t FAC = MISC + 2560;   // scan totals [16][128]; then factors
    static constexpr uint32_t BETA = FAC + 8192;   // [64]
    static constexpr uint32_t END = BETA + 256;
    // factor tables inside FAC after the scan: P0 [4][128] = 2^{G_16b},
    // X [6][128] = 2^{G_16b - G_16b'} (b' < b), C [4][128] = 2^{G_63 - G_16b}
    static constexpr uint32_t P0 = FAC, X = FAC + 2048, CF = FAC + 5120;
    // reuse after the relation MMAs
    static constexpr uint32_t AF = RA, LF = RA + 16384;  // Aqk, L fp32 [64][64]
    static constexpr uint32_t IF = RB;                   // (I + L)^{-1} fp32 [64][64]
    static constexpr uint32_t AIA = RB + 16384;          // (I + L)^{-1} bf16 [128][64]
    static constexpr uint32_t WST = KT, UST = VT;        // after the W/U MMA
};
constexpr size_t kIntraSmem = IntraMap::END + 1024;  // + alignment slack

__global__ void __launch_bounds__(kIntraThreads, 2)
kda_intra_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
             const float* __restrict__ beta, float scale, int H, const int4* __restrict__ chunk_tab,
             const int* __restrict__ count, long long max_chunks, uint8_t* __restrict__ records,
             int* __restrict__ status) {
    using M = IntraMap;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar_tma, bar_rel, bar_wu;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    // chunks run from the last to the first so that the records of early chunks, which
    // the recurrence reads first, are the most recently written (still in L2)
    const long long blk = blockIdx.x;
    const int h = (int)(blk % H);
    const long long c = max_chunks - 1 - blk / H;
    if (c >= *count) return;
    const int4 ent = chunk_tab[c];
    const int t0 = ent.y, len = ent.z;
    uint8_t* rec = records + ((size_t)c * H + h) * TcRecord::bytes;

    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sb = smem_u32(sm);
    float* refs = reinterpret_cast<float*>(sm + M::REFS);
    float* tot = reinterpret_cast<float*>(sm + M::FAC);
    float* P0 = reinterpret_cast<float*>(sm + M::P0);
    float* X = reinterpret_cast<float*>(sm + M::X);
    float* CF = reinterpret_cast<float*>(sm + M::CF);
    float* betas = reinterpret_cast<float*>(sm + M::BETA);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dc = tid & 15, rg = tid >> 4;  // 8 key channels 8dc.., rows 4rg..4rg+3
    const int P = dc >> 3, cc = dc & 7;      // key panel, chunk within the panel row
    const int swap = (dc >> 2) & 1;

    if (warp == 0) tmem_alloc(&tmem_base, 256);
    if (tid == 0) {
        s_abort = 0;
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_rel, 1);
        mbar_init(&bar_wu, 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    volatile int* abort_flag = &s_abort;

    // a1: tiles by TMA (rows past the end of the tensor read as zero)
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_tma, 3 * 16384 + 32768);
        for (int p = 0; p < 2; ++p)
            for (int pp = 0; pp < 2; ++pp)
                tma_load_2d(sm + M::RB + (p * 2 + pp) * 8192, &tm_q, h * 128 + 64 * pp, t0 + 32 * p,
                            &bar_tma);
        for (int pp = 0; pp < 2; ++pp) {
            tma_load_2d(sm + M::KT + pp * 8192, &tm_k, h * 128 + 64 * pp, t0, &bar_tma);
            tma_load_2d(sm + M::VT + pp * 8192, &tm_v, h * 128 + 64 * pp, t0, &bar_tma);
        }
        tma_load_2d(sm + M::RA, &tm_g, h * 128, t0, &bar_tma);
    }
    if (tid < 64) betas[tid] = tid < len ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
    mbar_wait_abortable(&bar_tma, 0, status, abort_flag);
    __syncthreads();
    if (*abort_flag) goto teardown;

    {
        // a2: cumsum of g over the chunk in registers
        float G[4][8];
        const float* gt = reinterpret_cast<const float*>(sm + M::RA);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * rg + r;
            ld8f(gt + i * 128 + dc * 8, swap, G[r]);
            if (i >= len) {
#pragma unroll
                for (int m = 0; m < 8; ++m) G[r][m] = 0.f;
            }
        }
#pragma unroll
        for (int r = 1; r < 4; ++r)
#pragma unroll
            for (int m = 0; m < 8; ++m) G[r][m] += G[r - 1][m];
        st8f(tot + rg * 128 + dc * 8, G[3]);
        __syncthreads();
        // exclusive scan of the 16 row-group totals down each key channel (one thread per
        // channel), in place
        if (tid < 128) {
            float run = 0.f;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float t = tot[q * 128 + tid];
                tot[q * 128 + tid] = run;
                run += t;
            }
        }
        __syncthreads();
        {
            float pre[8];
            ld8f(tot + rg * 128 + dc * 8, swap, pre);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int m = 0; m < 8; ++m) G[r][m] = (G[r][m] + pre[m]) * kLog2e;
        }
        if ((rg & 3) == 0) st8f(refs + (rg >> 2) * 128 + dc * 8, G[0]);
        if (rg == 15) st8f(refs + 4 * 128 + dc * 8, G[3]);
        __syncthreads();

        // block factors (overwrite the scan totals) and gamma^C = 2^{G_63}: threads 0-127
        // take P0 and gamma of channel d, threads 128-255 the X and C tables of channel d
        {
            const int d = tid & 127;
            float gr[5];
#pragma unroll
            for (int b = 0; b < 5; ++b) gr[b] = refs[b * 128 + d];
            if (tid < 128) {
#pragma unroll
                for (int b = 0; b < 4; ++b) P0[b * 128 + d] = exp2f(gr[b]);
                reinterpret_cast<float*>(rec + TcRecord::gamma)[d] = exp2f(gr[4]);
            } else {
#pragma unroll
                for (int b = 1; b < 4; ++b)
#pragma unroll
                    for (int bp = 0; bp < b; ++bp)
                        X[pair_index(b, bp) * 128 + d] = exp2f(gr[b] - gr[bp]);
#pragma unroll
                for (int b = 0; b < 4; ++b) CF[b * 128 + d] = exp2f(gr[4] - gr[b]);
            }
        }
        __syncthreads();

        // a3/a4 operands, row by row (the 4 rows of a thread lie in one 16-row block b)
        float R[4][8];  // key factor rows k_j 2^{G_16b(j) - G_j}, kept for the second round
        const int b = rg >> 2;
        float gref[8], p0[8], cf[8], x10[8];
        ld8f(refs + b * 128 + dc * 8, swap, gref);
        ld8f(P0 + b * 128 + dc * 8, swap, p0);
        ld8f(CF + b * 128 + dc * 8, swap, cf);
        if (b == 0) ld8f(X + pair_index(1, 0) * 128 + dc * 8, swap, x10);
        // the shared-memory loads of two rows are issued before their first store
        uint4 qr[2], kr[2], vr[2];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if ((r & 1) == 0) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int i = 4 * rg + r + rr;
                    qr[rr] = lds128(sm, M::RB + ((i >> 5) * 2 + P) * 8192 + sw128_chunk(i & 31, cc));
                    kr[rr] = lds128(sm, M::KT + P * 8192 + sw128_chunk(i, cc));
                    vr[rr] = lds128(sm, M::VT + P * 8192 + sw128_chunk(i, cc));
                }
            }
            const int i = 4 * rg + r, grp = i >> 5, ii = i & 31;
            const float inb = i < len ? 1.f : 0.f;
            const float bi = betas[i];
            float e[8], ei[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                e[m] = exp2f(G[r][m] - gref[m]);
                ei[m] = exp2f(gref[m] - G[r][m]);
            }
            // query: relation B row (in place) and the gated query of the record
            {
                const uint32_t a = M::RB + (grp * 2 + P) * 8192 + sw128_chunk(ii, cc);
                float qv[8], qs[8], qg[8];
                unpack8(qr[r & 1], qv);
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    qs[m] = scale * qv[m] * inb * e[m];
                    qg[m] = qs[m] * p0[m];
                }
                sts128(sm, a, pack8(qs));
                *reinterpret_cast<uint4*>(rec + TcRecord::wq + P * 16384 + 8192 +
                                          sw128_chunk(i, cc)) = pack8(qg);
            }
            // key: relation B row, D_beta K+ (in place), key factor rows, K_bar
            {
                const uint32_t a = M::KT + P * 8192 + sw128_chunk(i, cc);
                float kv[8], kp[8], kpl[8], kb[8];
                unpack8(kr[r & 1], kv);
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    kv[m] *= inb;
                    kp[m] = bi * kv[m] * e[m];
                    kpl[m] = kp[m] * p0[m];
                    R[r][m] = kv[m] * ei[m];
                    kb[m] = R[r][m] * cf[m];
                }
                sts128(sm, M::RB + (grp * 2 + P) * 8192 + sw128_chunk(32 + ii, cc), pack8(kp));
                sts128(sm, a, pack8(kpl));
                *reinterpret_cast<uint4*>(rec + TcRecord::kbar + P * 8192 + sw128_chunk(i, cc)) =
                    pack8(kb);
                // round 0 of relation A: R_0 (rows 0-63) and R_1 (rows 64-127)
                const uint32_t ra = M::RA + P * 16384;
                if (b == 0) {
                    float t[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) t[m] = R[r][m] * x10[m];
                    sts128(sm, ra + sw128_chunk(i, cc), pack8(R[r]));
                    sts128(sm, ra + sw128_chunk(64 + i, cc), pack8(t));
                } else if (b == 1) {
                    sts128(sm, ra + sw128_chunk(64 + i, cc), pack8(R[r]));
                }
            }
            // value: D_beta V in place
            {
                const uint32_t a = M::VT + P * 8192 + sw128_chunk(i, cc);
                float vv[8];
                unpack8(vr[r & 1], vv);
#pragma unroll
                for (int m = 0; m < 8; ++m) vv[m] *= bi * inb;
                sts128(sm, a, pack8(vv));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // relation round 0: query blocks 0 and 1 -> TMEM columns 0-63
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, 64);
            for (int ks = 0; ks < 8; ++ks) {
                const int pp = ks >> 2, kk = ks & 3;
                mma_bf16(tmem, desc_sw128(sb + M::RA + pp * 16384 + kk * 32),
                         desc_sw128(sb + M::RB + pp * 8192 + kk * 32), idesc, ks > 0 ? 1u : 0u);
            }
            mma_commit(&bar_rel);
        }
        mbar_wait_abortable(&bar_rel, 0, status, abort_flag);
        tc_fence_after();
        // round 1 of relation A: R_2 (rows 0-63) and R_3 (rows 64-127), same buffer
        {
            float x2[8], x3[8];
            if (b < 2) ld8f(X + pair_index(2, b) * 128 + dc * 8, swap, x2);
            if (b < 3) ld8f(X + pair_index(3, b) * 128 + dc * 8, swap, x3);
            const uint32_t ra = M::RA + P * 16384;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = 4 * rg + r;
                float t[8];
                if (b < 2) {
#pragma unroll
                    for (int m = 0; m < 8; ++m) t[m] = R[r][m] * x2[m];
                    sts128(sm, ra + sw128_chunk(i, cc), pack8(t));
                } else if (b == 2) {
                    sts128(sm, ra + sw128_chunk(i, cc), pack8(R[r]));
                }
                if (b < 3) {
#pragma unroll
                    for (int m = 0; m < 8; ++m) t[m] = R[r][m] * x3[m];
                    sts128(sm, ra + sw128_chunk(64 + i, cc), pack8(t));
                } else {
                    sts128(sm, ra + sw128_chunk(64 + i, cc), pack8(R[r]));
                }
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) goto teardown;
    if (tid == 0) {  // relation round 1: query blocks 2 and 3 -> TMEM columns 64-127
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(128, 64);
        for (int ks = 0; ks < 8; ++ks) {
            const int pp = ks >> 2, kk = ks & 3;
            mma_bf16(tmem + 64, desc_sw128(sb + M::RA + pp * 16384 + kk * 32),
                     desc_sw128(sb + M::RB + (2 + pp) * 8192 + kk * 32), idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(&bar_rel);
    }
    mbar_wait_abortable(&bar_rel, 1, status, abort_flag);
    tc_fence_after();
    __syncthreads();
    if (*abort_flag) goto teardown;

    {
        // relation epilogue: TMEM lane L = key j (L < 64: rebased for the first block of
        // the round, L >= 64: for the second); columns 0-31 the round's 32 query rows,
        // 32-63 its 32 beta-scaled key rows
        float* AF = reinterpret_cast<float*>(sm + M::AF);
        float* LF = reinterpret_cast<float*>(sm + M::LF);
        float* IF = reinterpret_cast<float*>(sm + M::IF);
        if (warp < 4) {
            const int L = warp * 32 + lane, j = L & 63, hi = L >> 6;
            for (int ro = 0; ro < 2; ++ro) {
                // this lane's block b = 2ro + hi: query columns 16hi.., key columns 32+16hi..
                float vq[16], vk[16];
                tmem_ld16(tmem_addr(tmem, warp, 64 * ro + 16 * hi), vq);
                tmem_ld16(tmem_addr(tmem, warp, 64 * ro + 32 + 16 * hi), vk);
                const int b = 2 * ro + hi;
#pragma unroll
                for (int ci = 0; ci < 16; ++ci) {
                    const int i = 16 * b + ci;
                    AF[i * 64 + j] = j <= i ? vq[ci] : 0.f;
                    LF[i * 64 + j] = j < i ? vk[ci] : 0.f;
                }
            }
        } else {
            for (int idx = tid - 128; idx < 4096; idx += 128) IF[idx] = 0.f;
        }
        tc_fence_before();
        __syncthreads();

        // Aqk (bf16) to the record
        for (int u = tid; u < 512; u += kIntraThreads) {
            const int i = u >> 3, jc = u & 7;
            float a[8];
            ld8f(AF + i * 64 + jc * 8, 0, a);
            *reinterpret_cast<uint4*>(rec + TcRecord::aqk + sw128_chunk(i, jc)) = pack8(a);
        }
        __syncthreads();  // AF is reused as scratch below
        // a4: (I + L)^{-1} in fp32 by blocks of 16 (Tokamax design doc 4.1.4 uses the same
        // finite expansion with MXU products).  With D the inverses of the diagonal
        // blocks and J = D F (F the blocks below the diagonal, J strictly block-lower, so
        // J^4 = 0): (I + L)^{-1} = (I + J)^{-1} D = (I - J + J^2 - J^3) D.
        // Stage 1, D: right-looking forward substitution, one column per thread
        //   (after x_m is final, every later row subtracts L[r][m] x_m).
        float* JS = reinterpret_cast<float*>(sm + M::AF);  // J [6][16][16] | J^2 [3] | J^3 [1]
        if (tid < 64) {
            const int bb = tid >> 4, cidx = tid & 15, o = 16 * bb;
            float acc[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) acc[r] = r == cidx ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < 15; ++m)
#pragma unroll
                for (int r = m + 1; r < 16; ++r)
                    acc[r] = fmaf(-LF[(o + r) * 64 + o + m], acc[m], acc[r]);
#pragma unroll
            for (int r = 0; r < 16; ++r) IF[(o + r) * 64 + o + cidx] = acc[r];
        }
        __syncthreads();
        // block (i, j) below the diagonal: index in J, in pair order (1,0)(2,0)(2,1)(3,0)(3,1)(3,2)
        const int r16 = (tid >> 4) & 15, c16 = tid & 15;
        // Stage 2: J_ij = D_i L_ij, six blocks, six elements per thread
        {
            float acc[6];
#pragma unroll
            for (int pi = 0; pi < 6; ++pi) {
                const int bi = pi < 1 ? 1 : (pi < 3 ? 2 : 3), bj = pi - pair_index(bi, 0);
                float a = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    a = fmaf(IF[(16 * bi + r16) * 64 + 16 * bi + m], LF[(16 * bi + m) * 64 + 16 * bj + c16], a);
                acc[pi] = a;
            }
#pragma unroll
            for (int pi = 0; pi < 6; ++pi) JS[pi * 256 + r16 * 16 + c16] = acc[pi];
        }
        __syncthreads();
        // Stage 3: J^2 blocks (2,0) = J21 J10, (3,1) = J32 J21, (3,0) = J31 J10 + J32 J20
        {
            const float* J = JS;
            auto jb = [&](int pi, int r, int c) { return J[pi * 256 + r * 16 + c]; };
            float a20 = 0.f, a31 = 0.f, a30 = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                a20 = fmaf(jb(2, r16, m), jb(0, m, c16), a20);
                a31 = fmaf(jb(5, r16, m), jb(2, m, c16), a31);
                a30 = fmaf(jb(4, r16, m), jb(0, m, c16), a30);
                a30 = fmaf(jb(5, r16, m), jb(1, m, c16), a30);
            }
            JS[1536 + 0 * 256 + r16 * 16 + c16] = a20;
            JS[1536 + 1 * 256 + r16 * 16 + c16] = a31;
            JS[1536 + 2 * 256 + r16 * 16 + c16] = a30;
        }
        __syncthreads();
        // Stage 4: J^3 block (3,0) = J32 (J^2)20
        {
            float a = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                a = fmaf(JS[5 * 256 + r16 * 16 + m], JS[1536 + m * 16 + c16], a);
            JS[2304 + r16 * 16 + c16] = a;
        }
        __syncthreads();
        // Stage 5: Ainv_ij = (-J + J^2 - J^3)_ij D_j for the six blocks below the diagonal
        {
            float acc[6];
#pragma unroll
            for (int pi = 0; pi < 6; ++pi) {
                const int bi = pi < 1 ? 1 : (pi < 3 ? 2 : 3), bj = pi - pair_index(bi, 0);
                const int k2 = (bi == 2 && bj == 0) ? 0 : (bi == 3 && bj == 1) ? 1 : (bi == 3 && bj == 0) ? 2 : -1;
                float a = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    float mv = -JS[pi * 256 + r16 * 16 + m];
                    if (k2 >= 0) mv += JS[1536 + k2 * 256 + r16 * 16 + m];
                    if (pi == 3) mv -= JS[2304 + r16 * 16 + m];
                    a = fmaf(mv, IF[(16 * bj + m) * 64 + 16 * bj + c16], a);
                }
                acc[pi] = a;
            }
#pragma unroll
            for (int pi = 0; pi < 6; ++pi) {
                const int bi = pi < 1 ? 1 : (pi < 3 ? 2 : 3), bj = pi - pair_index(bi, 0);
                IF[(16 * bi + r16) * 64 + 16 * bj + c16] = acc[pi];
            }
        }
        __syncthreads();
        // (I + L)^{-1} as the bf16 A operand of the W/U product (rows 64-127 unused)
        for (int u = tid; u < 512; u += kIntraThreads) {
            const int r = u >> 3, jc = u & 7;
            float a[8];
            ld8f(IF + r * 64 + jc * 8, 0, a);
            sts128(sm, M::AIA + sw128_chunk(r, jc), pack8(a));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    }

    // [W | U] = (I+L)^{-1} [D_beta K+ | D_beta V]: M 128 (tokens, 64 used), N 256, K 64;
    // B is the token-major k|v tiles (4 atoms of 64 columns, 8 KB apart)
    if (tid == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(128, 256, false, true);
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem, desc_sw128(sb + M::AIA + kk * 32),
                     desc_sw128_mn(sb + M::KT + kk * 2048, 8192, 1024), idesc, kk > 0 ? 1u : 0u);
        mma_commit(&bar_wu);
    }
    mbar_wait_abortable(&bar_wu, 0, status, abort_flag);
    tc_fence_after();
    __syncthreads();
    if (*abort_flag) goto teardown;

    // W rows (warps 0,1) and U rows (warps 4,5) into staging images of the record tiles
    if (warp == 0 || warp == 1 || warp == 4 || warp == 5) {
        const int r = (warp & 1) * 32 + lane;
        const uint32_t dst = warp < 4 ? M::WST : M::UST;
        const uint32_t col0 = warp < 4 ? 0 : 128;
        for (int cb = 0; cb < 4; ++cb) {
            float v[32];
            tmem_ld32(tmem_addr(tmem, warp, col0 + 32 * cb), v);
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                float f[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) f[m] = v[qd * 8 + m];
                sts128(sm, dst + (cb >> 1) * 8192 + sw128_chunk(r, (cb & 1) * 4 + qd), pack8(f));
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        bulk_store(rec + TcRecord::wq, sm + M::WST, 8192);
        bulk_store(rec + TcRecord::wq + 16384, sm + M::WST + 8192, 8192);
        bulk_store(rec + TcRecord::u, sm + M::UST, 16384);
        bulk_commit();
        // only the shared-memory source must outlive the copies; the stores themselves
        // are complete for any later kernel on the stream
        bulk_wait_read_all();
    }

teardown:
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// recurrence + output kernel
// ---------------------------------------------------------------------------

constexpr int kVT = 64;                   // value columns per CTA
constexpr int kHoThreads = 160;           // 4 epilogue warps (thread d <-> TMEM lane d <->
                                          // key row d of S) + 1 issuer warp
constexpr uint32_t kStageBytes = 66560;   // wq|aqk|kbar 56K | U panel 8K | gamma 512 (65 KB)
constexpr uint32_t kStTx = 57344 + 8192 + 512;
constexpr int kStages = 3;                // record ring depth: copies run 2 chunk steps ahead
// named barriers between the epilogue warps and the issuer warp
constexpr uint32_t kBarVnew = 1;          // warps 0-1 -> issuer: V_new tile written
constexpr uint32_t kBarState = 2;         // warps 0-3 -> issuer: S tile written, D1/D3 read

struct HoMap {
    static constexpr uint32_t ST = kStages * kStageBytes;  // S tile bf16 [128 keys][64 values]
    static constexpr uint32_t VN = ST + 16384;              // V_new tile bf16 [64 tokens][64 values]
    static constexpr uint32_t END = VN + 8192;
    // inside a stage
    static constexpr uint32_t WQ = 0, AQK = 32768, KB = 40960, U = 57344, GAM = 65536;
};
constexpr size_t kHoSmem = HoMap::END + 1024;

__global__ void __launch_bounds__(kHoThreads, 1)
kda_h_o_tc(const uint8_t* __restrict__ records, const int4* __restrict__ chunk_tab,
           const int2* __restrict__ seq_tab, long long max_chunks, const float* __restrict__ s0,
           __nv_bfloat16* __restrict__ o, float* __restrict__ sN, int H,
           int* __restrict__ status) {
    using M = HoMap;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[kStages], bar_m1, bar_m3, bar_m2;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    const int slice = blockIdx.x & 1;
    const int h = (blockIdx.x >> 1) % H;
    const int n = (blockIdx.x >> 1) / H;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int2 sq = seq_tab[n];
    const long long first = sq.x;
    int nch = sq.y;
    if (first + nch > max_chunks) {  // inconsistent cu_seqlens: stop rather than overrun
        if (tid == 0) atomicCAS(status, 0, (int)KDA_ERR_INVALID_ARG);
        nch = (int)(max_chunks > first ? max_chunks - first : 0);
    }

    if (warp == 0) tmem_alloc(&tmem_base, 256);
    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
        mbar_init(&bar_m1, 1);
        mbar_init(&bar_m3, 1);
        mbar_init(&bar_m2, 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // D1 (two buffers, alternating by chunk): [W ; Qg] S, then rows 64-127 += Aqk V_new
    // (the output); D3: K_bar^T V_new (the state update)
    const uint32_t tmem = tmem_base, D3 = tmem + 128;
    volatile int* abort_flag = &s_abort;
    const size_t st_off = ((size_t)n * H + h) * 128 * 128 + slice * kVT;

    if (warp == 4) {
        // ---- issuer warp: record copies and every MMA (lane 0 issues).  The whole warp
        // runs the loop so that its named-barrier syncs are warp-uniform; every exit
        // decision is made uniform with a warp vote. ----
        auto load = [&](int ci) {  // record of chunk ci into stage ci % kStages (lane 0)
            const int sg = ci % kStages;
            const uint8_t* rec = records + ((size_t)(first + ci) * H + h) * TcRecord::bytes;
            uint8_t* st = sm + sg * kStageBytes;
            mbar_arrive_expect_tx(&full[sg], kStTx);
            bulk_load(st + M::WQ, rec + TcRecord::wq, 57344, &full[sg]);  // wq, aqk, kbar
            bulk_load(st + M::U, rec + TcRecord::u + slice * 8192, 8192, &full[sg]);
            bulk_load(st + M::GAM, rec + TcRecord::gamma, 512, &full[sg]);
        };
        if (lane == 0)
            for (int ci = 0; ci < kStages && ci < nch; ++ci) load(ci);
        __syncwarp();
        const uint32_t idesc_a = idesc_bf16(128, kVT, false, true);  // B MN-major
        const uint32_t idesc_t = idesc_bf16(128, kVT, true, true);   // A MN-major too
        const uint64_t dS = desc_sw128_mn(sb + M::ST, 16384, 1024);
        const uint64_t dVN = desc_sw128_mn(sb + M::VN, 8192, 1024);
        for (int ci = 0; ci < nch; ++ci) {
            const int sg = ci % kStages;
            const uint32_t stb = sb + sg * kStageBytes;
            const uint32_t D1 = tmem + 64 * (ci & 1);
            bool ok = mbar_wait_abortable(&full[sg], (ci / kStages) & 1, status, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            named_bar_sync(kBarState, 160);  // S_ci written, D1/D3 of earlier chunks read
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            if (lane == 0) {
                tc_fence_after();
                // MMA1: D1 = [W ; Qg] S   (K = 128 keys over two panels)
                const uint64_t dWQ = desc_sw128(stb + M::WQ);
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16(D1, dWQ + (uint64_t)(((ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                             dS + (uint64_t)((ks * 2048) >> 4), idesc_a, ks > 0 ? 1u : 0u);
                mma_commit(&bar_m1);
            }
            __syncwarp();
            // refill the stage chunk ci-1 used: its MMA2 precedes this MMA1 on the pipe
            if (ci >= 1 && ci - 1 + kStages < nch) {
                ok = mbar_wait_abortable(&bar_m2, (ci - 1) & 1, status, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) break;
                if (lane == 0) load(ci - 1 + kStages);
                __syncwarp();
            }
            named_bar_sync(kBarVnew, 96);  // V_new tile written by warps 0-1
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            if (lane == 0) {
                tc_fence_after();
                // MMA3 first (it feeds the state): D3 = K_bar^T V_new (K_bar token-major:
                // MN-major A, 2 atoms 8 KB apart)
                const uint64_t dKB = desc_sw128_mn(stb + M::KB, 8192, 1024);
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(D3, dKB + (uint64_t)((kk * 2048) >> 4),
                             dVN + (uint64_t)((kk * 2048) >> 4), idesc_t, kk > 0 ? 1u : 0u);
                mma_commit(&bar_m3);
                // MMA2: D1 += [Qg panel-1 rows ; Aqk] V_new  (only rows 64-127 are used)
                const uint64_t dQA = desc_sw128(stb + M::WQ + 16384 + 8192);
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(D1, dQA + (uint64_t)((kk * 32) >> 4),
                             dVN + (uint64_t)((kk * 2048) >> 4), idesc_a, 1u);
                mma_commit(&bar_m2);
            }
            __syncwarp();
        }
    } else {
        // ---- epilogue warps: thread d owns row d of the state slice, fp32 ----
        const int d = tid;
        float S[kVT];
        {
            const float4* src = reinterpret_cast<const float4*>(s0 + st_off + (size_t)d * 128);
#pragma unroll
            for (int x = 0; x < kVT / 4; ++x) {
                const float4 f = s0 ? src[x] : make_float4(0.f, 0.f, 0.f, 0.f);
                S[4 * x] = f.x;
                S[4 * x + 1] = f.y;
                S[4 * x + 2] = f.z;
                S[4 * x + 3] = f.w;
            }
        }
        // S tile: key-major [128][64] bf16 (MN-major B operand), row d = 8 chunks of 16 B
        auto write_state = [&]() {
#pragma unroll
            for (int qd = 0; qd < 8; ++qd) {
                float f[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) f[m] = S[qd * 8 + m];
                sts128(sm, M::ST + sw128_chunk(d, qd), pack8(f));
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_arrive(kBarState, 160);
        };
        // output of chunk ci (warps 2 and 3, token = lane index - 64)
        auto emit_output = [&](int ci) {
            if (!__all_sync(0xffffffffu, mbar_wait_abortable(&bar_m2, ci & 1, status, abort_flag)))
                return;
            tc_fence_after();
            float ov[64];
            const uint32_t D1 = tmem + 64 * (ci & 1);
            tmem_ld32(tmem_addr(D1, warp, 0), *reinterpret_cast<float(*)[32]>(ov));
            tmem_ld32(tmem_addr(D1, warp, 32), *reinterpret_cast<float(*)[32]>(ov + 32));
            const int4 ent = chunk_tab[first + ci];
            const int i = d - 64;
            if (i < ent.z) {
                uint4* dst = reinterpret_cast<uint4*>(o + ((size_t)(ent.y + i) * H + h) * 128 +
                                                      slice * kVT);
#pragma unroll
                for (int qd = 0; qd < 8; ++qd) {
                    float f[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) f[m] = ov[qd * 8 + m];
                    dst[qd] = pack8(f);
                }
            }
        };
        write_state();
        for (int ci = 0; ci < nch; ++ci) {
            const int sg = ci % kStages;
            const uint32_t stb = sb + sg * kStageBytes;
            const uint8_t* st = sm + sg * kStageBytes;
            const uint32_t D1 = tmem + 64 * (ci & 1);
            if (!__all_sync(0xffffffffu,
                            mbar_wait_abortable(&full[sg], (ci / kStages) & 1, status, abort_flag)))
                break;
            // the previous chunk's output is read while MMA1 runs
            if (warp >= 2 && ci > 0) emit_output(ci - 1);
            if (!__all_sync(0xffffffffu, mbar_wait_abortable(&bar_m1, ci & 1, status, abort_flag)))
                break;
            tc_fence_after();
            if (warp < 2) {
                // ep1: V_new[i] = U[i] - (W S)[i], token i = TMEM lane = d
                float ws[64];
                tmem_ld32(tmem_addr(D1, warp, 0), *reinterpret_cast<float(*)[32]>(ws));
                tmem_ld32(tmem_addr(D1, warp, 32), *reinterpret_cast<float(*)[32]>(ws + 32));
                const uint32_t stb_off = (uint32_t)sg * kStageBytes;
                uint4 ur[8];
#pragma unroll
                for (int qd = 0; qd < 8; ++qd) ur[qd] = lds128(sm, stb_off + M::U + sw128_chunk(d, qd));
#pragma unroll
                for (int qd = 0; qd < 8; ++qd) {
                    float uf[8], vn[8];
                    unpack8(ur[qd], uf);
#pragma unroll
                    for (int m = 0; m < 8; ++m) vn[m] = uf[m] - ws[qd * 8 + m];
                    sts128(sm, M::VN + sw128_chunk(d, qd), pack8(vn));
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_arrive(kBarVnew, 96);
            }
            if (!__all_sync(0xffffffffu, mbar_wait_abortable(&bar_m3, ci & 1, status, abort_flag)))
                break;
            tc_fence_after();
            {
                const float gam = reinterpret_cast<const float*>(st + M::GAM)[d];
                float upd[32];
                tmem_ld32(tmem_addr(D3, warp, 0), upd);
#pragma unroll
                for (int x = 0; x < 32; ++x) S[x] = fmaf(gam, S[x], upd[x]);
                tmem_ld32(tmem_addr(D3, warp, 32), upd);
#pragma unroll
                for (int x = 0; x < 32; ++x) S[32 + x] = fmaf(gam, S[32 + x], upd[x]);
            }
            write_state();  // S_{ci+1}; releases the issuer for the next chunk
        }
        // after an expired wait, release the issuer from whichever named barrier it may
        // be waiting at (surplus arrivals are harmless: the CTA ends)
        if (__any_sync(0xffffffffu, *abort_flag != 0)) {
            named_bar_arrive(kBarState, 160);
            if (warp < 2) named_bar_arrive(kBarVnew, 96);
        }
        if (warp >= 2 && nch > 0 && !*abort_flag) emit_output(nch - 1);
        if (sN && !*abort_flag) {
            float4* dst = reinterpret_cast<float4*>(sN + st_off + (size_t)d * 128);
#pragma unroll
            for (int x = 0; x < kVT / 4; ++x)
                dst[x] = make_float4(S[4 * x], S[4 * x + 1], S[4 * x + 2], S[4 * x + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

cudaError_t launch_tc(const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float scale, const float* s0, void* o, float* sN, int B,
                      int T, int H, const Layout& L, char* ws, cudaStream_t s,
                      void* const* ev) {
    uint8_t* records = reinterpret_cast<uint8_t*>(ws + L.inter_off);
    const int4* ctab = reinterpret_cast<const int4*>(ws + L.chunk_tab_off);
    const int2* stab = reinterpret_cast<const int2*>(ws + L.seq_tab_off);
    const int* count = reinterpret_cast<const int*>(ws + L.count_off);
    int* status = reinterpret_cast<int*>(ws + L.status_off);
    if (L.max_chunks > 0) {
        const uint64_t rows = (uint64_t)B * T, inner = (uint64_t)H * 128;
        CUtensorMap tq, tk, tv, tg;
        if (!make_tmap_2d(&tq, q, true, inner, rows, inner * 2, 64, 32, true) ||
            !make_tmap_2d(&tk, k, true, inner, rows, inner * 2, 64, 64, true) ||
            !make_tmap_2d(&tv, v, true, inner, rows, inner * 2, 64, 64, true) ||
            !make_tmap_2d(&tg, g, false, inner, rows, inner * 4, 128, 64, false))
            return cudaErrorInvalidValue;
        cudaFuncSetAttribute(kda_intra_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kIntraSmem);
        const unsigned blocks = (unsigned)(L.max_chunks * H);
        kda_intra_tc<<<blocks, kIntraThreads, kIntraSmem, s>>>(tq, tk, tv, tg, beta, scale, H, ctab,
                                                               count, L.max_chunks, records, status);
        if (cudaError_t e = cudaGetLastError()) return e;
    }
    if (!record_event(ev, 0, s)) return cudaErrorInvalidResourceHandle;
    if (L.N > 0) {
        cudaFuncSetAttribute(kda_h_o_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kHoSmem);
        const unsigned blocks = (unsigned)L.N * H * 2;
        kda_h_o_tc<<<blocks, kHoThreads, kHoSmem, s>>>(records, ctab, stab, L.max_chunks, s0,
                                                       static_cast<__nv_bfloat16*>(o), sN, H, status);
        if (cudaError_t e = cudaGetLastError()) return e;
    }
    if (!record_event(ev, 1, s)) return cudaErrorInvalidResourceHandle;
    return cudaSuccess;
}

}  // namespace kda
