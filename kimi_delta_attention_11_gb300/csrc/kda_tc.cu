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
//     MMA2  D1 += [Qg rows ; Aqk] V_new                   (rows 64-127: O = Qg S + Aqk V_new)
//     MMA3  D3 = K_bar^T V_new                            (M 128 keys, N 64, K 64)
//     ep2   S = Diag(gamma^C) S + D3; O rows stored.
//   Thread 0 issues the MMAs and the record copies between CTA barriers.
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

__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint4 v) {
    st_shared_v4(addr, v.x, v.y, v.z, v.w);
}

__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
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
    static constexpr uint32_t TS = FAC;                  // solve scratch [3][16][16]
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
        {
            float pre[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int q = 0; q < rg; ++q) {
                float t[8];
                ld8f(tot + q * 128 + dc * 8, swap, t);
#pragma unroll
                for (int m = 0; m < 8; ++m) pre[m] += t[m];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int m = 0; m < 8; ++m) G[r][m] = (G[r][m] + pre[m]) * kLog2e;
        }
        if ((rg & 3) == 0) st8f(refs + (rg >> 2) * 128 + dc * 8, G[0]);
        if (rg == 15) st8f(refs + 4 * 128 + dc * 8, G[3]);
        __syncthreads();

        // block factors (overwrite the scan totals) and gamma^C = 2^{G_63}
        for (int idx = tid; idx < 15 * 128; idx += kIntraThreads) {
            const int f = idx >> 7, d = idx & 127;
            if (f < 4) {
                P0[f * 128 + d] = exp2f(refs[f * 128 + d]);
            } else if (f < 10) {
                const int pi = f - 4;  // (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
                const int b = pi < 1 ? 1 : (pi < 3 ? 2 : 3);
                const int bp = pi - pair_index(b, 0);
                X[pi * 128 + d] = exp2f(refs[b * 128 + d] - refs[bp * 128 + d]);
            } else if (f < 14) {
                const int b = f - 10;
                CF[b * 128 + d] = exp2f(refs[4 * 128 + d] - refs[b * 128 + d]);
            } else {
                reinterpret_cast<float*>(rec + TcRecord::gamma)[d] = exp2f(refs[4 * 128 + d]);
            }
        }
        __syncthreads();

        // a3/a4 operands, row by row
        float R[4][8];  // key factor rows k_j 2^{G_16b(j) - G_j}, kept for the second round
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * rg + r, b = i >> 4, grp = i >> 5, ii = i & 31;
            const float inb = i < len ? 1.f : 0.f;
            const float bi = betas[i];
            float gref[8], e[8], ei[8], p0[8], cf[8];
            ld8f(refs + b * 128 + dc * 8, swap, gref);
            ld8f(P0 + b * 128 + dc * 8, swap, p0);
            ld8f(CF + b * 128 + dc * 8, swap, cf);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                e[m] = exp2f(G[r][m] - gref[m]);
                ei[m] = exp2f(gref[m] - G[r][m]);
            }
            // query: relation B row (in place) and the gated query of the record
            {
                const uint32_t a = sb + M::RB + (grp * 2 + P) * 8192 + sw128_chunk(ii, cc);
                float qv[8], qs[8], qg[8];
                unpack8(ld_shared_u4(a), qv);
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    qs[m] = scale * qv[m] * inb * e[m];
                    qg[m] = qs[m] * p0[m];
                }
                st_shared_u4(a, pack8(qs));
                *reinterpret_cast<uint4*>(rec + TcRecord::wq + P * 16384 + 8192 +
                                          sw128_chunk(i, cc)) = pack8(qg);
            }
            // key: relation B row, D_beta K+ (in place), key factor rows, K_bar
            {
                const uint32_t a = sb + M::KT + P * 8192 + sw128_chunk(i, cc);
                float kv[8], kp[8], kpl[8], kb[8];
                unpack8(ld_shared_u4(a), kv);
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    kv[m] *= inb;
                    kp[m] = bi * kv[m] * e[m];
                    kpl[m] = kp[m] * p0[m];
                    R[r][m] = kv[m] * ei[m];
                    kb[m] = R[r][m] * cf[m];
                }
                st_shared_u4(sb + M::RB + (grp * 2 + P) * 8192 + sw128_chunk(32 + ii, cc), pack8(kp));
                st_shared_u4(a, pack8(kpl));
                *reinterpret_cast<uint4*>(rec + TcRecord::kbar + P * 8192 + sw128_chunk(i, cc)) =
                    pack8(kb);
                // round 0 of relation A: R_0 (rows 0-63) and R_1 (rows 64-127)
                const uint32_t ra = sb + M::RA + P * 16384;
                if (b == 0) {
                    float x10[8], t[8];
                    ld8f(X + pair_index(1, 0) * 128 + dc * 8, swap, x10);
#pragma unroll
                    for (int m = 0; m < 8; ++m) t[m] = R[r][m] * x10[m];
                    st_shared_u4(ra + sw128_chunk(i, cc), pack8(R[r]));
                    st_shared_u4(ra + sw128_chunk(64 + i, cc), pack8(t));
                } else if (b == 1) {
                    st_shared_u4(ra + sw128_chunk(64 + i, cc), pack8(R[r]));
                }
            }
            // value: D_beta V in place
            {
                const uint32_t a = sb + M::VT + P * 8192 + sw128_chunk(i, cc);
                float vv[8];
                unpack8(ld_shared_u4(a), vv);
#pragma unroll
                for (int m = 0; m < 8; ++m) vv[m] *= bi * inb;
                st_shared_u4(a, pack8(vv));
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
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * rg + r, b = i >> 4;
            const uint32_t ra = sb + M::RA + P * 16384;
            float t[8], x[8];
            if (b < 2) {
                ld8f(X + pair_index(2, b) * 128 + dc * 8, swap, x);
#pragma unroll
                for (int m = 0; m < 8; ++m) t[m] = R[r][m] * x[m];
                st_shared_u4(ra + sw128_chunk(i, cc), pack8(t));
            } else if (b == 2) {
                st_shared_u4(ra + sw128_chunk(i, cc), pack8(R[r]));
            }
            if (b < 3) {
                ld8f(X + pair_index(3, b) * 128 + dc * 8, swap, x);
#pragma unroll
                for (int m = 0; m < 8; ++m) t[m] = R[r][m] * x[m];
                st_shared_u4(ra + sw128_chunk(64 + i, cc), pack8(t));
            } else {
                st_shared_u4(ra + sw128_chunk(64 + i, cc), pack8(R[r]));
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
        // a4: (I + L)^{-1}.  Diagonal 16x16 blocks by forward substitution, one column
        // per thread: x_r = delta_rc - sum_{m<r} L[r][m] x_m.
        if (tid < 64) {
            const int b = tid >> 4, cidx = tid & 15, o = 16 * b;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = r == cidx ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) acc = fmaf(-LF[(o + r) * 64 + o + m], x[m], acc);
                x[r] = acc;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) IF[(o + r) * 64 + o + cidx] = x[r];
        }
        __syncthreads();
        // off-diagonal blocks by distance l = i - j:
        //   Ainv_ij = - D_i sum_{k=j}^{i-1} L_ik Ainv_kj   (D_i = Ainv_ii)
        float* TS = reinterpret_cast<float*>(sm + M::TS);
        for (int l = 1; l <= 3; ++l) {
            const int nt = 4 - l;
            for (int e = tid; e < nt * 256; e += kIntraThreads) {
                const int t = e >> 8, r = (e >> 4) & 15, cx = e & 15, i = l + t, j = i - l;
                float acc = 0.f;
                for (int kb = j; kb < i; ++kb)
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        acc = fmaf(LF[(16 * i + r) * 64 + 16 * kb + m],
                                   IF[(16 * kb + m) * 64 + 16 * j + cx], acc);
                TS[t * 256 + r * 16 + cx] = acc;
            }
            __syncthreads();
            for (int e = tid; e < nt * 256; e += kIntraThreads) {
                const int t = e >> 8, r = (e >> 4) & 15, cx = e & 15, i = l + t, j = i - l;
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    acc = fmaf(IF[(16 * i + r) * 64 + 16 * i + m], TS[t * 256 + m * 16 + cx], acc);
                IF[(16 * i + r) * 64 + 16 * j + cx] = -acc;
            }
            __syncthreads();
        }
        // (I + L)^{-1} as the bf16 A operand of the W/U product (rows 64-127 unused)
        for (int u = tid; u < 512; u += kIntraThreads) {
            const int r = u >> 3, jc = u & 7;
            float a[8];
            ld8f(IF + r * 64 + jc * 8, 0, a);
            st_shared_u4(sb + M::AIA + sw128_chunk(r, jc), pack8(a));
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
        const uint32_t dst = warp < 4 ? sb + M::WST : sb + M::UST;
        const uint32_t col0 = warp < 4 ? 0 : 128;
        for (int cb = 0; cb < 4; ++cb) {
            float v[32];
            tmem_ld32(tmem_addr(tmem, warp, col0 + 32 * cb), v);
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                float f[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) f[m] = v[qd * 8 + m];
                st_shared_u4(dst + (cb >> 1) * 8192 + sw128_chunk(r, (cb & 1) * 4 + qd), pack8(f));
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
        bulk_wait_all();
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
constexpr int kHoThreads = 128;           // thread d <-> TMEM lane d <-> key row d of S
constexpr uint32_t kStageBytes = 66560;   // wq|aqk|kbar 56K | U panel 8K | gamma 512 (65 KB)
constexpr uint32_t kStTx = 57344 + 8192 + 512;

struct HoMap {
    static constexpr uint32_t ST = 2 * kStageBytes;   // S tile bf16 [128 keys][64 values]
    static constexpr uint32_t VN = ST + 16384;        // V_new tile bf16 [64 tokens][64 values]
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
    __shared__ uint64_t full[2], bar_m1, bar_m23;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    const int slice = blockIdx.x & 1;
    const int h = (blockIdx.x >> 1) % H;
    const int n = (blockIdx.x >> 1) / H;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int2 sq = seq_tab[n];
    const long long first = sq.x;
    int nch = sq.y;
    if (first + nch > max_chunks) {  // inconsistent cu_seqlens: stop rather than overrun
        if (tid == 0) atomicCAS(status, 0, (int)KDA_ERR_INVALID_ARG);
        nch = (int)(max_chunks > first ? max_chunks - first : 0);
    }

    if (warp == 0) tmem_alloc(&tmem_base, 128);
    if (tid == 0) {
        s_abort = 0;
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&bar_m1, 1);
        mbar_init(&bar_m23, 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base, D1 = tmem, D3 = tmem + 64;
    volatile int* abort_flag = &s_abort;
    const size_t st_off = ((size_t)n * H + h) * 128 * 128 + slice * kVT;

    auto load = [&](int ci) {  // one thread: record of chunk ci into stage ci & 1
        const uint8_t* rec = records + ((size_t)(first + ci) * H + h) * TcRecord::bytes;
        uint8_t* st = sm + (ci & 1) * kStageBytes;
        mbar_arrive_expect_tx(&full[ci & 1], kStTx);
        bulk_load(st + M::WQ, rec + TcRecord::wq, 57344, &full[ci & 1]);  // wq, aqk, kbar
        bulk_load(st + M::U, rec + TcRecord::u + slice * 8192, 8192, &full[ci & 1]);
        bulk_load(st + M::GAM, rec + TcRecord::gamma, 512, &full[ci & 1]);
    };
    if (tid == 0)
        for (int ci = 0; ci < 2 && ci < nch; ++ci) load(ci);

    // thread d owns row d of the state slice, fp32
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
    // S tile: row d of a token... of a key-major [128][64] bf16 operand, 8 chunks of 16 B
    auto write_state = [&]() {
#pragma unroll
        for (int qd = 0; qd < 8; ++qd) {
            float f[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) f[m] = S[qd * 8 + m];
            st_shared_u4(sb + M::ST + sw128_chunk(d, qd), pack8(f));
        }
        fence_proxy_async_smem();
    };
    write_state();
    tc_fence_before();
    __syncthreads();

    const uint32_t idesc_a = idesc_bf16(128, kVT, false, true);  // A K-major, B MN-major
    const uint32_t idesc_t = idesc_bf16(128, kVT, true, true);   // A MN-major (K_bar^T)
    for (int ci = 0; ci < nch; ++ci) {
        const uint32_t stb = sb + (ci & 1) * kStageBytes;
        const uint8_t* st = sm + (ci & 1) * kStageBytes;
        const int4 ent = chunk_tab[first + ci];
        const int t0 = ent.y, len = ent.z;
        if (!mbar_wait_abortable(&full[ci & 1], (ci >> 1) & 1, status, abort_flag)) break;
        if (tid == 0) {
            tc_fence_after();
            // MMA1: D1 = [W ; Qg] S   (K = 128 keys over two panels; S tile MN-major)
            for (int ks = 0; ks < 8; ++ks) {
                const int pp = ks >> 2, kk = ks & 3;
                mma_bf16(D1, desc_sw128(stb + M::WQ + pp * 16384 + kk * 32),
                         desc_sw128_mn(sb + M::ST + ks * 2048, 16384, 1024), idesc_a,
                         ks > 0 ? 1u : 0u);
            }
            mma_commit(&bar_m1);
        }
        if (!mbar_wait_abortable(&bar_m1, ci & 1, status, abort_flag)) break;
        tc_fence_after();
        if (warp < 2) {
            // ep1: V_new[i] = U[i] - (W S)[i], token i = TMEM lane = d
            float ws[64];
            tmem_ld32(tmem_addr(D1, warp, 0), *reinterpret_cast<float(*)[32]>(ws));
            tmem_ld32(tmem_addr(D1, warp, 32), *reinterpret_cast<float(*)[32]>(ws + 32));
#pragma unroll
            for (int qd = 0; qd < 8; ++qd) {
                float uf[8], vn[8];
                unpack8(ld_shared_u4(stb + M::U + sw128_chunk(d, qd)), uf);
#pragma unroll
                for (int m = 0; m < 8; ++m) vn[m] = uf[m] - ws[qd * 8 + m];
                st_shared_u4(sb + M::VN + sw128_chunk(d, qd), pack8(vn));
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            // MMA2: D1 += [Qg panel-1 rows ; Aqk] V_new  (only rows 64-127 are used)
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(D1, desc_sw128(stb + M::WQ + 16384 + 8192 + kk * 32),
                         desc_sw128_mn(sb + M::VN + kk * 2048, 8192, 1024), idesc_a, 1u);
            // MMA3: D3 = K_bar^T V_new (K_bar token-major: MN-major A, 2 atoms 8 KB apart)
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(D3, desc_sw128_mn(stb + M::KB + kk * 2048, 8192, 1024),
                         desc_sw128_mn(sb + M::VN + kk * 2048, 8192, 1024), idesc_t,
                         kk > 0 ? 1u : 0u);
            mma_commit(&bar_m23);
        }
        if (!mbar_wait_abortable(&bar_m23, ci & 1, status, abort_flag)) break;
        tc_fence_after();
        float ov[64];
        if (warp >= 2) {  // O rows: token = lane index - 64
            tmem_ld32(tmem_addr(D1, warp, 0), *reinterpret_cast<float(*)[32]>(ov));
            tmem_ld32(tmem_addr(D1, warp, 32), *reinterpret_cast<float(*)[32]>(ov + 32));
        }
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
        write_state();
        tc_fence_before();
        __syncthreads();
        // the stage of chunk ci is free (its MMAs are complete, U/gamma read): refill it
        if (tid == 0 && ci + 2 < nch) load(ci + 2);
        if (warp >= 2) {
            const int i = d - 64;
            if (i < len) {
                uint4* dst =
                    reinterpret_cast<uint4*>(o + ((size_t)(t0 + i) * H + h) * 128 + slice * kVT);
#pragma unroll
                for (int qd = 0; qd < 8; ++qd) {
                    float f[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) f[m] = ov[qd * 8 + m];
                    dst[qd] = pack8(f);
                }
            }
        }
    }
    if (sN && !*abort_flag) {
        float4* dst = reinterpret_cast<float4*>(sN + st_off + (size_t)d * 128);
#pragma unroll
        for (int x = 0; x < kVT / 4; ++x)
            dst[x] = make_float4(S[4 * x], S[4 * x + 1], S[4 * x + 2], S[4 * x + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
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
