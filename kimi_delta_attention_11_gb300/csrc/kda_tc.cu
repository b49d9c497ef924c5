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
//   a4  (I + L)^{-1} from 16 x 16 blocks: D = inverses of the diagonal blocks (fp32
//       forward substitution on CUDA cores), J = D F (F the blocks below the diagonal),
//       X = (I + J)^{-1} by block forward substitution, (I + L)^{-1} = X D; the block
//       products on the warp-level TF32 instruction (tcgen05 needs M >= 64).
//       W = (I + L)^{-1} D_beta K+ and U = (I + L)^{-1} D_beta V (Tokamax design doc
//       Eq. (6)-(7)) with the k and v tiles rescaled in place as operands (token-major,
//       read MN-major): one M 128 x N 256 x K 64 MMA for the value-sliced record; for the
//       per-chain record W (N 128) and U^T = (D_beta V)^T ((I + L)^{-1})^T (N 64).
//       K_bar = k 2^{G_C - G} and the gated, scaled query Qg (9.1.5).
//   The results form one record per (chunk, head) (TcRecord), written as tensor-core
//   operand images.
//
// kda_h_o_tc: the ordered chunk recurrence (Eq. (8)) fused with the output (Eq. (9)), one
//   CTA per (sequence, head) with all 128 value columns, in transposed form: the state
//   S^T (bf16 copy) and V_new^T live in tensor memory as A operands, one lane per value
//   column, so no shared-memory tile or proxy fence sits in the chain.  Per chunk:
//     MMA1  D1 = S^T [W ; Qg]^T                          (M 128 values, N 128, K 128 keys)
//     ep1   V_new^T = U^T - (W S)^T  -> tensor memory     (D1 columns 0-63)
//     MMA3  D3 = V_new^T K_bar                            (N 128 keys, K 64 tokens)
//     MMA2  D1[64:128] += V_new^T Aqk^T                   (O^T = (Qg S)^T + (Aqk V_new)^T)
//     ep2   S^T = S^T Diag(gamma^C) + D3  -> tensor memory.
//   Eight warps hold the fp32 state (lane = value column, half the keys each); four more
//   warps read the output rows, so that reading them (which waits while the next chunk's
//   product runs) stays off the chain; one warp issues copies and products.
// sliced::kda_h_o_sliced_tc: the same recurrence untransposed with operands in shared
//   memory, one CTA per 64-column value slice: faster when the chains are few and the two
//   stages run as separate kernels.
// kda_fused_tc: both stages in one cooperative launch for few fixed-length chains: some
//   CTAs run the per-chain recurrence (ho_chain) and poll record flags that the other
//   CTAs' persistent intra lanes (intra_unit, two per CTA) set as they finish records.
// kda_h_o_scan / kda_scan_merge: chunk-parallel state scan for very few long chains:
//   segment summaries by the per-chain recurrence, a merge of segment start states, and
//   the replay of every segment (Tokamax design doc, context-parallel section).
//   MMAs are issued by a whole converged warp through elect.sync (mma_bf16_w): a tcgen05
//   product then runs at the pipe's rate (about 48 cycles per M128 x K16 step for N <= 64,
//   64 for N 128, whatever the operand majorness), and the chained recurrence is bound by
//   its dependent product groups and hand-offs, so it keeps its products to the three the
//   method needs.
#include <mutex>

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

// Divides a row of 128 channels, held as 8 channels by each of 16 consecutive lanes, by
// max(||row||_2, 1e-6) ("KDAChunkwise", FP32 core: F.normalize with eps 1e-6).
__device__ __forceinline__ void l2_scale_row(float (&x)[8]) {
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) ss = fmaf(x[m], x[m], ss);
#pragma unroll
    for (int o2 = 8; o2 > 0; o2 >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o2);
    const float inv = 1.f / fmaxf(sqrtf(ss), 1e-6f);
#pragma unroll
    for (int m = 0; m < 8; ++m) x[m] *= inv;
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
    // after the relation MMAs
    static constexpr uint32_t AQS = RA;                  // Aqk bf16 [64][64] K-major
    static constexpr uint32_t LF = RA + 8192;            // L fp32 [64][kLs]
    static constexpr uint32_t DB = RB;                   // D blocks fp32 [4][16][kBs]
    static constexpr uint32_t JB = RB + 4 * 1280;        // J blocks fp32 [6][16][kBs]
    static constexpr uint32_t XB = MISC;                 // X20, X31, X30, scratch [4][16][kBs]
    static constexpr uint32_t AIA = RB + 16384;          // (I + L)^{-1} bf16 [128][64]
    // after the W/U MMA
    static constexpr uint32_t WST = KT;                  // W staging (token-major)
    static constexpr uint32_t UTS = VT;                  // U (token-major) or U^T staging
};
constexpr size_t kIntraSmem = IntraMap::END + 1024;  // + alignment slack
// Row strides (floats) of the solve's fp32 tiles, chosen so that the fragment loads of
// the 16x16 block products hit distinct banks.
constexpr int kLs = 72, kBs = 20;
// The thread that issues (and, for published records, completes) the record's bulk stores:
// lane 0 of the last warp.
constexpr int kStoreThread = kIntraThreads - 32;
static_assert(IntraMap::LF + 64 * kLs * 4 <= IntraMap::RA + 32768, "L tile overflows");
static_assert(IntraMap::JB + 6 * 16 * kBs * 4 <= IntraMap::AIA, "J blocks overflow");
static_assert(4 * 16 * kBs * 4 <= IntraMap::END - IntraMap::MISC, "X blocks overflow");

// One chunk-head of the intra-chunk stage, run by one "lane" of kIntraThreads threads
// (lane-local named barrier 1 + lid, lane-local mbarriers): the standalone kernel has one
// lane per CTA; the fused kernel two per CTA, each working through many chunk-heads.
// kOpts: the in-kernel gate activation / q-k normalisation are compiled in (a separate
// instantiation, so the plain kernel carries none of their code or registers).
// Rec: the record form (TcRecord for the per-chain recurrence kernel, TcRecordS for the
// value-sliced one).
// `sm` is the lane's 1024-aligned shared-memory base, `tmem` its 256 tensor-memory
// columns, k the number of chunk-heads the lane ran before (mbarrier phases).  With
// `prev_flag`, the lane's previous record is published during this one's second relation
// product: the thread that stored it waits for its bulk stores, then sets *prev_flag with
// release semantics (the recurrence CTA of the same launch polls it).  Returns false after
// an expired wait.
template <bool kOpts, typename Rec, int kLid>
__device__ __forceinline__ bool intra_unit(const CUtensorMap* tmq, const CUtensorMap* tmk,
                                           const CUtensorMap* tmv, const CUtensorMap* tmg,
                                           const float* __restrict__ beta, float scale,
                                           const GateArgs& ga, int H, const int4 ent, int h,
                                           uint8_t* __restrict__ rec,
                                           int* __restrict__ prev_flag,
                                           uint8_t* sm, uint32_t tmem, int lid_arg,
                                           int tid, uint32_t k, int* __restrict__ status) {
    // kLid >= 0: the lane index is a constant (the standalone kernel); -1: lid_arg
    const int lid = kLid >= 0 ? kLid : lid_arg;
    using M = IntraMap;
    __shared__ uint64_t s_bar_tma[2], s_bar_rel[2], s_bar_wu[2];
    __shared__ int s_abort_l[2];
    uint64_t& bar_tma = s_bar_tma[lid];
    uint64_t& bar_rel = s_bar_rel[lid];
    uint64_t& bar_wu = s_bar_wu[lid];
    const uint32_t lane_bar = 1 + (uint32_t)lid;
    auto lane_sync = [&]() { named_bar_sync(lane_bar, kIntraThreads); };
    const int t0 = ent.y, len = ent.z;
    const uint32_t sb = smem_u32(sm);
    float* refs = reinterpret_cast<float*>(sm + M::REFS);
    float* tot = reinterpret_cast<float*>(sm + M::FAC);
    float* P0 = reinterpret_cast<float*>(sm + M::P0);
    float* X = reinterpret_cast<float*>(sm + M::X);
    float* CF = reinterpret_cast<float*>(sm + M::CF);
    float* betas = reinterpret_cast<float*>(sm + M::BETA);
    const int warp = tid >> 5, lane = tid & 31;
    const int dc = tid & 15, rg = tid >> 4;  // 8 key channels 8dc.., rows 4rg..4rg+3
    const int P = dc >> 3, cc = dc & 7;      // key panel, chunk within the panel row
    const int swap = (dc >> 2) & 1;

    // k counts the chunk-heads this lane has run: the mbarriers are set up once and then
    // keep their phases (bar_tma and bar_wu complete once per chunk-head, bar_rel twice).
    // The previous chunk-head's shared-memory accesses are ordered before this one's
    // tensor-copy writes by the proxy fence.
    if (tid == 0) {
        s_abort_l[lid] = 0;
        if (k == 0) {
            mbar_init(&bar_tma, 1);
            mbar_init(&bar_rel, 1);
            mbar_init(&bar_wu, 1);
            fence_barrier_init();
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    lane_sync();
    tc_fence_after();
    volatile int* abort_flag = &s_abort_l[lid];

    // a1: tiles by TMA (rows past the end of the tensor read as zero)
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_tma, 3 * 16384 + 32768);
        for (int p = 0; p < 2; ++p)
            for (int pp = 0; pp < 2; ++pp)
                tma_load_2d(sm + M::RB + (p * 2 + pp) * 8192, tmq, h * 128 + 64 * pp, t0 + 32 * p,
                            &bar_tma);
        for (int pp = 0; pp < 2; ++pp) {
            tma_load_2d(sm + M::KT + pp * 8192, tmk, h * 128 + 64 * pp, t0, &bar_tma);
            tma_load_2d(sm + M::VT + pp * 8192, tmv, h * 128 + 64 * pp, t0, &bar_tma);
        }
        tma_load_2d(sm + M::RA, tmg, h * 128, t0, &bar_tma);
    }
    if (tid < 64) betas[tid] = tid < len ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
    mbar_wait_abortable(&bar_tma, k & 1u, status, abort_flag);
    lane_sync();
    if (*abort_flag) goto teardown;

    {
        // a2: cumsum of g over the chunk in registers
        float G[4][8];
        const float* gt = reinterpret_cast<const float*>(sm + M::RA);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = 4 * rg + r;
            ld8f(gt + i * 128 + dc * 8, swap, G[r]);
            if (kOpts && ga.mode != 0) {  // raw gate -> ln(alpha) (Tokamax design doc 9.1.3)
#pragma unroll
                for (int m = 0; m < 8; ++m) G[r][m] = gate_log_decay(ga, G[r][m], h, dc * 8 + m, 128);
            }
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
        lane_sync();
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
        lane_sync();
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
        lane_sync();

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
                reinterpret_cast<float*>(rec + Rec::gamma)[d] = exp2f(gr[4]);
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
        lane_sync();

        // a3/a4 operands, row by row (the 4 rows of a thread lie in one 16-row block b)
        float R[4][8];  // key factor rows k_j 2^{G_16b(j) - G_j}, kept for the second round
        const int b = rg >> 2;
        float gref[8], p0[8], cf[8], x10[8];
        ld8f(refs + b * 128 + dc * 8, swap, gref);
        ld8f(P0 + b * 128 + dc * 8, swap, p0);
        ld8f(CF + b * 128 + dc * 8, swap, cf);
        if (b == 0) ld8f(X + pair_index(1, 0) * 128 + dc * 8, swap, x10);
        uint4 qr[2], kr[2], vr[2];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            {
                const int i = 4 * rg + r;
                qr[r & 1] = lds128(sm, M::RB + ((i >> 5) * 2 + P) * 8192 + sw128_chunk(i & 31, cc));
                kr[r & 1] = lds128(sm, M::KT + P * 8192 + sw128_chunk(i, cc));
                vr[r & 1] = lds128(sm, M::VT + P * 8192 + sw128_chunk(i, cc));
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
                if (kOpts && ga.qk_l2norm) l2_scale_row(qv);
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    qs[m] = scale * qv[m] * inb * e[m];
                    qg[m] = qs[m] * p0[m];
                }
                sts128(sm, a, pack8(qs));
                *reinterpret_cast<uint4*>(rec + Rec::wq + P * 16384 + 8192 +
                                          sw128_chunk(i, cc)) = pack8(qg);  // rows 64-127
            }
            // key: relation B row, D_beta K+ (in place), key factor rows, K_bar
            {
                const uint32_t a = M::KT + P * 8192 + sw128_chunk(i, cc);
                float kv[8], kp[8], kpl[8], kb[8];
                unpack8(kr[r & 1], kv);
                if (kOpts && ga.qk_l2norm) l2_scale_row(kv);
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
                *reinterpret_cast<uint4*>(rec + (P ? Rec::kb1 : Rec::kb0) +
                                          sw128_chunk(i, cc)) = pack8(kb);
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
        lane_sync();

        // relation round 0: query blocks 0 and 1 -> TMEM columns 0-63
        if (warp == 0) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, 64);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int pp = ks >> 2, kk = ks & 3;
                mma_bf16_w(tmem, desc_sw128(sb + M::RA + pp * 16384 + kk * 32),
                           desc_sw128(sb + M::RB + pp * 8192 + kk * 32), idesc, ks > 0 ? 1u : 0u);
            }
            mma_commit_w(&bar_rel);
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
    lane_sync();
    if (*abort_flag) goto teardown;
    if (warp == 0) {  // relation round 1: query blocks 2 and 3 -> TMEM columns 64-127
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(128, 64);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int pp = ks >> 2, kk = ks & 3;
            mma_bf16_w(tmem + 64, desc_sw128(sb + M::RA + pp * 16384 + kk * 32),
                       desc_sw128(sb + M::RB + (2 + pp) * 8192 + kk * 32), idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit_w(&bar_rel);
    }
    // The lane's previous record is published while these products run, by the thread that
    // stored it (lane 0 of the last warp): its bulk stores, issued some microseconds ago,
    // are waited for, then the flag is set with release semantics.  The other threads'
    // direct stores to that record precede the lane barriers passed since.
    if (prev_flag && tid == kStoreThread) {
        bulk_wait_all();
        fence_proxy_async_global();
        __threadfence();
        st_release_gpu(prev_flag, 1);
    }
    mbar_wait_abortable(&bar_rel, 1, status, abort_flag);
    tc_fence_after();
    lane_sync();
    if (*abort_flag) goto teardown;

    {
        // relation epilogue (all 8 warps; warps q and q+4 share TMEM lanes 32q..32q+31,
        // warps 0-3 take round 0, warps 4-7 round 1).  TMEM lane L = key j (L < 64:
        // rebased for the first block of the round, L >= 64: for the second); columns
        // 0-31 the round's 32 query rows, 32-63 its 32 beta-scaled key rows.  Aqk goes
        // straight to its bf16 operand image, L to fp32 for the solve; masked entries are
        // exact zeros.
        float* LF = reinterpret_cast<float*>(sm + M::LF);
        {
            const int qd = warp & 3, ro = warp >> 2;
            const int L = qd * 32 + lane, j = L & 63, hi = L >> 6;
            const int b = 2 * ro + hi;
            float vq[16], vk[16];
            tmem_ld16(tmem_addr(tmem, qd, 64 * ro + 16 * hi), vq);
            tmem_ld16(tmem_addr(tmem, qd, 64 * ro + 32 + 16 * hi), vk);
#pragma unroll
            for (int ci = 0; ci < 16; ++ci) {
                const int i = 16 * b + ci;
                *reinterpret_cast<__nv_bfloat16*>(sm + M::AQS + sw128_offset(i, j)) =
                    __float2bfloat16_rn(j <= i ? vq[ci] : 0.f);
                LF[i * kLs + j] = j < i ? vk[ci] : 0.f;
            }
        }
        tc_fence_before();
        lane_sync();

        // a4: (I + L)^{-1} (Tokamax design doc 4.1.4 expands the same block inverse with
        // MXU products).  L = Lb + F with Lb the strictly lower parts of the 16 x 16
        // diagonal blocks and F the blocks below them.  With D = (I + Lb)^{-1} (block
        // diagonal) and J = D F: I + L = (I + Lb)(I + J), so (I + L)^{-1} = (I + J)^{-1} D
        // = X D, X unit block-lower-triangular with X_i0 = -sum_{k<i} J_ik X_k0 (block
        // forward substitution).  D in fp32 on CUDA cores; the 16 x 16 block products on
        // the warp-level tensor-core instruction in TF32 (inputs rounded to 10 mantissa
        // bits, fp32 accumulation): the result is rounded to bf16 for the W/U product
        // anyway, 4x coarser.
        float* DB = reinterpret_cast<float*>(sm + M::DB);
        float* JB = reinterpret_cast<float*>(sm + M::JB);
        float* XB = reinterpret_cast<float*>(sm + M::XB);
        constexpr int kBlk = 16 * kBs;
        auto put_ai = [&](int r, int cidx, float x) {  // element (r, c) of the bf16 operand
            *reinterpret_cast<__nv_bfloat16*>(sm + M::AIA + sw128_offset(r, cidx)) =
                __float2bfloat16_rn(x);
        };
        // Stage 1 (warps 0-1): D, one column per thread, right-looking forward
        // substitution (after x_m is final, every later row subtracts L[r][m] x_m).
        // Warps 2-7 meanwhile zero the bf16 blocks above the diagonal (192 chunks).
        if (tid < 64) {
            const int bb = tid >> 4, cidx = tid & 15, o = 16 * bb;
            float acc[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) acc[r] = r == cidx ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < 15; ++m)
#pragma unroll
                for (int r = m + 1; r < 16; ++r)
                    acc[r] = fmaf(-LF[(o + r) * kLs + o + m], acc[m], acc[r]);
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                DB[bb * kBlk + r * kBs + cidx] = acc[r];
                put_ai(o + r, o + cidx, acc[r]);
            }
        } else {
            const int t = tid - 64;  // rows 0-15: chunks 2-7; 16-31: 4-7; 32-47: 6-7
            int r, ch;
            if (t < 96) { r = t / 6; ch = 2 + t % 6; }
            else if (t < 160) { r = 16 + (t - 96) / 4; ch = 4 + (t - 96) % 4; }
            else { r = 32 + (t - 160) / 2; ch = 6 + (t - 160) % 2; }
            sts128(sm, M::AIA + sw128_chunk(r, ch), make_uint4(0u, 0u, 0u, 0u));
        }
        lane_sync();

        // Block products: one warp per 16 x 16 result, acc[nt] the two m16n8 tiles.
        // Pair order of the blocks below the diagonal: (1,0) (2,0) (2,1) (3,0) (3,1) (3,2).
        const int fg = lane >> 2, ft = lane & 3;  // fragment row group / thread in group
        auto pair_bi = [](int pi) { return pi < 1 ? 1 : (pi < 3 ? 2 : 3); };
        // acc += sa * A B  (A, B fp32 16 x 16 with row strides lda, ldb)
        auto blk_mma = [&](float (&acc)[2][4], const float* A, int lda, const float* B, int ldb,
                           float sa) {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t a[4];
                a[0] = f32_to_tf32(sa * A[fg * lda + 8 * ks + ft]);
                a[1] = f32_to_tf32(sa * A[(fg + 8) * lda + 8 * ks + ft]);
                a[2] = f32_to_tf32(sa * A[fg * lda + 8 * ks + ft + 4]);
                a[3] = f32_to_tf32(sa * A[(fg + 8) * lda + 8 * ks + ft + 4]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    uint32_t b[2];
                    b[0] = f32_to_tf32(B[(8 * ks + ft) * ldb + 8 * nt + fg]);
                    b[1] = f32_to_tf32(B[(8 * ks + ft + 4) * ldb + 8 * nt + fg]);
                    mma_tf32_16x8x8(acc[nt], a, b);
                }
            }
        };
        // accumulator tile <-> a [16][kBs] block (element (r, c) of tile nt, slot e:
        // r = fg + 8 (e >> 1), c = 8 nt + 2 ft + (e & 1))
        auto acc_load = [&](float (&acc)[2][4], const float* C, float sc) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[nt][e] = sc * C[(fg + 8 * (e >> 1)) * kBs + 8 * nt + 2 * ft + (e & 1)];
        };
        auto acc_store = [&](const float (&acc)[2][4], float* C) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
                    *reinterpret_cast<float2*>(C + (fg + 8 * hr) * kBs + 8 * nt + 2 * ft) =
                        make_float2(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
        };
        // Stage 2 (warps 0-5, warp = pair): J_ij = D_i F_ij.
        if (warp < 6) {
            const int pi = warp, bi = pair_bi(pi), bj = pi - pair_index(bi, 0);
            float acc[2][4] = {};
            blk_mma(acc, DB + bi * kBlk, kBs, LF + (16 * bi) * kLs + 16 * bj, kLs, 1.f);
            acc_store(acc, JB + pi * kBlk);
        }
        lane_sync();
        // Stage 3 (warps 0-2): X20 = J21 J10 - J20, X31 = J32 J21 - J31,
        // X30 = J31 J10 + J32 J20 - J30 - J32 (J21 J10) (warp 2, through a scratch block).
        if (warp < 3) {
            float acc[2][4];
            const float* J = JB;
            if (warp == 0) {
                acc_load(acc, J + 1 * kBlk, -1.f);
                blk_mma(acc, J + 2 * kBlk, kBs, J + 0 * kBlk, kBs, 1.f);
                acc_store(acc, XB + 0 * kBlk);
            } else if (warp == 1) {
                acc_load(acc, J + 4 * kBlk, -1.f);
                blk_mma(acc, J + 5 * kBlk, kBs, J + 2 * kBlk, kBs, 1.f);
                acc_store(acc, XB + 1 * kBlk);
            } else {
                float y[2][4] = {};
                blk_mma(y, J + 2 * kBlk, kBs, J + 0 * kBlk, kBs, 1.f);  // J21 J10
                acc_store(y, XB + 3 * kBlk);
                acc_load(acc, J + 3 * kBlk, -1.f);
                blk_mma(acc, J + 4 * kBlk, kBs, J + 0 * kBlk, kBs, 1.f);
                blk_mma(acc, J + 5 * kBlk, kBs, J + 1 * kBlk, kBs, 1.f);
                __syncwarp();
                blk_mma(acc, J + 5 * kBlk, kBs, XB + 3 * kBlk, kBs, -1.f);
                acc_store(acc, XB + 2 * kBlk);
            }
        }
        lane_sync();
        // Stage 5 (warps 0-5, warp = pair): (I + L)^{-1}_ij = X_ij D_j, written as bf16;
        // X_10 = -J10, X_21 = -J21, X_32 = -J32.
        if (warp < 6) {
            const int pi = warp, bi = pair_bi(pi), bj = pi - pair_index(bi, 0);
            const float* xl = pi == 1 ? XB : (pi == 4 ? XB + kBlk : (pi == 3 ? XB + 2 * kBlk : JB + pi * kBlk));
            const float sgn = (pi == 0 || pi == 2 || pi == 5) ? -1.f : 1.f;
            float acc[2][4] = {};
            blk_mma(acc, xl, kBs, DB + bj * kBlk, kBs, sgn);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
                    *reinterpret_cast<uint32_t*>(sm + M::AIA +
                                                 sw128_offset(16 * bi + fg + 8 * hr, 16 * bj + 8 * nt + 2 * ft)) =
                        pack_bf16x2(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        lane_sync();
    }

    // W = (I+L)^{-1} D_beta K+ (M 128 tokens, 64 used; K 64) with B the token-major k
    // tile rescaled in place (2 atoms, 8 KB apart), and U = (I+L)^{-1} D_beta V:
    //  - sliced record: one N 256 product over the k | v tiles -> TMEM columns 0-255;
    //  - per-chain record: U^T = (D_beta V)^T ((I+L)^{-1})^T instead, M 128 values (A = the
    //    token-major v tile read as MN-major), N 64 tokens (B = (I+L)^{-1} itself, K-major)
    //    -> columns 128-191, so the recurrence reads U^T rows.
    // The same thread then stores Aqk to the record, overlapping the products.
    if (warp == 0) {
        tc_fence_after();
        if constexpr (Rec::sliced) {
            const uint32_t idesc = idesc_bf16(128, 256, false, true);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_w(tmem, desc_sw128(sb + M::AIA + kk * 32),
                           desc_sw128_mn(sb + M::KT + kk * 2048, 8192, 1024), idesc, kk > 0 ? 1u : 0u);
        } else {
            const uint32_t id_w = idesc_bf16(128, 128, false, true);
            const uint32_t id_u = idesc_bf16(128, 64, true, false);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_w(tmem, desc_sw128(sb + M::AIA + kk * 32),
                           desc_sw128_mn(sb + M::KT + kk * 2048, 8192, 1024), id_w, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16_w(tmem + 128, desc_sw128_mn(sb + M::VT + kk * 2048, 8192, 1024),
                           desc_sw128(sb + M::AIA + kk * 32), id_u, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(&bar_wu);
    }
    if (tid == kStoreThread) {
        bulk_store(rec + Rec::aqk, sm + M::AQS, 8192);
        bulk_commit();
    }
    mbar_wait_abortable(&bar_wu, k & 1u, status, abort_flag);
    tc_fence_after();
    lane_sync();
    if (*abort_flag) goto teardown;

    // W rows (warps 0,1; lane = token, 128 keys) into the token-major staging tile of the
    // [W ; Qg] panels.  U: token-major rows (warps 4,5, sliced record) or U^T rows (warps
    // 4-7; lane = value, 64 tokens) into a K-major [128][64] tile.  All go to the record by
    // bulk copies (whole lines, where per-thread row stores would not be).
    if (warp == 0 || warp == 1 || (Rec::sliced && (warp == 4 || warp == 5))) {
        const int r = (warp & 1) * 32 + lane;
        const uint32_t dst = warp < 4 ? M::WST : M::UTS;
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
    } else if (!Rec::sliced && warp >= 4) {
        const int r = (warp & 3) * 32 + lane;
        for (int cb = 0; cb < 2; ++cb) {
            float v[32];
            tmem_ld32(tmem_addr(tmem, warp, 128 + 32 * cb), v);
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                float f[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) f[m] = v[qd * 8 + m];
                sts128(sm, M::UTS + sw128_chunk(r, cb * 4 + qd), pack8(f));
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    lane_sync();
    if (tid == kStoreThread) {
        bulk_store(rec + Rec::wq, sm + M::WST, 8192);
        bulk_store(rec + Rec::wq + 16384, sm + M::WST + 8192, 8192);
        if constexpr (Rec::sliced) {
            bulk_store(rec + TcRecordS::u0, sm + M::UTS, 8192);
            bulk_store(rec + TcRecordS::u1, sm + M::UTS + 8192, 8192);
        } else {
            bulk_store(rec + TcRecord::ut, sm + M::UTS, 16384);
        }
        bulk_commit();
        // only the shared-memory sources must outlive the copies here; a record that is
        // published is waited for during the next one's relation products (or after the last)
        bulk_wait_read_all();
    }
    // A published record's direct stores (query and key rows, gamma) by every thread are
    // ordered before its flag by the lane barriers that follow and the publishing
    // thread's gpu-scope fence before the release store (the fence is cumulative).

teardown:
    tc_fence_before();
    lane_sync();
    return *abort_flag == 0;
}

template <bool kOpts, typename Rec>
__global__ void __launch_bounds__(kIntraThreads, 2)
kda_intra_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
             const float* __restrict__ beta, float scale, GateArgs ga, int H, ChunkIndex cx,
             long long max_chunks, RangeArgs ra, uint8_t* __restrict__ records,
             int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_base;
    const long long blk = blockIdx.x;
    const int h = (int)(blk % H);
    long long c, slot;
    if (ra.span == 0) {
        // whole problem: chunks from the last to the first, so that the records of early
        // chunks, which the recurrence reads first, are the most recently written
        c = max_chunks - 1 - blk / H;
        if (c >= cx.num_chunks(max_chunks)) return;
        slot = c;
    } else {
        // chunks j0 <= j < j0 + span of every sequence (j = index within the sequence)
        const long long rest = blk / H;
        const int jj = (int)(rest % ra.span), n = (int)(rest / ra.span);
        const int2 sq = cx.seq(n);
        if (ra.j0 + jj >= sq.y) return;
        c = sq.x + ra.j0 + jj;
        slot = (long long)n * ra.span + jj;
    }
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    if (threadIdx.x < 32) tmem_alloc(&tmem_base, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_base, 0);
    intra_unit<kOpts, Rec, 0>(&tm_q, &tm_k, &tm_v, &tm_g, beta, scale, ga, H, cx.chunk(c), h,
                              records + ((size_t)slot * H + h) * Rec::bytes, nullptr, sm, tmem,
                              0, threadIdx.x, 0u, status);
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// recurrence + output kernel
// ---------------------------------------------------------------------------

constexpr int kEpiWarps = 8;              // warp w: TMEM lanes 32 (w % 4).. = value columns,
                                          // half w / 4 of the keys / tokens
constexpr int kIssuerWarp = kEpiWarps;    // record copies and MMA issue
constexpr int kOutWarp0 = kEpiWarps + 1;  // 4 output warps (one per TMEM lane quadrant)
constexpr int kHoThreads = (kEpiWarps + 5) * 32;
constexpr uint32_t kChainThreads = (kEpiWarps + 1) * 32;  // named-barrier participants
constexpr int kStages = 3;                // record ring depth: copies run 2 chunk steps ahead
constexpr uint32_t kStage = TcRecord::bytes;
// named barriers between the epilogue warps and the issuer warp
constexpr uint32_t kBarVnew = 1;          // V_new^T written to tensor memory
constexpr uint32_t kBarState = 2;         // S^T (bf16 operand) written, D3 / D1 read
// tensor-memory columns (512 allocated: one CTA per SM)
constexpr uint32_t kColD1 = 0;            // 2 x 128: [(W S)^T | O^T] per chunk, alternating
constexpr uint32_t kColD3 = 256;          // 128: (K_bar^T V_new)^T
constexpr uint32_t kColS = 384;           // 64: S^T as bf16 A operand (128 keys)
constexpr uint32_t kColVn = 448;          // 32: V_new^T as bf16 A operand (64 tokens)
constexpr size_t kHoSmem = kStages * kStage + 1024;
static_assert(kHoSmem <= 232448, "recurrence kernel exceeds the shared-memory limit");
static_assert(TcRecord::used <= kStage && TcRecord::kb1 == TcRecord::kb0 + 8192,
              "record layout assumed by the recurrence kernel");

// Whole warp: 16 consecutive 32-bit columns of the thread's own TMEM lane, then waits for
// the stores to complete.
__device__ __forceinline__ void tmem_st16_wait(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// Chunk-parallel state scan (Tokamax design doc, context-parallel section: the chunk
// transition S' = Phi_c S + Psi_c with Phi_c = Diag(gamma_c) - K_bar_c^T W_c and
// Psi_c = K_bar_c^T U_c is affine, so segments compose).  Mode 1 runs segment `seg` of a
// chain from S = 0 with the chunk's U (var 0: the segment's Psi) or from S = I with U = 0
// (var 1: its Phi, column by column) and writes the end state to summ; mode 2 runs the
// segment from its merged start state with the output on.  The recurrence of each column
// of S is independent of the others, which is what lets the identity start give Phi.
struct ScanArgs {
    int mode = 0, P = 0, L = 0, nc = 0;
    const float* starts = nullptr;  // [P][nc][K][V] segment start states (mode 2)
    float* summ = nullptr;          // [2][P][nc][K][V] segment end states (mode 1)
};

// The chain (sequence n, head h) of the per-chain recurrence, run by the whole CTA (at
// least kHoThreads threads; warps past the roles idle).  With `flags`, the records are
// produced by other CTAs of the same launch: a loader warp polls each record's flag
// before copying it, and a stage is refilled once the products that read it are done.
template <bool kPublished>
__device__ __forceinline__ void ho_chain(int n, int h, const int* __restrict__ flags,
                                         const uint8_t* __restrict__ records, const ChunkIndex& cx,
                                         long long max_chunks, const RangeArgs& ra,
                                         const float* __restrict__ s0, __nv_bfloat16* __restrict__ o,
                                         float* __restrict__ sN, int H, int* __restrict__ status,
                                         const ScanArgs& sc = ScanArgs{}, int seg = 0, int var = 0) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[kStages], empty[kStages], bar_m1, bar_m3, bar_m2[2], bar_out[2];
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int2 sq = cx.seq(n);
    int seq_chunks = sq.y;
    if ((long long)sq.x + seq_chunks > max_chunks) {  // inconsistent cu_seqlens: stop rather than overrun
        if (tid == 0) atomicCAS(status, 0, (int)KDA_ERR_INVALID_ARG);
        seq_chunks = (int)(max_chunks > sq.x ? max_chunks - sq.x : 0);
    }
    // this launch runs chunks lo <= j < hi of the sequence (all of them, or one range of a
    // pipelined call); the state comes from initial_state (or zeros) at j = 0, else from
    // the carry buffer, and goes to final_state after the sequence's last chunk, else to
    // the carry buffer
    // (scan mode: segment seg of the chain, see ScanArgs)
    const int lo = sc.mode ? seg * sc.L : (ra.span ? ra.j0 : 0);
    const int hi = sc.mode ? min(lo + sc.L, seq_chunks) : (ra.span ? min(ra.j0 + ra.span, seq_chunks) : seq_chunks);
    if (lo >= hi && !(lo == 0 && seq_chunks == 0)) return;  // nothing of this sequence here
    const int nch = hi > lo ? hi - lo : 0;
    const long long first = (long long)sq.x + lo;            // global index of chunk lo
    const long long slot0 = ra.span ? (long long)n * ra.span : first;
    const size_t seg_off = (size_t)seg * sc.nc * 128 * 128;  // (seg, chain 0) in a [P][nc][K][V] buffer
    const float* s_in = lo == 0 ? s0 : ra.carry;
    float* s_out = hi == seq_chunks ? sN : ra.carry;
    bool s_identity = false, zero_u = false;
    if (sc.mode == 1) {
        s_in = nullptr;
        s_identity = zero_u = var == 1;
        s_out = sc.summ + (size_t)var * sc.P * sc.nc * 128 * 128 + seg_off;
        o = nullptr;
    } else if (sc.mode == 2) {
        s_in = seg == 0 ? s0 : sc.starts + seg_off;
        s_out = hi == seq_chunks ? sN : nullptr;
    }
    auto rec_of = [&](int ci) {
        return records + ((size_t)(slot0 + ci) * H + h) * TcRecord::bytes;
    };

    if (warp == 0) tmem_alloc(&tmem_base, 512);
    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&bar_m1, 1);
        mbar_init(&bar_m3, 1);
        mbar_init(&bar_m2[0], 1);
        mbar_init(&bar_m2[1], 1);
        mbar_init(&bar_out[0], 4 * 32);
        mbar_init(&bar_out[1], 4 * 32);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    volatile int* abort_flag = &s_abort;

    if (warp >= kOutWarp0 + 4) {
        // ---- loader warp (published records only): copy record ci into stage ci % 3
        // once its flag is set and the products of chunk ci - 3 are done ----
        if (kPublished && warp == kOutWarp0 + 4 && lane == 0) {
            for (int ci = 0; ci < nch; ++ci) {
                const int sg = ci % kStages;
                if (ci >= kStages &&
                    !mbar_wait_abortable(&empty[sg], ((ci / kStages) - 1) & 1, status, abort_flag))
                    break;
                const int* f = flags + (size_t)(first + ci) * H + h;
                uint32_t it = 0;
                while (ld_acquire_gpu(f) == 0 && *abort_flag == 0 && ++it < kWaitLimit) __nanosleep(128);
                if (it >= kWaitLimit) {
                    atomicCAS(status, 0, (int)KDA_ERR_DEVICE_TIMEOUT);
                    *abort_flag = 1;
                }
                if (*abort_flag) break;
                fence_proxy_async_global();
                mbar_arrive_expect_tx(&full[sg], TcRecord::used);
                bulk_load(sm + sg * kStage, rec_of(ci), TcRecord::used, &full[sg]);
            }
        }
        __syncwarp();
    } else if (warp >= kOutWarp0) {
        // ---- output warps: O^T of chunk ci from D1 columns 64-127 (lane = value v, all 64
        // query rows), read while the chain goes on, then the D1 buffer is handed back ----
        // a warp reaches only the TMEM lanes of its own sub-partition (warp % 4)
        const int qd = warp & 3, v = qd * 32 + lane;
        for (int ci = 0; ci < nch; ++ci) {
            if (!__all_sync(0xffffffffu, mbar_wait_abortable(&bar_m2[ci & 1], (ci >> 1) & 1, status,
                                                             abort_flag)))
                break;
            tc_fence_after();
            const int4 ent = cx.chunk(first + ci);
            if (o) {
                __nv_bfloat16* dst = o + ((size_t)ent.y * H + h) * 128 + v;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float ov[32];
                    tmem_ld32(tmem_addr(tmem + kColD1 + 128 * (ci & 1) + 64 + 32 * hh, qd, 0), ov);
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const int i = 32 * hh + x;
                        if (i < ent.z) dst[(size_t)i * H * 128] = __float2bfloat16_rn(ov[x]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bar_out[ci & 1]);
        }
    } else if (warp == kIssuerWarp) {
        // ---- issuer warp: record copies and every MMA (lane 0 issues).  The whole warp
        // runs the loop so that its named-barrier syncs are warp-uniform; every exit
        // decision is made uniform with a warp vote. ----
        auto load = [&](int ci) {  // record of chunk ci into stage ci % kStages (lane 0)
            const int sg = ci % kStages;
            mbar_arrive_expect_tx(&full[sg], TcRecord::used);
            bulk_load(sm + sg * kStage, rec_of(ci), TcRecord::used, &full[sg]);
        };
        if (lane == 0 && !kPublished)
            for (int ci = 0; ci < kStages && ci < nch; ++ci) load(ci);
        __syncwarp();
        const uint32_t id_1 = idesc_bf16(128, 128, false, false);  // D1 = S^T [W ; Qg]^T
        const uint32_t id_3 = idesc_bf16(128, 128, false, true);   // D3 = V_new^T K_bar
        const uint32_t id_2 = idesc_bf16(128, 64, false, false);   // O^T += V_new^T Aqk^T
        for (int ci = 0; ci < nch; ++ci) {
            const int sg = ci % kStages;
            const uint32_t stb = sb + sg * kStage;
            const uint32_t D1 = tmem + kColD1 + 128 * (ci & 1);
            bool ok = mbar_wait_abortable(&full[sg], (ci / kStages) & 1, status, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            named_bar_sync(kBarState, kChainThreads);  // S_ci^T in tensor memory
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            // chunk ci - 1's stage is free once its products are done (the commit tracks
            // them) and its epilogue, which reads gamma there, has passed the sync above
            if (kPublished && ci >= 1) mma_commit_w(&empty[(ci - 1) % kStages]);
            if (ci >= 2) {  // D1 buffer of chunk ci-2 read by the output warps
                ok = mbar_wait_abortable(&bar_out[ci & 1], ((ci - 2) >> 1) & 1, status, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            tc_fence_after();
            // MMA1: D1 = S^T [W ; Qg]^T   (K = 128 keys: A 8 columns per step, B two
            // K-major panels)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16_ta_w(D1, tmem + kColS + 8 * ks,
                              desc_sw128(stb + TcRecord::wq + (ks >> 2) * 16384 + (ks & 3) * 32),
                              id_1, ks > 0 ? 1u : 0u);
            mma_commit_w(&bar_m1);
            __syncwarp();
            // refill the stage chunk ci-1 used: its MMA2 precedes this MMA1 on the pipe
            if (!kPublished && ci >= 1 && ci - 1 + kStages < nch) {
                ok = mbar_wait_abortable(&bar_m2[(ci - 1) & 1], ((ci - 1) >> 1) & 1, status, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) break;
                if (lane == 0) load(ci - 1 + kStages);
                __syncwarp();
            }
            named_bar_sync(kBarVnew, kChainThreads);  // V_new^T in tensor memory
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            tc_fence_after();
            {
                // MMA3 first (it feeds the state): D3 = V_new^T K_bar (K = 64 tokens; K_bar
                // token-major: MN-major B, 2 atoms 8 KB apart)
                const uint64_t dKB = desc_sw128_mn(stb + TcRecord::kb0, 8192, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ta_w(tmem + kColD3, tmem + kColVn + 8 * kk,
                                  dKB + (uint64_t)((kk * 2048) >> 4), id_3, kk > 0 ? 1u : 0u);
                mma_commit_w(&bar_m3);
                // MMA2: D1 columns 64-127 += V_new^T Aqk^T  (O^T = (Qg S)^T + (Aqk V_new)^T)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ta_w(D1 + 64, tmem + kColVn + 8 * kk,
                                  desc_sw128(stb + TcRecord::aqk + kk * 32), id_2, 1u);
                mma_commit_w(&bar_m2[ci & 1]);
            }
            __syncwarp();
        }
    } else {
        // ---- epilogue warps: thread (v, half) owns value column v (TMEM lane) and keys
        // 64 half .. 64 half + 63 of the state, fp32 ----
        const int qd = warp & 3, half = warp >> 2, v = qd * 32 + lane;
        const size_t st_base = ((size_t)n * H + h) * 128 * 128 + (size_t)(64 * half) * 128 + v;
        float S[64];
#pragma unroll
        for (int x = 0; x < 64; ++x)
            S[x] = s_in ? s_in[st_base + (size_t)x * 128] : (s_identity && 64 * half + x == v ? 1.f : 0.f);
        // S^T as bf16 operand columns (2 keys per column) of this thread's lane
        auto write_state = [&]() {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t pk[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) pk[m] = pack_bf16x2(S[32 * hh + 2 * m], S[32 * hh + 2 * m + 1]);
                tmem_st16_wait(tmem_addr(tmem + kColS + 32 * half + 16 * hh, qd, 0), pk);
            }
            tc_fence_before();
            named_bar_arrive(kBarState, kChainThreads);
        };
        write_state();
        for (int ci = 0; ci < nch; ++ci) {
            const int sg = ci % kStages;
            const uint32_t D1 = tmem + kColD1 + 128 * (ci & 1);
            const uint8_t* st = sm + sg * kStage;
            if (!__all_sync(0xffffffffu,
                            mbar_wait_abortable(&full[sg], (ci / kStages) & 1, status, abort_flag)))
                break;
            // U^T is fetched before the product it combines with completes
            uint4 ur[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) ur[q4] = lds128(st, TcRecord::ut + sw128_chunk(v, 4 * half + q4));
            if (!__all_sync(0xffffffffu, mbar_wait_abortable(&bar_m1, ci & 1, status, abort_flag)))
                break;
            tc_fence_after();
            {
                // ep1: V_new^T[v][t] = U^T[v][t] - (W S)^T[v][t], tokens 32 half .. + 31
                float ws[32];
                tmem_ld32(tmem_addr(D1 + 32 * half, qd, 0), ws);
                uint32_t pk[16];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float uf[8];
                    unpack8(zero_u ? make_uint4(0u, 0u, 0u, 0u) : ur[q4], uf);
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        pk[4 * q4 + m] = pack_bf16x2(uf[2 * m] - ws[8 * q4 + 2 * m],
                                                     uf[2 * m + 1] - ws[8 * q4 + 2 * m + 1]);
                }
                tmem_st16_wait(tmem_addr(tmem + kColVn + 16 * half, qd, 0), pk);
                tc_fence_before();
                named_bar_arrive(kBarVnew, kChainThreads);
            }
            if (!__all_sync(0xffffffffu, mbar_wait_abortable(&bar_m3, ci & 1, status, abort_flag)))
                break;
            tc_fence_after();
            // ep2: S[v][key] = gamma[key] S[v][key] + D3[v][key], keys 64 half .. + 63
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float upd[32];
                tmem_ld32(tmem_addr(tmem + kColD3 + 64 * half + 32 * hh, qd, 0), upd);
                const float4* gp =
                    reinterpret_cast<const float4*>(st + TcRecord::gamma) + 16 * half + 8 * hh;
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const float4 g4 = gp[x];
                    float* sx = S + 32 * hh + 4 * x;
                    sx[0] = fmaf(g4.x, sx[0], upd[4 * x]);
                    sx[1] = fmaf(g4.y, sx[1], upd[4 * x + 1]);
                    sx[2] = fmaf(g4.z, sx[2], upd[4 * x + 2]);
                    sx[3] = fmaf(g4.w, sx[3], upd[4 * x + 3]);
                }
            }
            write_state();  // S_{ci+1}; releases the issuer for the next chunk
        }
        // after an expired wait, release the issuer from whichever named barrier it may
        // be waiting at (surplus arrivals are harmless: the CTA ends)
        if (__any_sync(0xffffffffu, *abort_flag != 0)) {
            named_bar_arrive(kBarState, kChainThreads);
            named_bar_arrive(kBarVnew, kChainThreads);
        }
        if (s_out && !*abort_flag) {
#pragma unroll
            for (int x = 0; x < 64; ++x) s_out[st_base + (size_t)x * 128] = S[x];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

__global__ void __launch_bounds__(kHoThreads, 1)
kda_h_o_tc(const uint8_t* __restrict__ records, ChunkIndex cx, long long max_chunks, RangeArgs ra,
           const float* __restrict__ s0, __nv_bfloat16* __restrict__ o, float* __restrict__ sN,
           int H, int* __restrict__ status) {
    ho_chain<false>(blockIdx.x / H, blockIdx.x % H, nullptr, records, cx, max_chunks, ra, s0, o, sN, H, status);
}

// Scan passes of the per-chain recurrence: block b = (var * P + seg) * nc + chain (mode 1)
// or seg * nc + chain (mode 2).
__global__ void __launch_bounds__(kHoThreads, 1)
kda_h_o_scan(const uint8_t* __restrict__ records, ChunkIndex cx, long long max_chunks, ScanArgs sc,
             const float* __restrict__ s0, __nv_bfloat16* __restrict__ o, float* __restrict__ sN,
             int H, int* __restrict__ status) {
    const int chain = (int)(blockIdx.x % sc.nc), rest = (int)(blockIdx.x / sc.nc);
    ho_chain<false>(chain / H, chain % H, nullptr, records, cx, max_chunks, RangeArgs{}, s0, o, sN, H,
                    status, sc, rest % sc.P, rest / sc.P);
}

// Segment start states of the scan: X_0 = S_0 (or 0), X_{s+1} = Phi_s X_s + Psi_s, in fp32
// (CUDA-core products; P - 1 dependent steps per chain).  Every column of X evolves on its
// own, so block (chain, 8-column slice of V) carries its slice through all steps; 256
// threads: thread (row r = t / 2, columns 4 (t % 2) ..) of the slice.  Phi_s is staged in
// shared memory with rows padded to 129 floats (conflict-free reads down a column), and
// the next step's Phi is loaded into registers while this step computes.
constexpr int kMergeThreads = 256;
constexpr int kMergeCols = 8;
__global__ void __launch_bounds__(kMergeThreads)
kda_scan_merge(ScanArgs sc, const float* __restrict__ s0, float* __restrict__ starts) {
    extern __shared__ float merge_smem[];
    float* Phs = merge_smem;                 // [128][129]
    float* X = merge_smem + 128 * 129;       // [128][kMergeCols]
    const int chain = blockIdx.x, c0 = kMergeCols * blockIdx.y;
    const int t = threadIdx.x, r = t >> 1, cc = 4 * (t & 1);
    const size_t cst = (size_t)chain * 128 * 128;
    const size_t plane = (size_t)sc.nc * 128 * 128;
    for (int x = 0; x < 4; ++x)
        X[r * kMergeCols + cc + x] = s0 ? s0[cst + (size_t)r * 128 + c0 + cc + x] : 0.f;
    float4 ph[16];
    auto load_phi = [&](int sg) {
        const float4* src = reinterpret_cast<const float4*>(sc.summ + (size_t)(sc.P + sg) * plane + cst);
#pragma unroll
        for (int i = 0; i < 16; ++i) ph[i] = src[t + kMergeThreads * i];
    };
    if (sc.P > 1) load_phi(0);
    for (int sg = 0; sg + 1 < sc.P; ++sg) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int e = 4 * (t + kMergeThreads * i), row = e >> 7, col = e & 127;
            float* d = Phs + row * 129 + col;
            d[0] = ph[i].x;
            d[1] = ph[i].y;
            d[2] = ph[i].z;
            d[3] = ph[i].w;
        }
        const float4 ps = *reinterpret_cast<const float4*>(sc.summ + (size_t)sg * plane + cst +
                                                          (size_t)r * 128 + c0 + cc);
        __syncthreads();
        if (sg + 2 < sc.P) load_phi(sg + 1);  // in flight while this step computes
        float acc[4] = {ps.x, ps.y, ps.z, ps.w};
        const float* prow = Phs + r * 129;
#pragma unroll 8
        for (int d = 0; d < 128; ++d) {
            const float f = prow[d];
            const float4 xv = *reinterpret_cast<const float4*>(X + d * kMergeCols + cc);
            acc[0] = fmaf(f, xv.x, acc[0]);
            acc[1] = fmaf(f, xv.y, acc[1]);
            acc[2] = fmaf(f, xv.z, acc[2]);
            acc[3] = fmaf(f, xv.w, acc[3]);
        }
        __syncthreads();
        float* dst = starts + (size_t)(sg + 1) * plane + cst + (size_t)r * 128 + c0 + cc;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            X[r * kMergeCols + cc + x] = acc[x];
            dst[x] = acc[x];
        }
        __syncthreads();
    }
}
constexpr size_t kMergeSmem = (128 * 129 + 128 * kMergeCols) * sizeof(float);

// Fused schedule for few chains of fixed-length sequences: one persistent CTA per SM.
// CTAs 0 .. nc - 1 each run the per-chain recurrence of chain b = n H + h; every other
// CTA runs two intra lanes, which work through the chunk-heads in chunk-major order
// (chunk 0 of every chain first, as the recurrences consume them) and publish each record
// through its flag.  The recurrence CTAs poll those flags, so the launch is cooperative:
// all CTAs are resident, and a producer never waits for a consumer.
constexpr int kFusedThreads = 2 * kIntraThreads;
static_assert(kFusedThreads >= kHoThreads + 32, "fused CTA must hold the recurrence roles and its loader");
constexpr uint32_t kIntraLane = (uint32_t)((IntraMap::END + 1023) / 1024 * 1024);
constexpr size_t kFusedSmem =
    (2ull * kIntraLane > (size_t)kStages * kStage ? 2ull * kIntraLane : (size_t)kStages * kStage) + 1024;
static_assert(kFusedSmem <= 232448, "fused kernel exceeds the shared-memory limit");

// The recurrence role of the fused kernel, compiled as its own function so that its
// registers are allocated apart from the intra lanes'.
__device__ __noinline__ void ho_chain_published(int n, int h, const int* __restrict__ flags,
                                                const uint8_t* __restrict__ records,
                                                const ChunkIndex& cx, long long max_chunks,
                                                const float* __restrict__ s0,
                                                __nv_bfloat16* __restrict__ o, float* __restrict__ sN,
                                                int H, int* __restrict__ status) {
    ho_chain<true>(n, h, flags, records, cx, max_chunks, RangeArgs{}, s0, o, sN, H, status);
}

// Arguments of the fused kernel (one grid-constant block, read in place by both roles).
struct FusedArgs {
    CUtensorMap tq, tk, tv, tg;
    const float* beta;
    float scale;
    GateArgs ga;
    int H;
    ChunkIndex cx;
    long long max_chunks;
    uint8_t* records;
    int* flags;
    const float* s0;
    __nv_bfloat16* o;
    float* sN;
    int nc;
    int* status;
};

// One intra lane of the fused kernel: units u0, u0 + lanes, ... (chunk j = u / nc of chain
// u % nc), each record published during the next one's relation products (the last at
// the end).
// Both lanes of a CTA run the same code (one copy: the kernel is large, and instruction
// fetch stalls when the SM alternates between two copies).
template <bool kOpts>
__device__ __forceinline__ void intra_lane(const FusedArgs& A, uint8_t* sm, uint32_t tmem, int lid, int tid) {
    const int nc = A.nc, H = A.H, T = A.cx.T;
    const long long lanes = 2ll * ((long long)gridDim.x - nc);
    const long long units = (long long)nc * A.cx.nct;
    long long u = 2ll * ((long long)blockIdx.x - nc) + lid;
    // unit u is chunk j = u / nc of chain n = u % nc; from one unit of the lane to the next
    // (j, n) advance by (lanes / nc, lanes % nc) with a carry: 64-bit divisions here took
    // ~0.7 us of the 2.2 us that passed between two chunk-heads of a lane
    const int dj = (int)(lanes / nc), dn = (int)(lanes % nc);
    int j = (int)(u / nc), n = (int)(u % nc);
    int* prev = nullptr;
    uint32_t k = 0;
    bool ok = true;
#pragma unroll 1
    for (; u < units; u += lanes, ++k) {
        // the thread index goes through an empty asm each unit, so that the compiler
        // derives the per-thread offsets inside the unit instead of holding them across
        // the loop (registers are the intra lane's limit)
        int tid_u = tid;
        asm volatile("" : "+r"(tid_u));
        const int b = n / H, h = n - b * H;  // sequence, head
        const long long c = (long long)b * A.cx.nct + j;
        const int4 ent = make_int4(b, b * T + j * kChunk, min(kChunk, T - j * kChunk), j);
        ok = intra_unit<kOpts, TcRecord, -1>(&A.tq, &A.tk, &A.tv, &A.tg, A.beta, A.scale, A.ga, H, ent,
                                             h, A.records + ((size_t)c * H + h) * TcRecord::bytes,
                                             prev, sm, tmem, lid, tid_u, k, A.status);
        if (!ok) break;
        prev = A.flags + (size_t)c * H + h;
        j += dj;
        n += dn;
        if (n >= nc) {
            n -= nc;
            ++j;
        }
    }
    if (ok && k > 0 && tid == kStoreThread) {  // the lane's last record (its storing thread)
        bulk_wait_all();
        fence_proxy_async_global();
        __threadfence();
        st_release_gpu(prev, 1);
    }
}

template <bool kOpts>
__global__ void __launch_bounds__(kFusedThreads, 1) kda_fused_tc(const __grid_constant__ FusedArgs A) {
    const int nc = A.nc, H = A.H;
    if ((int)blockIdx.x < nc) {
        ho_chain_published((int)blockIdx.x / H, (int)blockIdx.x % H, A.flags, A.records, A.cx,
                           A.max_chunks, A.s0, A.o, A.sN, H, A.status);
        return;
    }
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_base;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int lid = (int)threadIdx.x / kIntraThreads, tid = (int)threadIdx.x % kIntraThreads;
    if (threadIdx.x < 32) tmem_alloc(&tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = __shfl_sync(0xffffffffu, tmem_base, 0);
    intra_lane<kOpts>(A, sm + lid * kIntraLane, tbase + 256u * (uint32_t)lid, lid, tid);
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) tmem_dealloc(tbase, 512);
}

// Value-sliced recurrence: one CTA (8 epilogue warps + 1 issuer warp) per (sequence,
// head, 64-column slice of V), untransposed products with both operands in shared
// memory.  Used when the chains are few (two CTAs per chain fill the SMs and the
// shorter chained products win); see kda_h_o_tc for the per-chain form.
//   MMA1  D1 = [W ; Qg] S                              (M 128, N 64, K 128)
//   ep1   V_new = U - W S                               (D1 rows 0-63)
//   MMA3  D3 = K_bar^T V_new                            (M 128 keys, N 64, K 64)
//   MMA2  D1 += [Qg rows ; Aqk] V_new                   (rows 64-127: O = Qg S + Aqk V_new)
//   ep2   S = Diag(gamma^C) S + D3.
namespace sliced {

constexpr int kVT = 64;                   // value columns per CTA
constexpr int kEpiWarps = 8;              // warp w: TMEM lanes 32 (w % 4).., value columns
                                          // 32 (w / 4).. of the slice
constexpr int kHoThreads = (kEpiWarps + 1) * 32;  // + 1 issuer warp
constexpr int kStages = 3;                // record ring depth: copies run 2 chunk steps ahead
constexpr uint32_t kStage = 65536;        // one contiguous run of the record per chunk
// named barriers between the epilogue warps and the issuer warp
constexpr uint32_t kBarVnew = 1;          // warps of lanes 0-63 -> issuer: V_new tile written
constexpr uint32_t kBarState = 2;         // all epilogue warps -> issuer: S tile written
constexpr uint32_t kVnewCount = 4 * 32 + 32;

struct HoMap {
    static constexpr uint32_t ST = kStages * kStage;  // S tile bf16 [128 keys][64 values]
    static constexpr uint32_t VN = ST + 16384;         // V_new tile bf16 [64 tokens][64 values]
    static constexpr uint32_t END = VN + 8192;
};
constexpr size_t kHoSmem = HoMap::END + 1024;
static_assert(kHoSmem <= 232448, "recurrence kernel exceeds the shared-memory limit");
static_assert(TcRecordS::u1 == 0 && TcRecordS::u0 == kStage && TcRecordS::gamma == kStage + 8192 &&
                  TcRecordS::aqk == TcRecordS::wq + 32768 && TcRecordS::kb1 == TcRecordS::kb0 + 8192,
              "record layout assumed by the recurrence kernel");

__global__ void __launch_bounds__(kHoThreads, 1)
kda_h_o_sliced_tc(const uint8_t* __restrict__ records, ChunkIndex cx, long long max_chunks, RangeArgs ra,
           const float* __restrict__ s0, __nv_bfloat16* __restrict__ o, float* __restrict__ sN,
           int H, int* __restrict__ status) {
    using M = HoMap;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[kStages], bar_m1, bar_m3, bar_m2[2];
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    const int slice = blockIdx.x & 1;
    const int h = (blockIdx.x >> 1) % H;
    const int n = (blockIdx.x >> 1) / H;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int2 sq = cx.seq(n);
    int seq_chunks = sq.y;
    if ((long long)sq.x + seq_chunks > max_chunks) {  // inconsistent cu_seqlens: stop rather than overrun
        if (tid == 0) atomicCAS(status, 0, (int)KDA_ERR_INVALID_ARG);
        seq_chunks = (int)(max_chunks > sq.x ? max_chunks - sq.x : 0);
    }
    // this launch runs chunks lo <= j < hi of the sequence (all of them, or one range of a
    // pipelined call); the state comes from initial_state (or zeros) at j = 0, else from
    // the carry buffer, and goes to final_state after the sequence's last chunk, else to
    // the carry buffer
    const int lo = ra.span ? ra.j0 : 0;
    const int hi = ra.span ? min(ra.j0 + ra.span, seq_chunks) : seq_chunks;
    if (lo >= hi && !(lo == 0 && seq_chunks == 0)) return;  // nothing of this sequence here
    const int nch = hi > lo ? hi - lo : 0;
    const long long first = (long long)sq.x + lo;            // global index of chunk lo
    const long long slot0 = ra.span ? (long long)n * ra.span : first;
    const float* s_in = lo == 0 ? s0 : ra.carry;
    float* s_out = hi == seq_chunks ? sN : ra.carry;
    auto rec_of = [&](int ci) {
        return records + ((size_t)(slot0 + ci) * H + h) * TcRecordS::bytes;
    };
    // slice s copies record bytes [cs, cs + kStage): stage offset = record offset - cs
    const uint32_t cs = slice ? TcRecordS::u1 : TcRecordS::wq;
    const uint32_t WQ = TcRecordS::wq - cs, AQK = TcRecordS::aqk - cs, KB = TcRecordS::kb0 - cs;
    const uint32_t UO = (slice ? TcRecordS::u1 : TcRecordS::u0) - cs;

    if (warp == 0) tmem_alloc(&tmem_base, 256);
    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
        mbar_init(&bar_m1, 1);
        mbar_init(&bar_m3, 1);
        mbar_init(&bar_m2[0], 1);
        mbar_init(&bar_m2[1], 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // D1 (two buffers, alternating by chunk): [W ; Qg] S, then rows 64-127 += Aqk V_new
    // (the output); D3: K_bar^T V_new (the state update)
    const uint32_t tmem = tmem_base, D3 = tmem + 128;
    volatile int* abort_flag = &s_abort;

    if (warp == kEpiWarps) {
        // ---- issuer warp: record copies and every MMA (lane 0 issues).  The whole warp
        // runs the loop so that its named-barrier syncs are warp-uniform; every exit
        // decision is made uniform with a warp vote. ----
        auto load = [&](int ci) {  // record of chunk ci into stage ci % kStages (lane 0)
            const int sg = ci % kStages;
            mbar_arrive_expect_tx(&full[sg], kStage);
            bulk_load(sm + sg * kStage, rec_of(ci) + cs, kStage, &full[sg]);
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
            const uint32_t stb = sb + sg * kStage;
            const uint32_t D1 = tmem + 64 * (ci & 1);
            bool ok = mbar_wait_abortable(&full[sg], (ci / kStages) & 1, status, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            named_bar_sync(kBarState, kHoThreads);  // S_ci written, D1/D3 of earlier chunks read
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            tc_fence_after();
            {
                // MMA1: D1 = [W ; Qg] S   (K = 128 keys over two panels)
                const uint64_t dWQ = desc_sw128(stb + WQ);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_w(D1, dWQ + (uint64_t)(((ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                               dS + (uint64_t)((ks * 2048) >> 4), idesc_a, ks > 0 ? 1u : 0u);
                mma_commit_w(&bar_m1);
            }
            __syncwarp();
            // refill the stage chunk ci-1 used: its MMA2 precedes this MMA1 on the pipe
            if (ci >= 1 && ci - 1 + kStages < nch) {
                ok = mbar_wait_abortable(&bar_m2[(ci - 1) & 1], ((ci - 1) >> 1) & 1, status, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) break;
                if (lane == 0) load(ci - 1 + kStages);
                __syncwarp();
            }
            named_bar_sync(kBarVnew, kVnewCount);  // V_new tile written
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            tc_fence_after();
            {
                // MMA3 first (it feeds the state): D3 = K_bar^T V_new (K_bar token-major:
                // MN-major A, 2 atoms 8 KB apart)
                const uint64_t dKB = desc_sw128_mn(stb + KB, 8192, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_w(D3, dKB + (uint64_t)((kk * 2048) >> 4),
                               dVN + (uint64_t)((kk * 2048) >> 4), idesc_t, kk > 0 ? 1u : 0u);
                mma_commit_w(&bar_m3);
                // MMA2: D1 += [Qg panel-1 rows ; Aqk] V_new  (only rows 64-127 are used)
                const uint64_t dQA = desc_sw128(stb + AQK - 8192);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_w(D1, dQA + (uint64_t)((kk * 32) >> 4),
                               dVN + (uint64_t)((kk * 2048) >> 4), idesc_a, 1u);
                mma_commit_w(&bar_m2[ci & 1]);
            }
            __syncwarp();
        }
    } else {
        // ---- epilogue warps: thread (d, half) owns 32 columns of row d of the state
        // slice, fp32 ----
        const int qd = warp & 3, half = warp >> 2, d = qd * 32 + lane;
        const size_t st_off = ((size_t)n * H + h) * 128 * 128 + (size_t)d * 128 + slice * kVT + 32 * half;
        float S[32];
        {
            const float4* src = reinterpret_cast<const float4*>(s_in + st_off);
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const float4 f = s_in ? src[x] : make_float4(0.f, 0.f, 0.f, 0.f);
                S[4 * x] = f.x;
                S[4 * x + 1] = f.y;
                S[4 * x + 2] = f.z;
                S[4 * x + 3] = f.w;
            }
        }
        // S tile: key-major [128][64] bf16 (MN-major B operand); this thread writes chunks
        // 4 half .. 4 half + 3 of row d
        auto write_state = [&]() {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float f[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) f[m] = S[q4 * 8 + m];
                sts128(sm, M::ST + sw128_chunk(d, 4 * half + q4), pack8(f));
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_arrive(kBarState, kHoThreads);
        };
        // output rows of chunk ci (TMEM lanes 64-127: token = lane index - 64)
        auto emit_output = [&](int ci) {
            if (!__all_sync(0xffffffffu, mbar_wait_abortable(&bar_m2[ci & 1], (ci >> 1) & 1, status,
                                                             abort_flag)))
                return;
            tc_fence_after();
            float ov[32];
            tmem_ld32(tmem_addr(tmem + 64 * (ci & 1), qd, 32 * half), ov);
            const int4 ent = cx.chunk(first + ci);
            const int i = d - 64;
            if (i < ent.z) {
                uint4* dst = reinterpret_cast<uint4*>(o + ((size_t)(ent.y + i) * H + h) * 128 +
                                                      slice * kVT + 32 * half);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float f[8];
#pragma unroll
                    for (int m = 0; m < 8; ++m) f[m] = ov[q4 * 8 + m];
                    dst[q4] = pack8(f);
                }
            }
        };
        // gamma^C of the next chunks, fetched two chunk steps ahead
        auto gamma_of = [&](int ci) {
            return ci < nch ? reinterpret_cast<const float*>(rec_of(ci) + TcRecordS::gamma)[d] : 0.f;
        };
        float gam0 = gamma_of(0), gam1 = gamma_of(1);
        write_state();
        for (int ci = 0; ci < nch; ++ci) {
            const int sg = ci % kStages;
            const uint32_t D1 = tmem + 64 * (ci & 1);
            const float gam2 = gamma_of(ci + 2);
            if (!__all_sync(0xffffffffu,
                            mbar_wait_abortable(&full[sg], (ci / kStages) & 1, status, abort_flag)))
                break;
            // the previous chunk's output is read while MMA1 runs; U rows are fetched
            // before MMA1 completes
            if (qd >= 2 && ci > 0) emit_output(ci - 1);
            uint4 ur[4];
            if (qd < 2) {
                const uint32_t ub = (uint32_t)sg * kStage + UO;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) ur[q4] = lds128(sm, ub + sw128_chunk(d, 4 * half + q4));
            }
            if (!__all_sync(0xffffffffu, mbar_wait_abortable(&bar_m1, ci & 1, status, abort_flag)))
                break;
            tc_fence_after();
            if (qd < 2) {
                // ep1: V_new[i] = U[i] - (W S)[i], token i = TMEM lane = d, 32 columns
                float ws[32];
                tmem_ld32(tmem_addr(D1, qd, 32 * half), ws);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float uf[8], vn[8];
                    unpack8(ur[q4], uf);
#pragma unroll
                    for (int m = 0; m < 8; ++m) vn[m] = uf[m] - ws[q4 * 8 + m];
                    sts128(sm, M::VN + sw128_chunk(d, 4 * half + q4), pack8(vn));
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_arrive(kBarVnew, kVnewCount);
            }
            if (!__all_sync(0xffffffffu, mbar_wait_abortable(&bar_m3, ci & 1, status, abort_flag)))
                break;
            tc_fence_after();
            {
                float upd[32];
                tmem_ld32(tmem_addr(D3, qd, 32 * half), upd);
#pragma unroll
                for (int x = 0; x < 32; ++x) S[x] = fmaf(gam0, S[x], upd[x]);
            }
            write_state();  // S_{ci+1}; releases the issuer for the next chunk
            gam0 = gam1;
            gam1 = gam2;
        }
        // after an expired wait, release the issuer from whichever named barrier it may
        // be waiting at (surplus arrivals are harmless: the CTA ends)
        if (__any_sync(0xffffffffu, *abort_flag != 0)) {
            named_bar_arrive(kBarState, kHoThreads);
            if (qd < 2) named_bar_arrive(kBarVnew, kVnewCount);
        }
        if (qd >= 2 && nch > 0 && !*abort_flag) emit_output(nch - 1);
        if (s_out && !*abort_flag) {
            float4* dst = reinterpret_cast<float4*>(s_out + st_off);
#pragma unroll
            for (int x = 0; x < 8; ++x)
                dst[x] = make_float4(S[4 * x], S[4 * x + 1], S[4 * x + 2], S[4 * x + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace sliced

}  // namespace

namespace {

// Second stream and events of the pipelined schedule, one set per device, created on
// first use and kept for the life of the process (no device memory is allocated).  The
// mutex keeps two host threads from interleaving their use of the shared events.
struct PipeRes {
    bool ready = false;
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, intra_done[3] = {}, ho_done[3] = {};
};
PipeRes g_pipe[64];
std::mutex g_pipe_mu;

cudaError_t pipe_res(int dev, PipeRes** out) {
    PipeRes& r = g_pipe[dev];
    if (!r.ready) {
        int lo = 0, hi = 0;
        if (cudaError_t e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) return e;
        // the recurrence (the ordered chain) gets the higher priority
        if (cudaError_t e = cudaStreamCreateWithPriority(&r.side, cudaStreamNonBlocking, hi))
            return e;
        cudaEvent_t* evs[] = {&r.fork, &r.join, &r.intra_done[0], &r.intra_done[1],
                              &r.intra_done[2], &r.ho_done[0], &r.ho_done[1], &r.ho_done[2]};
        for (cudaEvent_t* e : evs)
            if (cudaError_t err = cudaEventCreateWithFlags(e, cudaEventDisableTiming)) return err;
        r.ready = true;
    }
    *out = &r;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_tc(const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float scale, const GateArgs& ga, const float* s0, void* o,
                      float* sN, int B, int T, int H, const Layout& L, char* ws, cudaStream_t s,
                      void* const* ev) {
    uint8_t* records = reinterpret_cast<uint8_t*>(ws + L.inter_off);
    ChunkIndex cx;
    cx.chunk_tab = reinterpret_cast<const int4*>(ws + L.chunk_tab_off);
    cx.seq_tab = reinterpret_cast<const int2*>(ws + L.seq_tab_off);
    cx.count = reinterpret_cast<const int*>(ws + L.count_off);
    if (L.fixed) {
        cx.fixed = 1;
        cx.T = T;
        cx.nct = (T + kChunk - 1) / kChunk;
    }
    int* status = reinterpret_cast<int*>(ws + L.status_off);
    CUtensorMap tq, tk, tv, tg;
    if (L.max_chunks > 0) {
        const uint64_t rows = (uint64_t)B * T, inner = (uint64_t)H * 128;
        if (!make_tmap_2d(&tq, q, true, inner, rows, inner * 2, 64, 32, true) ||
            !make_tmap_2d(&tk, k, true, inner, rows, inner * 2, 64, 64, true) ||
            !make_tmap_2d(&tv, v, true, inner, rows, inner * 2, 64, 64, true) ||
            !make_tmap_2d(&tg, g, false, inner, rows, inner * 4, 128, 64, false))
            return cudaErrorInvalidValue;
    }
    // Recurrence form: value-sliced (two CTAs per chain, shorter chained products) while
    // two CTAs per chain fit in one wave of SMs, else one CTA per chain (no work repeated
    // per slice).  The intra-chunk kernel writes the record form that kernel reads.
    int dev = 0, sms = 0;
    if (cudaError_t e = cudaGetDevice(&dev)) return e;
    if (cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) return e;
    const bool sliced = 2ll * L.N * H <= sms;
    const bool opts = ga.mode != 0 || ga.qk_l2norm;
    auto* intra = sliced ? (opts ? kda_intra_tc<true, TcRecordS> : kda_intra_tc<false, TcRecordS>)
                         : (opts ? kda_intra_tc<true, TcRecord> : kda_intra_tc<false, TcRecord>);
    auto* ho = sliced ? sliced::kda_h_o_sliced_tc : kda_h_o_tc;
    const unsigned ho_blocks = (unsigned)L.N * H * (sliced ? 2 : 1);
    const unsigned ho_threads = sliced ? sliced::kHoThreads : kHoThreads;
    const size_t ho_smem = sliced ? sliced::kHoSmem : kHoSmem;
    if (L.max_chunks > 0)
        cudaFuncSetAttribute(intra, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kIntraSmem);
    cudaFuncSetAttribute(ho, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ho_smem);
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);

    // Scan schedule: the intra-chunk kernel (per-chain records), the segment summaries,
    // their merge, and the replay of every segment from its merged start state.
    if (L.scan && !ev) {
        auto* ik = opts ? kda_intra_tc<true, TcRecord> : kda_intra_tc<false, TcRecord>;
        if (cudaError_t e = cudaFuncSetAttribute(ik, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kIntraSmem))
            return e;
        if (cudaError_t e = cudaFuncSetAttribute(kda_h_o_scan, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kHoSmem))
            return e;
        ik<<<(unsigned)(L.max_chunks * H), kIntraThreads, kIntraSmem, s>>>(
            tq, tk, tv, tg, beta, scale, ga, H, cx, L.max_chunks, RangeArgs{}, records, status);
        if (cudaError_t e = cudaGetLastError()) return e;
        ScanArgs sc;
        sc.P = L.scan_P;
        sc.L = L.scan_L;
        sc.nc = L.N * H;
        sc.summ = reinterpret_cast<float*>(ws + L.summ_off);
        sc.starts = reinterpret_cast<const float*>(ws + L.starts_off);
        sc.mode = 1;
        kda_h_o_scan<<<(unsigned)(2 * sc.P * sc.nc), kHoThreads, kHoSmem, s>>>(records, cx, L.max_chunks, sc,
                                                                             s0, ob, sN, H, status);
        if (cudaError_t e = cudaGetLastError()) return e;
        if (cudaError_t e = cudaFuncSetAttribute(kda_scan_merge, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kMergeSmem))
            return e;
        kda_scan_merge<<<dim3((unsigned)sc.nc, 128 / kMergeCols), kMergeThreads, kMergeSmem, s>>>(
            sc, s0, reinterpret_cast<float*>(ws + L.starts_off));
        if (cudaError_t e = cudaGetLastError()) return e;
        sc.mode = 2;
        kda_h_o_scan<<<(unsigned)(sc.P * sc.nc), kHoThreads, kHoSmem, s>>>(records, cx, L.max_chunks, sc,
                                                                         s0, ob, sN, H, status);
        return cudaGetLastError();
    }

    // Fused schedule: one cooperative launch, one CTA per SM (the recurrence CTAs poll
    // flags the other CTAs set, so all CTAs must be resident); the flags start cleared.
    if (L.fused && !ev) {
        int* flags = reinterpret_cast<int*>(ws + L.flags_off);
        if (cudaError_t e = cudaMemsetAsync(flags, 0, (size_t)L.max_chunks * H * sizeof(int), s)) return e;
        auto* fk = opts ? kda_fused_tc<true> : kda_fused_tc<false>;
        if (cudaError_t e = cudaFuncSetAttribute(fk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kFusedSmem))
            return e;
        int per_sm = 0;
        if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fk, kFusedThreads,
                                                                          kFusedSmem))
            return e;
        int nc = L.N * H;
        if (per_sm < 1 || nc >= sms) return cudaErrorInvalidConfiguration;
        FusedArgs fa{tq, tk, tv, tg, beta, scale, ga, H, cx, L.max_chunks, records, flags,
                     s0, ob, sN, nc, status};
        void* args[] = {&fa};
        return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fk), dim3((unsigned)sms),
                                           dim3(kFusedThreads), args, kFusedSmem, s);
    }

    // Whole-problem schedule: one launch of each kernel (and the only one with per-kernel
    // timing events).
    if (L.span == 0 || ev) {
        if (L.max_chunks > 0) {
            const unsigned blocks = (unsigned)(L.max_chunks * H);
            intra<<<blocks, kIntraThreads, kIntraSmem, s>>>(
                tq, tk, tv, tg, beta, scale, ga, H, cx, L.max_chunks, RangeArgs{}, records, status);
            if (cudaError_t e = cudaGetLastError()) return e;
        }
        if (!record_event(ev, 0, s)) return cudaErrorInvalidResourceHandle;
        if (L.N > 0) {
            ho<<<ho_blocks, ho_threads, ho_smem, s>>>(records, cx, L.max_chunks, RangeArgs{}, s0, ob,
                                                      sN, H, status);
            if (cudaError_t e = cudaGetLastError()) return e;
        }
        if (!record_event(ev, 1, s)) return cudaErrorInvalidResourceHandle;
        return cudaSuccess;
    }

    // Pipelined schedule: range r's intra-chunk kernel on the caller's stream, its
    // recurrence on the side stream once range r's records exist and range r - 1's
    // recurrence has handed over the state; records live in a ring of L.ring range slots,
    // so intra of range r waits for the recurrence of range r - ring to have read them.
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    PipeRes* P = nullptr;
    if (cudaError_t e = pipe_res(dev, &P)) return e;
    float* carry = reinterpret_cast<float*>(ws + L.carry_off);
    const size_t slot_bytes = (size_t)L.N * L.span * H * TcRecord::bytes;
    if (cudaError_t e = cudaEventRecord(P->fork, s)) return e;
    if (cudaError_t e = cudaStreamWaitEvent(P->side, P->fork, 0)) return e;
    for (int r = 0; r < L.ranges; ++r) {
        const int sl = r % L.ring;
        uint8_t* rec = records + sl * slot_bytes;
        const RangeArgs ra{r * L.span, L.span, carry};
        if (r >= L.ring)
            if (cudaError_t e = cudaStreamWaitEvent(s, P->ho_done[sl], 0)) return e;
        intra<<<(unsigned)(L.N * L.span * H), kIntraThreads, kIntraSmem, s>>>(
            tq, tk, tv, tg, beta, scale, ga, H, cx, L.max_chunks, ra, rec, status);
        if (cudaError_t e = cudaGetLastError()) return e;
        if (cudaError_t e = cudaEventRecord(P->intra_done[sl], s)) return e;
        if (cudaError_t e = cudaStreamWaitEvent(P->side, P->intra_done[sl], 0)) return e;
        ho<<<ho_blocks, ho_threads, ho_smem, P->side>>>(rec, cx, L.max_chunks, ra, s0, ob, sN, H,
                                                          status);
        if (cudaError_t e = cudaGetLastError()) return e;
        if (cudaError_t e = cudaEventRecord(P->ho_done[sl], P->side)) return e;
    }
    if (cudaError_t e = cudaEventRecord(P->join, P->side)) return e;
    return cudaStreamWaitEvent(s, P->join, 0);
}

}  // namespace kda
