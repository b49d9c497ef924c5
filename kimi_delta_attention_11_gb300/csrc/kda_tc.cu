// kda_tc.cu -- bf16 tensor-core path of the chunkwise KDA forward (K = V = 128, C = 64).
//
//   kda_intra_tc  one CTA (8 warps) per (chunk, head), fed by TMA:
//     a1  q, k, v (bf16) and g (fp32) tiles by TMA, rows past the sequence end zeroed;
//     a2  gate cumsum G = log2(e) * cumsum(g) within the chunk (Tokamax design doc 9.1.3);
//     a3  Aqk and L by tcgen05 MMAs ("KDA Doesn't Care About the Future", "The rebasing
//         trick", "Sixteen keys, sixty-four queries"): for the 16-row block b of queries
//         the gate ratio 2^{G_i - G_j} is split at the block's first row G_{16b} into a
//         query factor 2^{G_i - G_{16b}} <= 1 and a key factor 2^{G_{16b} - G_j} (at most
//         2^108 at the -5 gate bound, so finite).  The reference is causal: it depends on
//         no later token.  Keys are the MMA's M side (R_b: 64 key rows rebased for query
//         block b, stacked in pairs to M = 128) and the 16 query rows and 16 beta-scaled key
//         rows of the block the N side (N = 64 for a pair of blocks);
//     a4  (I + L)^{-1} by blocked forward substitution in fp32 (16 x 16 diagonal blocks,
//         then three levels of block products), then W = A (D_beta K+) and U = A (D_beta V)
//         by one M = 128 x N = 256 x K = 64 tcgen05 MMA (Tokamax design doc Eq. (6)-(7));
//         K_bar = k 2^{G_C - G} and the gated query scale q 2^{G} (9.1.5);
//     results are written as the record of TcRecord (shared-memory images of tcgen05
//     operands) for the recurrence kernel.
//   kda_h_o_tc    one CTA (4 epilogue warps + 1 producer/MMA warp) per (sequence, head,
//     32-column slice of V), the ordered chunk recurrence (Eq. (8)) fused with the output
//     (Eq. (9)); records double-buffered by bulk copies; the state slice is held in fp32
//     registers (one key row per thread) and fed to the tensor core as bf16:
//       MMA1  D1 = [W ; Qg] S               (M 128, N 32, K 128)
//       ep1   V_new = U - W S               (rows 0-63 of D1)
//       MMA2  D1 += [K_bar^T(64..127) ; Aqk] V_new   (rows 64-127: O = Qg S + Aqk V_new)
//       MMA3  D3 = K_bar^T V_new           (M 128 keys, N 32, K 64)
//       ep2   O stored; S = Diag(gamma^C) S + D3.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {

namespace {

using namespace sm100;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kIntraThreads = 256;

// ---------------------------------------------------------------------------
// intra-chunk kernel
// ---------------------------------------------------------------------------

// shared-memory map (offsets from a 1024-aligned base)
struct IntraMap {
    static constexpr uint32_t QT = 0;          // q tile: 2 panels [64][64] bf16 (TMA)
    static constexpr uint32_t KT = 16384;      // k tile
    static constexpr uint32_t VT = 32768;      // v tile
    static constexpr uint32_t GT = 49152;      // g -> G, fp32 [64][128] (TMA)
    static constexpr uint32_t RA = 81920;      // relation A: group p, panel P at (2p+P)*16K
    static constexpr uint32_t RB = 147456;     // relation B: group p, panel P at (2p+P)*8K
    static constexpr uint32_t WB = 180224;     // W/U B operand: [256 rows][64 tok]
    static constexpr uint32_t MISC = 212992;   // beta[64], P0[4][128], X[6][128], tot[128]
    static constexpr uint32_t END = MISC + 256 + 2048 + 3072 + 512;
    // reuse after the relation MMA has completed (inside RA .. WB)
    static constexpr uint32_t LF = RA;              // L fp32 [64][64]
    static constexpr uint32_t AF = RA + 16384;      // Aqk fp32 [64][64]
    static constexpr uint32_t IF = RA + 32768;      // (I+L)^-1 fp32 [64][64]
    static constexpr uint32_t TS = RA + 49152;      // solve scratch [3][16][16] fp32
    static constexpr uint32_t AIA = RB;             // (I+L)^-1 bf16 A operand [128][64]
    static constexpr uint32_t WST = RB + 16384;     // W staging: 2 panels [64][64]
    static constexpr uint32_t UST = WB;             // U staging (after the W/U MMA)
};
constexpr size_t kIntraSmem = IntraMap::END + 1024;  // + alignment slack

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

__device__ __forceinline__ float bf16_at(const uint8_t* base, uint32_t off) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(base + off));
}

// index of the (b, b') pair, b' < b, in X
__device__ __forceinline__ int pair_index(int b, int bp) { return b * (b - 1) / 2 + bp; }

__global__ void __launch_bounds__(kIntraThreads, 1)
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
    float* Gf = reinterpret_cast<float*>(sm + M::GT);
    float* betas = reinterpret_cast<float*>(sm + M::MISC);
    float* P0 = betas + 64;   // [4][128]  2^{G_{16b}}
    float* X = P0 + 512;      // [6][128]  2^{G_{16b} - G_{16b'}}, b' < b
    float* tot = X + 768;     // [128]     cumsum of rows 0-31
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

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
        tma_load_2d(sm + M::QT, &tm_q, h * 128, t0, &bar_tma);
        tma_load_2d(sm + M::QT + 8192, &tm_q, h * 128 + 64, t0, &bar_tma);
        tma_load_2d(sm + M::KT, &tm_k, h * 128, t0, &bar_tma);
        tma_load_2d(sm + M::KT + 8192, &tm_k, h * 128 + 64, t0, &bar_tma);
        tma_load_2d(sm + M::VT, &tm_v, h * 128, t0, &bar_tma);
        tma_load_2d(sm + M::VT + 8192, &tm_v, h * 128 + 64, t0, &bar_tma);
        tma_load_2d(sm + M::GT, &tm_g, h * 128, t0, &bar_tma);
    }
    if (tid < 64) betas[tid] = tid < len ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
    mbar_wait_abortable(&bar_tma, 0, status, abort_flag);
    __syncthreads();
    if (*abort_flag) goto teardown;

    // rows at or past len belong to the next sequence: q = k = v = 0, g = 0 there, an
    // identity step (Tokamax design doc 9.1.7)
    if (len < 64) {
        for (int idx = tid; idx < (64 - len) * 8; idx += kIntraThreads) {
            const int r = len + idx / 8, ch = idx % 8;
            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int P = 0; P < 2; ++P) {
                st_shared_u4(sb + M::QT + P * 8192 + r * 128 + ch * 16, z);
                st_shared_u4(sb + M::KT + P * 8192 + r * 128 + ch * 16, z);
                st_shared_u4(sb + M::VT + P * 8192 + r * 128 + ch * 16, z);
            }
        }
        for (int idx = tid; idx < (64 - len) * 128; idx += kIntraThreads) Gf[len * 128 + idx] = 0.f;
        __syncthreads();
    }

    // a2: G = log2(e) * inclusive cumsum of g over the chunk, per key channel
    {
        const int d = tid & 127, half = tid >> 7;
        float x[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) x[r] = Gf[(half * 32 + r) * 128 + d];
#pragma unroll
        for (int r = 1; r < 32; ++r) x[r] += x[r - 1];
        if (half == 0) tot[d] = x[31];
        __syncthreads();
        const float base = half ? tot[d] : 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) Gf[(half * 32 + r) * 128 + d] = (x[r] + base) * kLog2e;
        __syncthreads();
    }

    // block factors and the chunk decay gamma^C = 2^{G_63}
    for (int idx = tid; idx < 11 * 128; idx += kIntraThreads) {
        const int f = idx >> 7, d = idx & 127;
        if (f < 4) {
            P0[f * 128 + d] = exp2f(Gf[(16 * f) * 128 + d]);
        } else if (f < 10) {
            const int pi = f - 4;  // (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
            const int b = pi < 1 ? 1 : (pi < 3 ? 2 : 3);
            const int bp = pi - pair_index(b, 0);
            X[pi * 128 + d] = exp2f(Gf[(16 * b) * 128 + d] - Gf[(16 * bp) * 128 + d]);
        } else {
            reinterpret_cast<float*>(rec + TcRecord::gamma)[d] = exp2f(Gf[63 * 128 + d]);
        }
    }
    __syncthreads();

    // a3 operands.  Relation B (queries): row (b&1)*32 + (i&15) = scale q_i 2^{G_i-G_16b},
    // row +16 = beta_i k_i 2^{G_i-G_16b}, group b>>1.  Same pass: the gated query
    // Qg = scale q_i 2^{G_i} goes straight to the record.
    for (int u = tid; u < 1024; u += kIntraThreads) {
        const int i = u >> 4, dc = u & 15, b = i >> 4, P = dc >> 3, cc = dc & 7;
        float qv[8], kv[8], e[8], qs[8], ks[8], qg[8];
        unpack8(*reinterpret_cast<const uint4*>(sm + M::QT + P * 8192 + sw128_chunk(i, cc)), qv);
        unpack8(*reinterpret_cast<const uint4*>(sm + M::KT + P * 8192 + sw128_chunk(i, cc)), kv);
        const float bi = betas[i];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int d = dc * 8 + m;
            e[m] = exp2f(Gf[i * 128 + d] - Gf[(16 * b) * 128 + d]);
            qs[m] = scale * qv[m] * e[m];
            ks[m] = bi * kv[m] * e[m];
            qg[m] = qs[m] * P0[b * 128 + d];
        }
        const int row = (b & 1) * 32 + (i & 15);
        const uint32_t base = sb + M::RB + ((b >> 1) * 2 + P) * 8192;
        st_shared_u4(base + sw128_chunk(row, cc), pack8(qs));
        st_shared_u4(base + sw128_chunk(row + 16, cc), pack8(ks));
        *reinterpret_cast<uint4*>(rec + TcRecord::wq + P * 16384 + 8192 + sw128_chunk(i, cc)) =
            pack8(qg);
    }
    // Relation A (keys): R_b[j] = k_j 2^{G_16b - G_j} for every query block b >= block(j);
    // rows of keys after block b are never read unmasked and are left unwritten.
    for (int u = tid; u < 1024; u += kIntraThreads) {
        const int j = u >> 4, dc = u & 15, bj = j >> 4, P = dc >> 3, cc = dc & 7;
        float kv[8], r0[8], rb[8];
        unpack8(*reinterpret_cast<const uint4*>(sm + M::KT + P * 8192 + sw128_chunk(j, cc)), kv);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int d = dc * 8 + m;
            r0[m] = kv[m] * exp2f(Gf[(16 * bj) * 128 + d] - Gf[j * 128 + d]);
        }
        for (int b = bj; b < 4; ++b) {
#pragma unroll
            for (int m = 0; m < 8; ++m)
                rb[m] = b == bj ? r0[m] : r0[m] * X[pair_index(b, bj) * 128 + dc * 8 + m];
            const uint32_t base = sb + M::RA + ((b >> 1) * 2 + P) * 16384;
            st_shared_u4(base + sw128_chunk((b & 1) * 64 + j, cc), pack8(rb));
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // relation MMAs: group p -> TMEM columns [64p, 64p+64)
    if (tid == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(128, 64);
        for (int p = 0; p < 2; ++p)
            for (int ks = 0; ks < 8; ++ks) {
                const int P = ks >> 2, kk = ks & 3;
                const uint64_t ad = desc_sw128(sb + M::RA + (p * 2 + P) * 16384 + kk * 32);
                const uint64_t bd = desc_sw128(sb + M::RB + (p * 2 + P) * 8192 + kk * 32);
                mma_bf16(tmem + 64 * p, ad, bd, idesc, ks > 0 ? 1u : 0u);
            }
        mma_commit(&bar_rel);
    }

    // meanwhile: K_bar^T [d][j] = k_j 2^{G_63 - G_j} to the record, (D_beta K+)^T [d][j] =
    // beta_j k_j 2^{G_j} and (D_beta V)^T [v][j] into the W/U B operand
    for (int u = tid; u < 1024; u += kIntraThreads) {
        const int d = u >> 3, tc = u & 7, P = d >> 6, dd = d & 63;
        const float g63 = Gf[63 * 128 + d];
        float kb[8], kp[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int j = tc * 8 + m;
            const float kv = bf16_at(sm + M::KT + P * 8192, sw128_offset(j, dd));
            const float gj = Gf[j * 128 + d];
            kb[m] = kv * exp2f(g63 - gj);
            kp[m] = betas[j] * kv * exp2f(gj);
        }
        *reinterpret_cast<uint4*>(rec + TcRecord::kbarT + sw128_chunk(d, tc)) = pack8(kb);
        st_shared_u4(sb + M::WB + sw128_chunk(d, tc), pack8(kp));
    }
    for (int u = tid; u < 1024; u += kIntraThreads) {
        const int vc = u >> 3, tc = u & 7, P = vc >> 6, vv = vc & 63;
        float vb[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int j = tc * 8 + m;
            vb[m] = betas[j] * bf16_at(sm + M::VT + P * 8192, sw128_offset(j, vv));
        }
        st_shared_u4(sb + M::WB + sw128_chunk(128 + vc, tc), pack8(vb));
    }
    fence_proxy_async_smem();

    // relation epilogue: lane L of TMEM = key j (L < 64: block 2p, L >= 64: block 2p+1);
    // columns: 16 query rows (Aqk^T), then 16 beta-scaled key rows (L^T) of that block
    mbar_wait_abortable(&bar_rel, 0, status, abort_flag);
    tc_fence_after();
    __syncthreads();
    if (*abort_flag) goto teardown;
    {
        float* LF = reinterpret_cast<float*>(sm + M::LF);
        float* AF = reinterpret_cast<float*>(sm + M::AF);
        if (warp < 4) {
            const int L = warp * 32 + lane, j = L & 63, hi = L >> 6;
            for (int p = 0; p < 2; ++p) {
                float v[32];
                tmem_ld32(tmem_addr(tmem, warp, 64 * p + 32 * hi), v);
                const int b = 2 * p + hi;
#pragma unroll
                for (int ci = 0; ci < 16; ++ci) {
                    const int i = 16 * b + ci;
                    AF[i * 64 + j] = j <= i ? v[ci] : 0.f;
                    LF[i * 64 + j] = j < i ? v[16 + ci] : 0.f;
                }
            }
        }
        float* IF = reinterpret_cast<float*>(sm + M::IF);
        for (int idx = tid; idx < 4096; idx += kIntraThreads) IF[idx] = 0.f;
        tc_fence_before();
        __syncthreads();

        // Aqk (bf16) to the record
        for (int u = tid; u < 512; u += kIntraThreads) {
            const int i = u >> 3, jc = u & 7;
            float a[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) a[m] = AF[i * 64 + jc * 8 + m];
            *reinterpret_cast<uint4*>(rec + TcRecord::aqk + sw128_chunk(i, jc)) = pack8(a);
        }

        // a4: (I + L)^{-1}.  Diagonal 16x16 blocks by forward substitution, one column per
        // thread: x_r = delta_rc - sum_{m<r} L[r][m] x_m.
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
        // off-diagonal blocks, by distance l = i - j:
        //   Ainv_ij = - D_i sum_{k=j}^{i-1} L_ik Ainv_kj   (D_i = Ainv_ii)
        float* TS = reinterpret_cast<float*>(sm + M::TS);
        for (int l = 1; l <= 3; ++l) {
            const int nt = 4 - l;
            for (int e = tid; e < nt * 256; e += kIntraThreads) {
                const int t = e >> 8, r = (e >> 4) & 15, cc = e & 15, i = l + t, j = i - l;
                float acc = 0.f;
                for (int kb = j; kb < i; ++kb)
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        acc = fmaf(LF[(16 * i + r) * 64 + 16 * kb + m],
                                   IF[(16 * kb + m) * 64 + 16 * j + cc], acc);
                TS[t * 256 + r * 16 + cc] = acc;
            }
            __syncthreads();
            for (int e = tid; e < nt * 256; e += kIntraThreads) {
                const int t = e >> 8, r = (e >> 4) & 15, cc = e & 15, i = l + t, j = i - l;
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    acc = fmaf(IF[(16 * i + r) * 64 + 16 * i + m], TS[t * 256 + m * 16 + cc], acc);
                IF[(16 * i + r) * 64 + 16 * j + cc] = -acc;
            }
            __syncthreads();
        }
        // (I+L)^{-1} as the bf16 A operand of the W/U product (rows 64-127 unused)
        for (int u = tid; u < 512; u += kIntraThreads) {
            const int r = u >> 3, jc = u & 7;
            float a[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) a[m] = IF[r * 64 + jc * 8 + m];
            st_shared_u4(sb + M::AIA + sw128_chunk(r, jc), pack8(a));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    }

    // [W | U] = (I+L)^{-1} [D_beta K+ | D_beta V]: M 128 (tokens, 64 used), N 256, K 64
    if (tid == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(128, 256);
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tmem, desc_sw128(sb + M::AIA + kk * 32), desc_sw128(sb + M::WB + kk * 32), idesc,
                     kk > 0 ? 1u : 0u);
        mma_commit(&bar_wu);
    }
    mbar_wait_abortable(&bar_wu, 0, status, abort_flag);
    tc_fence_after();
    __syncthreads();
    if (*abort_flag) goto teardown;

    // W rows (warps 0,1) into the staging image of record rows 0-63 of both panels;
    // U rows (warps 4,5) into the staging image of the U block
    if (warp == 0 || warp == 1) {
        const int r = warp * 32 + lane;
        for (int cb = 0; cb < 4; ++cb) {
            float v[32];
            tmem_ld32(tmem_addr(tmem, warp, 32 * cb), v);
            const uint32_t base = sb + M::WST + (cb >> 1) * 8192;
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                float f[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) f[m] = v[qd * 8 + m];
                st_shared_u4(base + sw128_chunk(r, (cb & 1) * 4 + qd), pack8(f));
            }
        }
    } else if (warp == 4 || warp == 5) {
        const int r = (warp - 4) * 32 + lane;
        for (int s = 0; s < 4; ++s) {
            float v[32];
            tmem_ld32(tmem_addr(tmem, warp, 128 + 32 * s), v);
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                float f[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) f[m] = v[qd * 8 + m];
                st_shared_u4(sb + M::UST + s * 4096 + r * 64 + ((qd ^ (r & 3)) << 4), pack8(f));
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

constexpr int kVT = 32;                 // value columns per CTA
constexpr int kHoThreads = 160;         // 4 epilogue warps + 1 producer/MMA warp
constexpr uint32_t kStageBytes = 62464; // WQ 32K | K_bar^T + Aqk 24K | U slice 4K | gamma 512
constexpr uint32_t kStTx = 32768 + 24576 + 4096 + 512;

struct HoMap {
    static constexpr uint32_t STAGE0 = 0;
    static constexpr uint32_t ST = 2 * kStageBytes;   // S^T bf16: 2 panels [32][64] (4 KB each)
    static constexpr uint32_t VN = ST + 8192;         // V_new^T bf16: [32][64]
    static constexpr uint32_t END = VN + 4096;
    // inside a stage
    static constexpr uint32_t WQ = 0, KA = 32768, U = 57344, GAM = 61440;
};
constexpr size_t kHoSmem = HoMap::END + 1024;

__global__ void __launch_bounds__(kHoThreads, 1)
kda_h_o_tc(const uint8_t* __restrict__ records, const int4* __restrict__ chunk_tab,
           const int2* __restrict__ seq_tab, long long max_chunks, const float* __restrict__ s0,
           __nv_bfloat16* __restrict__ o, float* __restrict__ sN, int H,
           int* __restrict__ status) {
    using M = HoMap;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[2], empty[2], s_ready, vnew_ready, mma1_done, mma23_done;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    const int slice = blockIdx.x & 3;
    const int h = (blockIdx.x >> 2) % H;
    const int n = (blockIdx.x >> 2) / H;
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

    if (warp == 0) tmem_alloc(&tmem_base, 64);
    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 128);
        }
        mbar_init(&s_ready, 128);
        mbar_init(&vnew_ready, 64);
        mbar_init(&mma1_done, 1);
        mbar_init(&mma23_done, 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base, D1 = tmem, D3 = tmem + 32;
    volatile int* abort_flag = &s_abort;
    const size_t st_off = ((size_t)n * H + h) * 128 * 128 + slice * kVT;

    if (warp == 4) {
        // producer + MMA issuer (one thread)
        if (lane == 0) {
            auto load = [&](int ci) {
                const long long cg = first + ci;
                const uint8_t* rec = records + ((size_t)cg * H + h) * TcRecord::bytes;
                uint8_t* st = sm + (ci & 1) * kStageBytes;
                mbar_arrive_expect_tx(&full[ci & 1], kStTx);
                bulk_load(st + M::WQ, rec + TcRecord::wq, 32768, &full[ci & 1]);
                bulk_load(st + M::KA, rec + TcRecord::kbarT, 24576, &full[ci & 1]);
                bulk_load(st + M::U, rec + TcRecord::u + slice * 4096, 4096, &full[ci & 1]);
                bulk_load(st + M::GAM, rec + TcRecord::gamma, 512, &full[ci & 1]);
            };
            for (int ci = 0; ci < 2 && ci < nch; ++ci) load(ci);
            const uint32_t idesc = idesc_bf16(128, kVT);
            for (int ci = 0; ci < nch; ++ci) {
                const uint32_t stb = sb + (ci & 1) * kStageBytes;
                if (!mbar_wait_abortable(&full[ci & 1], (ci >> 1) & 1, status, abort_flag)) break;
                if (!mbar_wait_abortable(&s_ready, ci & 1, status, abort_flag)) break;
                tc_fence_after();
                // MMA1: D1 = [W ; Qg] S   (K = 128 keys over two panels)
                for (int ks = 0; ks < 8; ++ks) {
                    const int P = ks >> 2, kk = ks & 3;
                    mma_bf16(D1, desc_sw128(stb + M::WQ + P * 16384 + kk * 32),
                             desc_sw128(sb + M::ST + P * 4096 + kk * 32), idesc, ks > 0 ? 1u : 0u);
                }
                mma_commit(&mma1_done);
                if (!mbar_wait_abortable(&vnew_ready, ci & 1, status, abort_flag)) break;
                tc_fence_after();
                // MMA2: D1 += [K_bar^T rows 64-127 ; Aqk] V_new ; MMA3: D3 = K_bar^T V_new
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(D1, desc_sw128(stb + M::KA + 8192 + kk * 32),
                             desc_sw128(sb + M::VN + kk * 32), idesc, 1u);
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(D3, desc_sw128(stb + M::KA + kk * 32), desc_sw128(sb + M::VN + kk * 32),
                             idesc, kk > 0 ? 1u : 0u);
                mma_commit(&mma23_done);
                if (ci + 2 < nch) {
                    if (!mbar_wait_abortable(&empty[ci & 1], (ci >> 1) & 1, status, abort_flag)) break;
                    load(ci + 2);
                }
            }
        }
        __syncwarp();
    } else {
        // epilogue warps: thread d = tid owns key row d of the state slice (fp32)
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
        auto write_state = [&]() {  // S^T tile: element (v, d) of [32 rows v][128 keys d]
            uint8_t* pan = sm + M::ST + (d >> 6) * 4096;
#pragma unroll
            for (int x = 0; x < kVT; ++x)
                *reinterpret_cast<__nv_bfloat16*>(pan + sw128_offset(x, d & 63)) =
                    __float2bfloat16_rn(S[x]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&s_ready);
        };
        write_state();
        for (int ci = 0; ci < nch; ++ci) {
            const uint8_t* st = sm + (ci & 1) * kStageBytes;
            const int4 ent = chunk_tab[first + ci];
            const int t0 = ent.y, len = ent.z;
            if (!mbar_wait_abortable(&mma1_done, ci & 1, status, abort_flag)) break;
            tc_fence_after();
            if (warp < 2) {
                // ep1: V_new[i] = U[i] - (W S)[i], token i = TMEM lane
                const int i = d;
                if (!mbar_wait_abortable(&full[ci & 1], (ci >> 1) & 1, status, abort_flag)) break;
                float ws[32];
                tmem_ld32(tmem_addr(D1, warp, 0), ws);
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                    float uf[8];
                    unpack8(*reinterpret_cast<const uint4*>(st + M::U + i * 64 + ((qd ^ (i & 3)) << 4)),
                            uf);
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const int x = qd * 8 + m;
                        *reinterpret_cast<__nv_bfloat16*>(sm + M::VN + sw128_offset(x, i)) =
                            __float2bfloat16_rn(uf[m] - ws[x]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&vnew_ready);
            }
            if (!mbar_wait_abortable(&mma23_done, ci & 1, status, abort_flag)) break;
            tc_fence_after();
            float ov[32];
            if (warp >= 2) tmem_ld32(tmem_addr(D1, warp, 0), ov);  // O rows (token = lane - 64)
            float upd[32];
            tmem_ld32(tmem_addr(D3, warp, 0), upd);                 // (K_bar^T V_new)[d]
            const float gam = reinterpret_cast<const float*>(st + M::GAM)[d];
#pragma unroll
            for (int x = 0; x < kVT; ++x) S[x] = fmaf(gam, S[x], upd[x]);
            write_state();
            mbar_arrive(&empty[ci & 1]);
            if (warp >= 2) {
                const int i = d - 64;
                if (i < len) {
                    uint4* dst = reinterpret_cast<uint4*>(o + ((size_t)(t0 + i) * H + h) * 128 +
                                                          slice * kVT);
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd) {
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
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
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
        if (!make_tmap_2d(&tq, q, true, inner, rows, inner * 2, 64, 64, true) ||
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
        const unsigned blocks = (unsigned)L.N * H * 4;
        kda_h_o_tc<<<blocks, kHoThreads, kHoSmem, s>>>(records, ctab, stab, L.max_chunks, s0,
                                                       static_cast<__nv_bfloat16*>(o), sN, H, status);
        if (cudaError_t e = cudaGetLastError()) return e;
    }
    if (!record_event(ev, 1, s)) return cudaErrorInvalidResourceHandle;
    return cudaSuccess;
}

}  // namespace kda
