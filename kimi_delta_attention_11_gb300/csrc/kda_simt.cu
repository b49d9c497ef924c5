// kda_simt.cu -- exact-fp32 path of the chunkwise KDA forward (CUDA cores, no MMA).
//
// Tokamax "chunk_kda_fwd_design_doc", 4.1.4 and 5.1: fp32 input takes an exact
// forward-substitution solve instead of the bf16 Neumann/MMA formulation, for
// numerical comparison.  Two kernels, both sized from the chunk index:
//
//   kda_intra_simt  one CTA per (chunk, head): gate cumsum (9.1.3), L and Aqk with the
//                   decay ratio 2^{G_i - G_j} evaluated per term (9.1.5; the ratio is
//                   never split, so no rebasing is needed), forward substitution for
//                   W = A (D_beta K+) and U = A (D_beta V) (Eq. (6)-(7)), K_bar, the
//                   gated query and the chunk decay gamma^C, all stored as fp32.
//   kda_h_o_simt    one CTA per (sequence, head, 32-wide slice of V): the ordered chunk
//                   recurrence of Eq. (8) with the output of Eq. (9) (4.3.2), the
//                   state slice held in shared memory in fp32.
//
// Columns of the state evolve independently given W, K_bar and gamma (Eq. (8)), which
// is what allows the V slicing of the recurrence.
#include <cuda_bf16.h>

#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <int K, int V>
struct IntraSmem {
    static constexpr int KP = K + 1, VP = V + 1, CP = kChunk + 1;
    static constexpr int q = 0, k = q + kChunk * KP, G = k + kChunk * KP, v = G + kChunk * KP,
                         L = v + kChunk * VP, A = L + kChunk * CP, beta = A + kChunk * CP,
                         floats = beta + kChunk;
    static constexpr size_t bytes = floats * sizeof(float);
};

template <typename Tin, int K, int V>
__global__ void __launch_bounds__(kThreads)
kda_intra_simt(const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
               const float* __restrict__ g, const float* __restrict__ beta, float scale, int H,
               GateArgs ga, const int4* __restrict__ chunk_tab, const int* __restrict__ count,
               float* __restrict__ inter, size_t inter_stride_floats) {
    using S = IntraSmem<K, V>;
    constexpr int C = kChunk, KP = S::KP, VP = S::VP, CP = S::CP;
    extern __shared__ float sm[];
    float* qs = sm + S::q;
    float* ks = sm + S::k;
    float* Gs = sm + S::G;
    float* vs = sm + S::v;
    float* Ls = sm + S::L;
    float* As = sm + S::A;
    float* bs = sm + S::beta;

    const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    if (c >= *count) return;
    const int4 ent = chunk_tab[c];
    const int t0 = ent.y, len = ent.z;

    // Load the chunk; rows past the sequence end read as q = k = v = 0, g = 0, beta = 0,
    // which is an identity step (Tokamax design doc 9.1.7).
    for (int idx = tid; idx < C * K; idx += kThreads) {
        const int r = idx / K, d = idx % K;
        const bool in = r < len;
        const size_t off = ((size_t)(t0 + r) * H + h) * K + d;
        qs[r * KP + d] = in ? to_f32(q[off]) : 0.f;
        ks[r * KP + d] = in ? to_f32(k[off]) : 0.f;
        Gs[r * KP + d] = in ? gate_log_decay(ga, g[off], h, d, K) : 0.f;
    }
    for (int idx = tid; idx < C * V; idx += kThreads) {
        const int r = idx / V, j = idx % V;
        vs[r * VP + j] = r < len ? to_f32(v[((size_t)(t0 + r) * H + h) * V + j]) : 0.f;
    }
    if (tid < C) bs[tid] = tid < len ? beta[(size_t)(t0 + tid) * H + h] : 0.f;
    __syncthreads();
    if (ga.qk_l2norm) {
        // rows of q and k divided by max(||.||_2, 1e-6), one warp per row
        const int warp = tid >> 5, lane = tid & 31;
        for (int r = warp; r < C; r += kThreads / 32) {
            float pq = 0.f, pk = 0.f;
            for (int d = lane; d < K; d += 32) {
                pq = fmaf(qs[r * KP + d], qs[r * KP + d], pq);
                pk = fmaf(ks[r * KP + d], ks[r * KP + d], pk);
            }
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) {
                pq += __shfl_xor_sync(0xffffffffu, pq, o2);
                pk += __shfl_xor_sync(0xffffffffu, pk, o2);
            }
            const float iq = 1.f / fmaxf(sqrtf(pq), 1e-6f), ik = 1.f / fmaxf(sqrtf(pk), 1e-6f);
            for (int d = lane; d < K; d += 32) {
                qs[r * KP + d] *= iq;
                ks[r * KP + d] *= ik;
            }
        }
        __syncthreads();
    }

    // 9.1.3: G^r = log2(e) * sum_{m <= r} g^m within the chunk.
    for (int d = tid; d < K; d += kThreads) {
        float acc = 0.f;
        for (int r = 0; r < C; ++r) {
            acc += Gs[r * KP + d];
            Gs[r * KP + d] = acc * kLog2e;
        }
    }
    __syncthreads();

    // 9.1.5: L[i][j] = beta_i sum_d k_i k_j 2^{G_i - G_j} (j < i),
    //        Aqk[i][j] = scale sum_d q_i k_j 2^{G_i - G_j} (j <= i).
    // The mask is applied before the exponential, so no masked entry is evaluated.
    for (int p = tid; p < C * C; p += kThreads) {
        const int i = p / C, j = p % C;
        float l = 0.f, a = 0.f;
        if (j <= i) {
            const float* Gi = Gs + i * KP;
            const float* Gj = Gs + j * KP;
            const float* ki = ks + i * KP;
            const float* kj = ks + j * KP;
            const float* qi = qs + i * KP;
            for (int d = 0; d < K; ++d) {
                const float e = exp2f(Gi[d] - Gj[d]);
                const float kje = kj[d] * e;
                l = fmaf(ki[d], kje, l);
                a = fmaf(qi[d], kje, a);
            }
        }
        Ls[i * CP + j] = j < i ? bs[i] * l : 0.f;
        As[i * CP + j] = j <= i ? scale * a : 0.f;
    }
    __syncthreads();

    float* rec = inter + ((size_t)c * H + h) * inter_stride_floats;
    float* Wg = rec + SimtRecord::w(K);
    float* Ug = rec + SimtRecord::u(K);
    float* Kbg = rec + SimtRecord::kbar(K, V);
    float* Qgg = rec + SimtRecord::qg(K, V);
    float* Ag = rec + SimtRecord::aqk(K, V);
    float* gam = rec + SimtRecord::gamma(K, V);

    // K_bar^r = k^r 2^{G^C - G^r}; gated query scale q^r 2^{G^r}; gamma^C = 2^{G^C}.
    for (int idx = tid; idx < C * K; idx += kThreads) {
        const int r = idx / K, d = idx % K;
        const float Gr = Gs[r * KP + d], Gc = Gs[(C - 1) * KP + d];
        Kbg[idx] = ks[r * KP + d] * exp2f(Gc - Gr);
        Qgg[idx] = scale * qs[r * KP + d] * exp2f(Gr);
    }
    for (int d = tid; d < K; d += kThreads) gam[d] = exp2f(Gs[(C - 1) * KP + d]);
    for (int idx = tid; idx < C * C; idx += kThreads) Ag[idx] = As[(idx / C) * CP + idx % C];
    __syncthreads();

    // Right-hand sides D_beta K+ (in the q buffer) and D_beta V (in place).
    for (int idx = tid; idx < C * K; idx += kThreads) {
        const int r = idx / K, d = idx % K;
        qs[r * KP + d] = bs[r] * ks[r * KP + d] * exp2f(Gs[r * KP + d]);
    }
    for (int idx = tid; idx < C * V; idx += kThreads) {
        const int r = idx / V, j = idx % V;
        vs[r * VP + j] *= bs[r];
    }
    __syncthreads();

    // Eq. (6)-(7): X = (I + L)^{-1} B by forward substitution, one column per thread:
    // X[r] = B[r] - sum_{j<r} L[r][j] X[j].
    for (int col = tid; col < K + V; col += kThreads) {
        float* X = col < K ? qs + col : vs + (col - K);
        const int ld = col < K ? KP : VP;
        for (int r = 1; r < C; ++r) {
            float x = X[r * ld];
            const float* Lr = Ls + r * CP;
            for (int j = 0; j < r; ++j) x = fmaf(-Lr[j], X[j * ld], x);
            X[r * ld] = x;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < C * K; idx += kThreads) Wg[idx] = qs[(idx / K) * KP + idx % K];
    for (int idx = tid; idx < C * V; idx += kThreads) Ug[idx] = vs[(idx / V) * VP + idx % V];
}

constexpr int kVT = 32;  // value columns per recurrence CTA

template <int K>
struct HoSmem {
    static constexpr int S = 0, W = S + K * kVT, Qg = W + kChunk * K, Kb = Qg + kChunk * K,
                         A = Kb + kChunk * K, U = A + kChunk * kChunk, Vn = U + kChunk * kVT,
                         gam = Vn + kChunk * kVT, floats = gam + K;
    static constexpr size_t bytes = floats * sizeof(float);
};

template <typename Tout, int K, int V>
__global__ void __launch_bounds__(kThreads)
kda_h_o_simt(const float* __restrict__ inter, size_t inter_stride_floats,
             const int4* __restrict__ chunk_tab, const int2* __restrict__ seq_tab,
             long long max_chunks, const float* __restrict__ s0, Tout* __restrict__ o,
             float* __restrict__ sN, int H, int* __restrict__ status) {
    using SM = HoSmem<K>;
    constexpr int C = kChunk, NVS = V / kVT;
    extern __shared__ float sm[];
    float* Ss = sm + SM::S;    // [K][kVT]
    float* Ws = sm + SM::W;    // [C][K]
    float* Qs = sm + SM::Qg;   // [C][K]
    float* Kb = sm + SM::Kb;   // [C][K]
    float* As = sm + SM::A;    // [C][C]
    float* Us = sm + SM::U;    // [C][kVT]
    float* Vn = sm + SM::Vn;   // [C][kVT]
    float* gs = sm + SM::gam;  // [K]

    const int vs = blockIdx.x % NVS;
    const int h = (blockIdx.x / NVS) % H;
    const int n = blockIdx.x / (NVS * H);
    const int tid = threadIdx.x, col = tid % kVT, grp = tid / kVT;  // 8 groups of 32
    const size_t st_off = ((size_t)n * H + h) * K * V + vs * kVT;

    for (int idx = tid; idx < K * kVT; idx += kThreads) {
        const int d = idx / kVT, j = idx % kVT;
        Ss[idx] = s0 ? s0[st_off + (size_t)d * V + j] : 0.f;
    }
    const int2 sq = seq_tab[n];
    for (int ci = 0; ci < sq.y; ++ci) {
        const long long c = (long long)sq.x + ci;
        if (c >= max_chunks) {  // inconsistent cu_seqlens: stop rather than overrun
            if (tid == 0) atomicCAS(status, 0, (int)KDA_ERR_INVALID_ARG);
            break;
        }
        const int4 ent = chunk_tab[c];
        const int t0 = ent.y, len = ent.z;
        const float* rec = inter + ((size_t)c * H + h) * inter_stride_floats;
        __syncthreads();  // previous chunk's readers are done with the tiles
        {
            float4* dW = reinterpret_cast<float4*>(Ws);
            float4* dQ = reinterpret_cast<float4*>(Qs);
            float4* dK = reinterpret_cast<float4*>(Kb);
            float4* dA = reinterpret_cast<float4*>(As);
            const float4* sW = reinterpret_cast<const float4*>(rec + SimtRecord::w(K));
            const float4* sQ = reinterpret_cast<const float4*>(rec + SimtRecord::qg(K, V));
            const float4* sK = reinterpret_cast<const float4*>(rec + SimtRecord::kbar(K, V));
            const float4* sA = reinterpret_cast<const float4*>(rec + SimtRecord::aqk(K, V));
            for (int i = tid; i < C * K / 4; i += kThreads) {
                dW[i] = sW[i];
                dQ[i] = sQ[i];
                dK[i] = sK[i];
            }
            for (int i = tid; i < C * C / 4; i += kThreads) dA[i] = sA[i];
            const float* sU = rec + SimtRecord::u(K) + vs * kVT;
            for (int i = tid; i < C * kVT; i += kThreads) Us[i] = sU[(i / kVT) * V + i % kVT];
            const float* sg = rec + SimtRecord::gamma(K, V);
            for (int d = tid; d < K; d += kThreads) gs[d] = sg[d];
        }
        __syncthreads();

        // Eq. (8)/(9) prerequisites: V_new = U - W S (rows grp*8 .. grp*8+7).
        float wsum[8], qsum[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) wsum[m] = qsum[m] = 0.f;
        for (int d = 0; d < K; ++d) {
            const float sd = Ss[d * kVT + col];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int i = grp * 8 + m;
                wsum[m] = fmaf(Ws[i * K + d], sd, wsum[m]);
                qsum[m] = fmaf(Qs[i * K + d], sd, qsum[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int i = grp * 8 + m;
            Vn[i * kVT + col] = Us[i * kVT + col] - wsum[m];
        }
        __syncthreads();

        // Eq. (9): O = (Gamma . Q~) S + Aqk V_new, stored for rows < len.
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int i = grp * 8 + m;
            float acc = qsum[m];
            for (int j = 0; j <= i; ++j) acc = fmaf(As[i * C + j], Vn[j * kVT + col], acc);
            if (i < len) store_out(&o[((size_t)(t0 + i) * H + h) * V + vs * kVT + col], acc);
        }

        // Eq. (8): S <- Diag(gamma^C) S + K_bar^T V_new (key rows grp*16 .. grp*16+15).
        constexpr int RPG = K / 8;
        float upd[RPG];
#pragma unroll
        for (int m = 0; m < RPG; ++m) upd[m] = 0.f;
        for (int j = 0; j < C; ++j) {
            const float vj = Vn[j * kVT + col];
#pragma unroll
            for (int m = 0; m < RPG; ++m) upd[m] = fmaf(Kb[j * K + grp * RPG + m], vj, upd[m]);
        }
#pragma unroll
        for (int m = 0; m < RPG; ++m) {
            const int d = grp * RPG + m;
            Ss[d * kVT + col] = fmaf(gs[d], Ss[d * kVT + col], upd[m]);
        }
    }
    __syncthreads();
    if (sN) {
        for (int idx = tid; idx < K * kVT; idx += kThreads) {
            const int d = idx / kVT, j = idx % kVT;
            sN[st_off + (size_t)d * V + j] = Ss[idx];
        }
    }
}

template <typename T, int K, int V>
cudaError_t launch_typed(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, float scale, const GateArgs& ga, const float* s0,
                         void* o, float* sN, int H, const Layout& L, char* ws, cudaStream_t s,
                         void* const* ev) {
    const size_t stride = L.inter_stride / sizeof(float);
    float* inter = reinterpret_cast<float*>(ws + L.inter_off);
    const int4* ctab = reinterpret_cast<const int4*>(ws + L.chunk_tab_off);
    const int2* stab = reinterpret_cast<const int2*>(ws + L.seq_tab_off);
    const int* count = reinterpret_cast<const int*>(ws + L.count_off);
    int* status = reinterpret_cast<int*>(ws + L.status_off);
    if (L.max_chunks > 0) {
        auto* kin = kda_intra_simt<T, K, V>;
        constexpr size_t smem = IntraSmem<K, V>::bytes;
        cudaFuncSetAttribute(kin, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        dim3 grid((unsigned)L.max_chunks, (unsigned)H);
        kin<<<grid, kThreads, smem, s>>>(static_cast<const T*>(q), static_cast<const T*>(k),
                                         static_cast<const T*>(v), g, beta, scale, H, ga, ctab,
                                         count, inter, stride);
        if (cudaError_t e = cudaGetLastError()) return e;
    }
    if (!record_event(ev, 0, s)) return cudaErrorInvalidResourceHandle;
    if (L.N > 0) {
        auto* kho = kda_h_o_simt<T, K, V>;
        constexpr size_t smem = HoSmem<K>::bytes;
        cudaFuncSetAttribute(kho, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        const unsigned blocks = (unsigned)L.N * H * (V / kVT);
        kho<<<blocks, kThreads, smem, s>>>(inter, stride, ctab, stab, L.max_chunks, s0,
                                           static_cast<T*>(o), sN, H, status);
        if (cudaError_t e = cudaGetLastError()) return e;
    }
    if (!record_event(ev, 1, s)) return cudaErrorInvalidResourceHandle;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_simt(const void* q, const void* k, const void* v, const float* g,
                        const float* beta, float scale, const GateArgs& ga, const float* s0,
                        void* o, float* sN, int H, int K, int V, kda_dtype dt, const Layout& L,
                        char* ws, cudaStream_t s, void* const* ev) {
#define KDA_SIMT_CASE(T_, K_, V_)                                                               \
    if (K == K_ && V == V_)                                                                     \
        return launch_typed<T_, K_, V_>(q, k, v, g, beta, scale, ga, s0, o, sN, H, L, ws, s, ev);
    if (dt == KDA_DTYPE_F32) {
        KDA_SIMT_CASE(float, 64, 64)
        KDA_SIMT_CASE(float, 64, 128)
        KDA_SIMT_CASE(float, 128, 64)
        KDA_SIMT_CASE(float, 128, 128)
    } else {
        KDA_SIMT_CASE(__nv_bfloat16, 64, 64)
        KDA_SIMT_CASE(__nv_bfloat16, 64, 128)
        KDA_SIMT_CASE(__nv_bfloat16, 128, 64)
        KDA_SIMT_CASE(__nv_bfloat16, 128, 128)
    }
#undef KDA_SIMT_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
