// kda_decode.cu -- one decode step of KDA: every sequence advances by one token.
//
// Tokamax "chunk_kda_fwd_design_doc", 9.1.2 (Eq. (1) in its delta-correction form) and
// "KDA Doesn't Care About the Future", "Chunkwise KDA in Broad Strokes" (the recurrent
// form is the one that serves decoding a token at a time):
//   S_bar = Diag(exp g) S;  e = v - S_bar^T k;  S' = S_bar + beta k e^T;  o = scale S'^T q.
// The output is folded so that the state is read and written once:
//   o = scale (S_bar^T q + beta (k . q) e).
//
// One CTA of 256 threads per (sequence, head) (the kernel can also cut V into slices of
// kDecCols columns, each column of the state being updated from its own dot products;
// 64-column slices of 128 threads measured slower, 34.1 against 32.3 us).  Thread (row
// group rg, column group cg) owns K / RG consecutive key rows of the 4 value columns
// 4 cg .. 4 cg + 3 in registers, read and written as 16-byte vectors (a warp's accesses
// to a row are contiguous); the two dot products are summed over the row groups in
// shared memory.  The step is bound by the state's HBM traffic (2 K V 4 bytes per
// sequence-head).
#include <cuda_bf16.h>

#include "kda_internal.cuh"

namespace kda {

namespace {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

constexpr int kDecThreads = 256;
constexpr int kDecCols = 128;  // value columns per CTA (all of V when V <= 128)

template <typename T, int K, int V>
__global__ void __launch_bounds__(kDecThreads)
kda_decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  const float* __restrict__ g, const float* __restrict__ beta, float scale,
                  GateArgs ga, float* __restrict__ state, T* __restrict__ o, int H) {
    constexpr int VS = V < kDecCols ? V : kDecCols, SPLIT = V / VS;
    constexpr int NT = kDecThreads, CG = VS / 4, RG = NT / CG, RPT = K / RG;
    static_assert(NT % CG == 0 && K % RG == 0 && V % VS == 0, "decode thread layout");
    __shared__ float sq[K], sk[K], sa[K], red[2][NT / 32], part[2][RG][VS];
    const int nh = blockIdx.x / SPLIT, c0 = VS * (blockIdx.x % SPLIT), h = nh % H, t = threadIdx.x;
    const int cg = t % CG, rg = t / CG;  // columns c0 + 4 cg .., rows RPT rg .. RPT rg + RPT - 1
    const size_t vec = (size_t)nh * K;
    // gate (activated in the kernel when asked, Tokamax design doc 9.1.3), decay, and
    // the (optionally L2-normalised) query and key, shared by the CTA
    for (int d = t; d < K; d += NT) {
        sa[d] = expf(gate_log_decay(ga, g[vec + d], h, d, K));
        sq[d] = to_f(q[vec + d]);
        sk[d] = to_f(k[vec + d]);
    }
    __syncthreads();
    if (ga.qk_l2norm) {
        // x / max(||x||_2, 1e-6) along K ("KDAChunkwise", F.normalize with eps 1e-6)
        float pq = 0.f, pk = 0.f;
        for (int d = t; d < K; d += NT) {
            pq = fmaf(sq[d], sq[d], pq);
            pk = fmaf(sk[d], sk[d], pk);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) {
            pq += __shfl_xor_sync(0xffffffffu, pq, o2);
            pk += __shfl_xor_sync(0xffffffffu, pk, o2);
        }
        if ((t & 31) == 0) {
            red[0][t >> 5] = pq;
            red[1][t >> 5] = pk;
        }
        __syncthreads();
        float nq = 0.f, nk = 0.f;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) {
            nq += red[0][w];
            nk += red[1][w];
        }
        const float iq = 1.f / fmaxf(sqrtf(nq), 1e-6f), ik = 1.f / fmaxf(sqrtf(nk), 1e-6f);
        __syncthreads();
        for (int d = t; d < K; d += NT) {
            sq[d] *= iq;
            sk[d] *= ik;
        }
        __syncthreads();
    }
    float4* rows = reinterpret_cast<float4*>(state + (size_t)nh * K * V + (size_t)(RPT * rg) * V + c0) + cg;
    const int d0 = RPT * rg;
    float4 s[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) s[r] = rows[(size_t)r * (V / 4)];  // all loads issued first
    float pred[4] = {0.f, 0.f, 0.f, 0.f}, rd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const float a = sa[d0 + r], kd = sk[d0 + r], qd = sq[d0 + r];
        s[r].x *= a;
        s[r].y *= a;
        s[r].z *= a;
        s[r].w *= a;
        pred[0] = fmaf(s[r].x, kd, pred[0]);
        pred[1] = fmaf(s[r].y, kd, pred[1]);
        pred[2] = fmaf(s[r].z, kd, pred[2]);
        pred[3] = fmaf(s[r].w, kd, pred[3]);
        rd[0] = fmaf(s[r].x, qd, rd[0]);
        rd[1] = fmaf(s[r].y, qd, rd[1]);
        rd[2] = fmaf(s[r].z, qd, rd[2]);
        rd[3] = fmaf(s[r].w, qd, rd[3]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        part[0][rg][4 * cg + c] = pred[c];
        part[1][rg][4 * cg + c] = rd[c];
    }
    float kq = 0.f;
#pragma unroll 8
    for (int d = 0; d < K; ++d) kq = fmaf(sk[d], sq[d], kq);
    __syncthreads();
    float be[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float p = 0.f, x = 0.f;
#pragma unroll
        for (int w = 0; w < RG; ++w) {
            p += part[0][w][4 * cg + c];
            x += part[1][w][4 * cg + c];
        }
        pred[c] = p;
        rd[c] = x;
        be[c] = beta[nh] * (to_f(v[(size_t)nh * V + c0 + 4 * cg + c]) - p);
    }
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const float kd = sk[d0 + r];
        rows[(size_t)r * (V / 4)] = make_float4(fmaf(be[0], kd, s[r].x), fmaf(be[1], kd, s[r].y),
                                           fmaf(be[2], kd, s[r].z), fmaf(be[3], kd, s[r].w));
    }
    if (rg == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            o[(size_t)nh * V + c0 + 4 * cg + c] = from_f<T>(scale * fmaf(be[c], kq, rd[c]));
    }
}

template <typename T, int K, int V>
cudaError_t launch_decode_typed(const void* q, const void* k, const void* v, const float* g,
                                const float* beta, float scale, const GateArgs& ga, float* state,
                                void* o, int N, int H, cudaStream_t s) {
    constexpr int split = V < kDecCols ? 1 : V / kDecCols;
    kda_decode_kernel<T, K, V><<<(unsigned)N * H * split, kDecThreads, 0, s>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), g, beta,
        scale, ga, state, static_cast<T*>(o), H);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const void* q, const void* k, const void* v, const float* g,
                          const float* beta, float scale, const GateArgs& ga, float* state,
                          void* o, int N, int H, int K, int V, kda_dtype dt, cudaStream_t s) {
#define KDA_DEC_CASE(T_, K_, V_)                                                              \
    if (K == K_ && V == V_)                                                                   \
        return launch_decode_typed<T_, K_, V_>(q, k, v, g, beta, scale, ga, state, o, N, H, s);
    if (dt == KDA_DTYPE_F32) {
        KDA_DEC_CASE(float, 64, 64)
        KDA_DEC_CASE(float, 64, 128)
        KDA_DEC_CASE(float, 128, 64)
        KDA_DEC_CASE(float, 128, 128)
    } else {
        KDA_DEC_CASE(__nv_bfloat16, 64, 64)
        KDA_DEC_CASE(__nv_bfloat16, 64, 128)
        KDA_DEC_CASE(__nv_bfloat16, 128, 64)
        KDA_DEC_CASE(__nv_bfloat16, 128, 128)
    }
#undef KDA_DEC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
