// kda_decode.cu -- one decode step of KDA: every sequence advances by one token.
//
// Tokamax "chunk_kda_fwd_design_doc", 9.1.2 (Eq. (1) in its delta-correction form) and
// "KDA Doesn't Care About the Future", "Chunkwise KDA in Broad Strokes" (the recurrent
// form is the one that serves decoding a token at a time):
//   S_bar = Diag(exp g) S;  e = v - S_bar^T k;  S' = S_bar + beta k e^T;  o = scale S'^T q.
// The output is folded so that the state is read and written once:
//   o = scale (S_bar^T q + beta (k . q) e).
//
// One CTA of V * K/64 threads per (sequence, head); thread (j, ks) owns rows 64 ks ..
// 64 ks + 63 of column j of the K x V fp32 state in registers (the warp's loads and stores
// of one row are contiguous); the two dot products are summed over the key slices in
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

template <typename T, int K, int V>
__global__ void __launch_bounds__(V * (K / 64))
kda_decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  const float* __restrict__ g, const float* __restrict__ beta, float scale,
                  GateArgs ga, float* __restrict__ state, T* __restrict__ o, int H) {
    constexpr int KS = K / 64, NT = V * KS;  // KS key slices of 64 rows per column
    __shared__ float sq[K], sk[K], sa[K], red[2][NT / 32], part[2][KS][V];
    const int nh = blockIdx.x, h = nh % H, t = threadIdx.x;
    const int j = t % V, ks = t / V;  // column j, key rows 64 ks .. 64 ks + 63
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
    float* col = state + (size_t)nh * K * V + (size_t)(64 * ks) * V + j;
    const float* kk = sk + 64 * ks;
    const float* qq = sq + 64 * ks;
    const float* aa = sa + 64 * ks;
    float s[64];
    float pred = 0.f, read = 0.f;
#pragma unroll
    for (int d = 0; d < 64; ++d) {
        s[d] = aa[d] * col[(size_t)d * V];
        pred = fmaf(s[d], kk[d], pred);
        read = fmaf(s[d], qq[d], read);
    }
    part[0][ks][j] = pred;
    part[1][ks][j] = read;
    float kq = 0.f;
#pragma unroll 8
    for (int d = 0; d < K; ++d) kq = fmaf(sk[d], sq[d], kq);
    __syncthreads();
    pred = 0.f;
    read = 0.f;
#pragma unroll
    for (int x = 0; x < KS; ++x) {
        pred += part[0][x][j];
        read += part[1][x][j];
    }
    const float e = to_f(v[(size_t)nh * V + j]) - pred;
    const float be = beta[nh] * e;
#pragma unroll
    for (int d = 0; d < 64; ++d) col[(size_t)d * V] = fmaf(be, kk[d], s[d]);
    if (ks == 0) o[(size_t)nh * V + j] = from_f<T>(scale * fmaf(be, kq, read));
}

template <typename T, int K, int V>
cudaError_t launch_decode_typed(const void* q, const void* k, const void* v, const float* g,
                                const float* beta, float scale, const GateArgs& ga, float* state,
                                void* o, int N, int H, cudaStream_t s) {
    kda_decode_kernel<T, K, V><<<(unsigned)N * H, V * (K / 64), 0, s>>>(
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
