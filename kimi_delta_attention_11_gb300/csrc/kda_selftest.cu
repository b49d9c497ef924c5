// kda_selftest.cu -- diagnostic GEMM through the same tcgen05 / TMA / tensor-memory
// building blocks as the bf16 kernels: D[128][N] = A[128][K] * B[N][K]^T.
// Mode 0 stages A and B by TMA (128-byte swizzle), mode 1 writes them from registers
// with the software swizzle (sw128_offset) that the kernels use for built operands.
// Mode 4 keeps A in tensor memory (written with tcgen05.st, lane m = row m, two bf16 per
// 32-bit column) and stages B by TMA.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {

namespace {

using namespace sm100;

constexpr int kSelfThreads = 128;

__global__ void __launch_bounds__(kSelfThreads)
selftest_mma_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                    const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B,
                    float* __restrict__ D, int N, int K, int mode, uint32_t tmem_cols,
                    int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t bar_full, bar_done;
    __shared__ uint32_t tmem_base;
    // 1024-byte aligned operand area (the dynamic allocation reserves the slack)
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int panels = (K + 63) / 64;
    uint8_t* sa = smem;                                   // panels x [128][64] bf16
    uint8_t* sb = smem + 2 * 128 * 128;                   // B operand (up to 64 KB)
    const int tid = threadIdx.x, warp = tid / 32;

    if (warp == 0) tmem_alloc(&tmem_base, tmem_cols);
    if (tid == 0) {
        mbar_init(&bar_full, 1);
        mbar_init(&bar_done, 1);
        fence_barrier_init();
    }
    if (mode == 1) {
        // software swizzle: element (r, c) of a K-major operand -> panel c/64, sw128_offset
        for (int idx = tid; idx < 128 * K; idx += kSelfThreads) {
            const int r = idx / K, c = idx % K;
            *reinterpret_cast<__nv_bfloat16*>(sa + (c / 64) * 128 * 128 + sw128_offset(r, c % 64)) =
                A[idx];
        }
        for (int idx = tid; idx < N * K; idx += kSelfThreads) {
            const int r = idx / K, c = idx % K;
            *reinterpret_cast<__nv_bfloat16*>(sb + (c / 64) * N * 128 + sw128_offset(r, c % 64)) =
                B[idx];
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    bool ok = true;
    if (mode == 4) {
        // A row m -> TMEM lane m (this thread), columns 256 + k/2 (bf16 pairs)
        const int m = tid;
        for (int c0 = 0; c0 < K / 2; c0 += 8) {
            uint32_t v[8];
            for (int j = 0; j < 8; ++j) {
                const __nv_bfloat16 lo = A[m * K + 2 * (c0 + j)], hi = A[m * K + 2 * (c0 + j) + 1];
                v[j] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
            }
            tmem_st8(tmem_addr(tmem, warp, 256 + c0), v);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    if (tid == 0) {
        if (mode == 0 || mode == 4) {
            mbar_arrive_expect_tx(&bar_full, (uint32_t)(panels * ((mode == 0 ? 128 : 0) + N) * 128));
            for (int p = 0; p < panels; ++p) {
                if (mode == 0) tma_load_2d(sa + p * 128 * 128, &tma_a, p * 64, 0, &bar_full);
                tma_load_2d(sb + p * N * 128, &tma_b, p * 64, 0, &bar_full);
            }
            ok = mbar_wait(&bar_full, 0, status);
        } else if (mode == 2) {  // A K-major panels; B given as [K][N]: N/64 atoms [K][64]
            mbar_arrive_expect_tx(&bar_full, (uint32_t)(panels * 128 * 128 + K * N * 2));
            for (int p = 0; p < panels; ++p) tma_load_2d(sa + p * 128 * 128, &tma_a, p * 64, 0, &bar_full);
            for (int a = 0; a < N / 64; ++a) tma_load_2d(sb + a * K * 128, &tma_b, a * 64, 0, &bar_full);
            ok = mbar_wait(&bar_full, 0, status);
        } else if (mode == 3) {  // A given as [K][128]: 2 atoms [K][64]; B K-major panels
            mbar_arrive_expect_tx(&bar_full, (uint32_t)(K * 128 * 2 + panels * N * 128));
            for (int a = 0; a < 2; ++a) tma_load_2d(sa + a * K * 128, &tma_a, a * 64, 0, &bar_full);
            for (int p = 0; p < panels; ++p) tma_load_2d(sb + p * N * 128, &tma_b, p * 64, 0, &bar_full);
            ok = mbar_wait(&bar_full, 0, status);
        }
        if (ok) {
            tc_fence_after();
            const bool a_mn = mode == 3, b_mn = mode == 2;
            const uint32_t idesc = idesc_bf16(128, (uint32_t)N, a_mn, b_mn);
            for (int ks = 0; ks < K / 16; ++ks) {
                const int p = ks / 4, kk = ks % 4;
                // K-major: panel p, +32 B per K step.  MN-major: atoms of [K rows][64] at a
                // stride of K*128 B, +2048 B (two 8-row groups) per K step.
                const uint64_t ad =
                    a_mn ? desc_sw128_mn(smem_u32(sa + ks * 2048), (uint32_t)K * 128, 1024)
                         : desc_sw128(smem_u32(sa + p * 128 * 128 + kk * 32));
                const uint64_t bd =
                    b_mn ? desc_sw128_mn(smem_u32(sb + ks * 2048), (uint32_t)K * 128, 1024)
                         : desc_sw128(smem_u32(sb + p * N * 128 + kk * 32));
                if (mode == 4)  // A from TMEM: 8 columns (16 bf16) per K step
                    mma_bf16_ta(tmem, tmem + 256 + ks * 8, bd, idesc, ks > 0 ? 1u : 0u);
                else
                    mma_bf16(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
            }
        }
        mma_commit(&bar_done);  // arrives even if nothing was issued
    }
    __syncwarp();
    ok = mbar_wait(&bar_done, 0, status);
    tc_fence_after();
    if (ok) {
        const int row = warp * 32 + (tid % 32);
        for (int c0 = 0; c0 < N; c0 += 32) {
            float v[32];
            tmem_ld32(tmem_addr(tmem, warp, c0), v);
            for (int j = 0; j < 32 && c0 + j < N; ++j) D[row * N + c0 + j] = v[j];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

}  // namespace

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_selftest_umma(const void* A, const void* B, float* D, int N, int K,
                                        int mode, int* status, void* stream) {
    if (!A || !B || !D || !status) return KDA_ERR_INVALID_ARG;
    if (!(N == 16 || N == 32 || N == 64 || N == 128 || N == 256)) return KDA_ERR_UNSUPPORTED;
    if (K < 16 || K > 128 || K % 16 != 0 || mode < 0 || mode > 4) return KDA_ERR_UNSUPPORTED;
    if (mode == 2 && N < 64) return KDA_ERR_UNSUPPORTED;
    CUtensorMap ta, tb;
    const bool a_mn = mode == 3, b_mn = mode == 2;
    const bool ok_a = a_mn ? make_tmap_2d(&ta, A, true, 128, (uint64_t)K, 256, 64, (uint32_t)K, true)
                           : make_tmap_2d(&ta, A, true, (uint64_t)K, 128, (uint64_t)K * 2, 64, 128, true);
    const bool ok_b = b_mn ? make_tmap_2d(&tb, B, true, (uint64_t)N, (uint64_t)K, (uint64_t)N * 2, 64,
                                          (uint32_t)K, true)
                           : make_tmap_2d(&tb, B, true, (uint64_t)K, (uint64_t)N, (uint64_t)K * 2, 64,
                                          (uint32_t)N, true);
    if (!ok_a || !ok_b) return KDA_ERR_CUDA;
    // operand area: both readings of the MN-major offsets stay inside these sizes
    const size_t smem = 2 * 128 * 128 + 256 * 128 * 2 + 1024;
    const uint32_t cols = mode == 4 ? 512u : (N < 32 ? 32u : (uint32_t)N);
    cudaFuncSetAttribute(selftest_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    selftest_mma_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
        ta, tb, static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B), D, N, K,
        mode, cols, status);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
