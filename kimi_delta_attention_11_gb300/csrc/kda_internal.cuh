// kda_internal.cuh -- shared definitions of the CUDA library (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kChunk = 64;  // chunk size C: the production path fixes C = 64

// Byte layout of the caller's workspace.
//   [0, 4)       int32 device status word (0 = ok, else a kda_status)
//   [16, 20)     int32 number of chunks, written by the chunk-index kernel
//   chunk table  int4 per chunk   {sequence, first token, length, index in sequence}
//   seq table    int2 per sequence {first chunk, number of chunks}
//   inter        per (chunk, head) intermediates of the intra-chunk stage
struct Layout {
    size_t status_off = 0;
    size_t count_off = 16;
    size_t chunk_tab_off = 0;
    size_t seq_tab_off = 0;
    size_t inter_off = 0;
    size_t inter_stride = 0;  // bytes per (chunk, head)
    size_t total = 0;
    long long max_chunks = 0;
    int N = 0;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Per-(chunk, head) intermediate record of the fp32 path (all fp32, row-major):
//   W [C][K], U [C][V], Kbar [C][K], Qg [C][K], Aqk [C][C], gamma [K]
struct SimtRecord {
    __host__ __device__ static size_t w(int) { return 0; }
    __host__ __device__ static size_t u(int K) { return (size_t)kChunk * K; }
    __host__ __device__ static size_t kbar(int K, int V) { return u(K) + (size_t)kChunk * V; }
    __host__ __device__ static size_t qg(int K, int V) { return kbar(K, V) + (size_t)kChunk * K; }
    __host__ __device__ static size_t aqk(int K, int V) { return qg(K, V) + (size_t)kChunk * K; }
    __host__ __device__ static size_t gamma(int K, int V) { return aqk(K, V) + (size_t)kChunk * kChunk; }
    __host__ __device__ static size_t floats(int K, int V) { return gamma(K, V) + K; }
};

// Per-(chunk, head) record of the bf16 tensor-core path (K = V = 128).  Every tile is
// stored as the exact shared-memory image the recurrence kernel feeds to tcgen05 (128-byte
// swizzled 64-element panels), so that kernel fetches it with plain bulk copies.
//   wq     [W ; Qg]  2 panels (key 0-63, 64-127) x [128 rows][64], K-major: rows 0-63 W
//                    (one per token), rows 64-127 the gated, scaled query.    32 KB
//   aqk    Aqk       [64 query rows][64 key cols], K-major, zero above the diagonal. 8 KB
//                    (rows 64-127 of panel 1 of wq followed by aqk form a 128-row A
//                    operand whose upper half only feeds accumulator rows the
//                    recurrence has already consumed.)
//   kbar   K_bar     [64 tokens][128 keys] as 2 panels [64][64] (token-major; read by
//                    the tensor core as the transposed operand K_bar^T).        16 KB
//   u      U         [64 tokens][128 values] as 2 panels [64][64] (token-major). 16 KB
//   gamma  gamma^C   [128] fp32 (decay of the whole chunk per key channel).
struct TcRecord {
    static constexpr uint32_t wq = 0;
    static constexpr uint32_t aqk = 32768;
    static constexpr uint32_t kbar = 40960;
    static constexpr uint32_t u = 57344;
    static constexpr uint32_t gamma = 73728;
    static constexpr uint32_t bytes = 74752;  // record stride (1024-aligned)
};

// The bf16 tensor-core path serves K = V = 128; other bf16 shapes and fp32 take the
// exact CUDA-core path.
inline bool use_tc_path(int K, int V, kda_dtype dt) {
    return dt == KDA_DTYPE_BF16 && K == 128 && V == 128;
}

// 2-D TMA tensor map over a row-major matrix of `outer` rows x `inner` elements
// (bf16 or fp32), box of box_outer rows x box_inner elements, optional 128-byte swizzle,
// zero fill outside the tensor.  Returns false if the driver rejects it.
bool make_tmap_2d(CUtensorMap* map, const void* base, bool bf16, uint64_t inner, uint64_t outer,
                  uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128);

Layout make_layout(int B, int T, int H, int K, int V, int num_seqs, bool packed, kda_dtype dt);

// Launchers (return cudaGetLastError() of their launches).
cudaError_t launch_chunk_index(const int32_t* cu_seqlens, int N, int T, const Layout& L,
                               char* ws, cudaStream_t s);
cudaError_t launch_tc(const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float scale, const float* s0, void* o, float* sN, int B,
                      int T, int H, const Layout& L, char* ws, cudaStream_t s,
                      void* const* events_after);
cudaError_t launch_simt(const void* q, const void* k, const void* v, const float* g,
                        const float* beta, float scale, const float* s0, void* o, float* sN,
                        int H, int K, int V, kda_dtype dt, const Layout& L, char* ws,
                        cudaStream_t s, void* const* events_after);

// Records events_after[i] (a cudaEvent_t) on s when events_after is non-null.
inline bool record_event(void* const* events_after, int i, cudaStream_t s) {
    return !events_after ||
           cudaEventRecord(static_cast<cudaEvent_t>(events_after[i]), s) == cudaSuccess;
}

}  // namespace kda
