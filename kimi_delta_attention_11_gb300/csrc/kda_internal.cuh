// kda_internal.cuh -- shared definitions of the CUDA library (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kChunk = 64;  // chunk size C: the production path fixes C = 64
constexpr int kPipeMinChunks = 512;  // chunks per sequence from which calls are pipelined

// Launch schedule of a call (see make_layout).
enum class Schedule { kAuto, kTwo, kPipelined, kFused, kScan };

// Byte layout of the caller's workspace.
//   [0, 4)       int32 device status word (0 = ok, else a kda_status)
//   [16, 20)     int32 number of chunks, written by the chunk-index kernel
//   chunk table  int4 per chunk   {sequence, first token, length, index in sequence}
//   seq table    int2 per sequence {first chunk, number of chunks}
//   inter        per (chunk, head) intermediates of the intra-chunk stage
//   carry        (pipelined calls) fp32 [N][H][K][V] state handed between chunk ranges
struct Layout {
    size_t status_off = 0;
    size_t count_off = 16;
    size_t chunk_tab_off = 0;
    size_t seq_tab_off = 0;
    size_t inter_off = 0;
    size_t inter_stride = 0;  // bytes per (chunk, head)
    size_t carry_off = 0;
    size_t total = 0;
    long long max_chunks = 0;
    int N = 0;
    // Pipelined schedule (bf16 tensor-core path, fixed-length input with few chains):
    // the chunks of every sequence are cut into ranges of `span`; the intra-chunk kernel
    // of range r + 1 runs on the caller's stream while the recurrence of range r runs on
    // a second stream.  span == 0: one launch of each kernel over the whole problem.
    int span = 0, ranges = 0, ring = 0;
    // fixed-length input on the tensor-core path: chunk facts are arithmetic (ChunkIndex)
    // and no chunk-index kernel runs
    bool fixed = false;
    // Fused schedule (tensor-core path, fixed-length input with few chains): one
    // cooperative launch in which some CTAs run the recurrences and the rest produce the
    // records, published through one flag word per (chunk, head) at flags_off.
    bool fused = false;
    size_t flags_off = 0;
    // Chunk-parallel scan schedule (tensor-core path, fixed-length input with very few,
    // long chains): segments of scan_L chunks, scan_P per sequence; segment summaries
    // [2][P][chains][K][V] at summ_off, merged segment start states [P][chains][K][V] at
    // starts_off.
    bool scan = false;
    int scan_P = 0, scan_L = 0;
    size_t summ_off = 0, starts_off = 0;
};

// Where the kernels find a chunk's sequence, first token, length and index within its
// sequence.  Packed input: the tables the chunk-index kernel builds in the workspace.
// Fixed-length input (the bf16 tensor-core path): sequence n is tokens [n T, (n + 1) T),
// so the same facts follow arithmetically and that path launches no index kernel.
struct ChunkIndex {
    const int4* chunk_tab = nullptr;  // {sequence, first token, length, index in sequence}
    const int2* seq_tab = nullptr;    // {first chunk, number of chunks}
    const int* count = nullptr;       // number of chunks
    int fixed = 0, T = 0, nct = 0;    // fixed length: T tokens, nct chunks per sequence
#ifdef __CUDACC__
    __device__ __forceinline__ int4 chunk(long long c) const {
        if (!fixed) return chunk_tab[c];
        const int n = (int)(c / nct), j = (int)(c - (long long)n * nct);
        return make_int4(n, n * T + j * kChunk, min(kChunk, T - j * kChunk), j);
    }
    __device__ __forceinline__ int2 seq(int n) const {
        return fixed ? make_int2(n * nct, nct) : seq_tab[n];
    }
    // number of chunks, given the launch's upper bound (exact for fixed length)
    __device__ __forceinline__ long long num_chunks(long long max_chunks) const {
        return fixed ? max_chunks : *count;
    }
#endif
};

// Gate activation and q/k normalisation inside the kernels (Tokamax design doc 9.1.3,
// use_gate_in_kernel; "KDAChunkwise", FP32 core: F.normalize with eps 1e-6).  mode 0: g
// holds ln(alpha) as given; mode 1: g is a raw gate, ln(alpha) = -exp(a_log[h]) *
// softplus(g + dt_bias); mode 2: ln(alpha) = lower_bound * sigmoid(exp(a_log[h]) *
// (g + dt_bias)).  qk_l2norm: q and k are divided by max(||.||_2, 1e-6) along K first.
struct GateArgs {
    int mode = 0;
    const float* a_log = nullptr;    // [H]
    const float* dt_bias = nullptr;  // [H * K] or null
    float lower_bound = 0.f;
    int qk_l2norm = 0;
};

#ifdef __CUDACC__
// ln(alpha) of key channel d of head h from the gate input x as the kernels read it.
__device__ __forceinline__ float gate_log_decay(const GateArgs& ga, float x, int h, int d, int K) {
    if (ga.mode == 0) return x;
    if (ga.dt_bias) x += ga.dt_bias[(size_t)h * K + d];
    const float lam = expf(ga.a_log[h]);
    if (ga.mode == 1) {
        // softplus, with the usual linear branch where exp would overflow the sum
        const float sp = x > 20.f ? x : log1pf(expf(x));
        return -lam * sp;
    }
    return ga.lower_bound / (1.f + expf(-lam * x));
}
#endif

// Chunk range of one kernel launch: chunks j0 <= j < j0 + span of every sequence
// (j = index within the sequence); span == 0 means all chunks.  carry: the state buffer
// between ranges (pipelined calls only).
struct RangeArgs {
    int j0 = 0;
    int span = 0;
    float* carry = nullptr;
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
// swizzled 64-element panels), so that kernel fetches the record with one bulk copy.
// The recurrence computes transposed products (state and V_new as tensor-memory operands
// with one lane per value column), so every tile here is its B operand:
//   wq     [W ; Qg]  2 panels (key 0-63, 64-127) x [128 rows][64], K-major: rows 0-63 W
//                    (one per token), rows 64-127 the gated, scaled query.    32 KB
//   aqk    Aqk       [64 query rows][64 key cols], K-major, zero above the diagonal. 8 KB
//   kb0, kb1  K_bar  keys 0-63 / 64-127: [64 tokens][64] token-major (MN-major B).  16 KB
//   ut     U^T       [128 value rows][64 tokens], K-major.                         16 KB
//   gamma  gamma^C   [128] fp32 (decay of the whole chunk per key channel).
// (Records for the value-sliced recurrence kernel, which computes the untransposed
// products with a state slice of 64 value columns per CTA, use TcRecordS below.)
struct TcRecord {
    static constexpr bool sliced = false;
    static constexpr uint32_t wq = 0;
    static constexpr uint32_t aqk = 32768;
    static constexpr uint32_t kb0 = 40960;
    static constexpr uint32_t kb1 = 49152;
    static constexpr uint32_t ut = 57344;
    static constexpr uint32_t gamma = 73728;
    static constexpr uint32_t used = gamma + 512;  // bytes the recurrence fetches
    static constexpr uint32_t bytes = 74752;        // record stride (1024-aligned)
};

// Record of the value-sliced recurrence kernel (one CTA per 64 value columns): the same
// tiles except U, which is token-major and split by value slice, placed so that each
// slice's CTA fetches one contiguous run per chunk, [u1, u0) for slice 1 and
// [wq, gamma) for slice 0:
//   u1     U, values 64-127: [64 tokens][64] token-major.                         8 KB
//   wq     [W ; Qg] as above (its panel 1 rows 64-127 followed by aqk form a 128-row A
//          operand whose upper half only feeds accumulator rows never read).       32 KB
//   aqk, kb0, kb1, gamma as above;  u0  U, values 0-63.                             8 KB
struct TcRecordS {
    static constexpr bool sliced = true;
    static constexpr uint32_t u1 = 0;
    static constexpr uint32_t wq = 8192;
    static constexpr uint32_t aqk = 40960;
    static constexpr uint32_t kb0 = 49152;
    static constexpr uint32_t kb1 = 57344;
    static constexpr uint32_t u0 = 65536;
    static constexpr uint32_t gamma = 73728;
    static constexpr uint32_t bytes = 74752;
};
static_assert(TcRecordS::bytes == TcRecord::bytes, "both record forms share the workspace stride");

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

// sm_count < 0: the current device's SM count (0 when no device is current)
Layout make_layout(int B, int T, int H, int K, int V, int num_seqs, bool packed, kda_dtype dt,
                   int sm_count = -1);

// Launchers (return cudaGetLastError() of their launches).
cudaError_t launch_chunk_index(const int32_t* cu_seqlens, int N, int T, const Layout& L,
                               char* ws, cudaStream_t s);
cudaError_t launch_tc(const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float scale, const GateArgs& ga, const float* s0, void* o,
                      float* sN, int B, int T, int H, const Layout& L, char* ws, cudaStream_t s,
                      void* const* events_after);
cudaError_t launch_decode(const void* q, const void* k, const void* v, const float* g,
                          const float* beta, float scale, const GateArgs& ga, float* state,
                          void* o, int N, int H, int K, int V, kda_dtype dt, cudaStream_t s);
cudaError_t launch_simt(const void* q, const void* k, const void* v, const float* g,
                        const float* beta, float scale, const GateArgs& ga, const float* s0,
                        void* o, float* sN, int H, int K, int V, kda_dtype dt, const Layout& L,
                        char* ws, cudaStream_t s, void* const* events_after);

// Records events_after[i] (a cudaEvent_t) on s when events_after is non-null.
inline bool record_event(void* const* events_after, int i, cudaStream_t s) {
    return !events_after ||
           cudaEventRecord(static_cast<cudaEvent_t>(events_after[i]), s) == cudaSuccess;
}

}  // namespace kda
