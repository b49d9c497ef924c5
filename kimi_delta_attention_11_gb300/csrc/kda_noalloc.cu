// kda_noalloc.cu -- kda_fwd for callers that cannot hand the library a workspace.
//
// kda_fwd needs a caller-provided device workspace (chunk index, status word and the
// per-chunk intermediates passed from the intra-chunk kernel to the recurrence kernel).
// Some callers have no way to obtain one: plug-ins hosted by an application that owns
// every device allocation through its own allocator, latency-critical request paths
// where an allocation is forbidden because cudaMalloc/cudaFree can synchronise the
// whole device, or thin bindings that have no device-memory allocator at all.
// kda_fwd_noalloc serves them with a fixed scratch area compiled into this library:
// a file-scope device array of KDA_NOALLOC_SCRATCH_BYTES bytes.
//
// Consequences a caller must know (also stated in include/kda.h):
//   - every GPU on which this library's module is loaded holds the array until the
//     process exits;
//   - all calls on one device share the array; it keeps whatever the previous call
//     left there (kda_fwd clears the parts that must start at zero itself), and two
//     calls whose work overlaps on the GPU (different streams, no ordering) race on it;
//   - the first call on a device looks up the array's device address (once per device,
//     with that device current); make that first call before any stream capture;
//   - problems whose workspace (kda_fwd_workspace_bytes) exceeds the array are
//     rejected with KDA_ERR_WORKSPACE before anything is launched.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "kda_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices];  // device address of the array, per device id

// Device address of the scratch array on the current device (looked up once per device).
kda_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return KDA_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                      const float* beta, float scale, int chunk_size,
                                      const float* initial_state, const int32_t* cu_seqlens,
                                      int num_seqs, void* o, float* final_state, int B, int T,
                                      int H, int K, int V, kda_dtype dtype, void* stream) {
    const int packed_seqs = cu_seqlens ? num_seqs : 0;
    const size_t need =
        kda_fwd_workspace_bytes(B, T, H, K, V, packed_seqs, chunk_size, dtype);
    if (need == 0)  // invalid sizes: let kda_fwd report which rule failed, launching nothing
        return kda_fwd(q, k, v, g, beta, scale, chunk_size, initial_state, cu_seqlens, num_seqs,
                       o, final_state, B, T, H, K, V, dtype, nullptr, 0, stream);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (kda_status st = scratch_address(&scratch)) return st;
    return kda_fwd(q, k, v, g, beta, scale, chunk_size, initial_state, cu_seqlens, num_seqs, o,
                   final_state, B, T, H, K, V, dtype, scratch, (size_t)KDA_NOALLOC_SCRATCH_BYTES,
                   stream);
}
