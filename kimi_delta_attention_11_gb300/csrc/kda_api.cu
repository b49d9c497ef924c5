// kda_api.cu -- the C ABI entry points declared in include/kda.h.
//
// Host-side validation happens before anything is enqueued; then the chunk index, the
// intra-chunk stage and the state/output recurrence are launched on the caller's
// stream with no host synchronisation and no allocation.
#include <atomic>
#include <limits.h>
#include <cstdlib>
#include <cstring>

#include "kda_internal.cuh"

namespace kda {

// Schedule request from the KDA_SCHEDULE environment variable ("two", "pipelined",
// "fused", "scan"; anything else or unset: automatic).  A forced schedule that does not apply to
// the sizes falls back to the automatic choice's next option (see make_layout).
Schedule schedule_request() {
    const char* e = std::getenv("KDA_SCHEDULE");
    if (!e) return Schedule::kAuto;
    if (!std::strcmp(e, "two")) return Schedule::kTwo;
    if (!std::strcmp(e, "pipelined")) return Schedule::kPipelined;
    if (!std::strcmp(e, "fused")) return Schedule::kFused;
    if (!std::strcmp(e, "scan")) return Schedule::kScan;
    return Schedule::kAuto;
}

// SM count of the current device, 0 without one (then no schedule depends on it).
int current_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return sms;
}

Layout make_layout(int B, int T, int H, int K, int V, int num_seqs, bool packed, kda_dtype dt,
                   int sm_count) {
    Layout L;
    const long long nct = ((long long)T + kChunk - 1) / kChunk;
    L.N = packed ? num_seqs : B;
    if (packed)
        L.max_chunks = T > 0 ? nct + num_seqs - 1 : 0;
    else
        L.max_chunks = (long long)B * nct;
    L.chunk_tab_off = 256;
    L.seq_tab_off = align_up(L.chunk_tab_off + (size_t)L.max_chunks * 16, 256);
    L.inter_off = align_up(L.seq_tab_off + (size_t)L.N * 8, 1024);
    L.inter_stride = use_tc_path(K, V, dt) ? (size_t)TcRecord::bytes
                                           : align_up(SimtRecord::floats(K, V) * sizeof(float), 1024);
    L.total = L.inter_off + (size_t)L.max_chunks * H * L.inter_stride;
    L.fixed = use_tc_path(K, V, dt) && !packed;
    const Schedule want = schedule_request();
    const long long chains = (long long)B * H;
    const int sms = !(L.fixed && L.max_chunks > 0) ? 0 : sm_count >= 0 ? sm_count : current_sm_count();
    // Fused: the recurrences of few chains occupy few SMs for the whole call, so the
    // records are produced on the other SMs while they run (one CTA per SM, both
    // stages in one cooperative launch).  Automatic up to a third of the SMs.
    const bool can_fuse = L.fixed && L.max_chunks > 0 && sms > 0 && 2 * chains <= sms;
    const bool auto_fuse = can_fuse && 3 * chains <= sms;
    // Pipelining pays when the recurrence has few, long chains (its ordered chunk steps,
    // not the SM count, set its time): fixed-length input, at most 128 (sequence, head)
    // chains and at least 512 chunks per sequence (measured on GB300: a 6 % gain at
    // 2048 chunks per sequence, a loss at 64, where the recurrence kernel's CTAs, which
    // need a whole SM each, wait for the next range's intra-chunk CTAs to drain).
    // Ranges of 32 chunks; a ring of 3 ranges of records so the intra-chunk kernel can
    // run up to 2 ranges ahead.
    const bool can_pipe = L.fixed && chains <= 128 && nct >= 2;
    const bool auto_pipe = can_pipe && nct >= kPipeMinChunks;
    // Scan: with very few chains the ordered chunk steps of each chain set the call's time
    // however fast the records are made, so each sequence is cut into segments whose
    // affine summaries (Phi, Psi) are formed in parallel, merged per chain, and then
    // replayed from the merged start states (three chunk-step passes instead of one, all
    // parallel over segments).  Automatic up to an eighth of the SMs' count of chains and
    // from 128 chunks per sequence.
    const bool can_scan = L.fixed && L.max_chunks > 0 && sms > 0 && nct >= 4 && chains <= sms;
    const bool auto_scan = can_scan && 8 * chains <= sms && nct >= 128;
    if (want == Schedule::kScan ? can_scan : (want == Schedule::kAuto && auto_scan)) {
        long long P = sms / (2 * chains);
        P = P < 2 ? 2 : P;
        if (P > nct / 2) P = nct / 2;
        const long long Ls = (nct + P - 1) / P;
        L.scan = true;
        L.scan_L = (int)Ls;
        L.scan_P = (int)((nct + Ls - 1) / Ls);
        const size_t plane = (size_t)chains * K * V * sizeof(float);
        L.summ_off = align_up(L.total, 1024);
        L.starts_off = align_up(L.summ_off + 2 * (size_t)L.scan_P * plane, 1024);
        L.total = L.starts_off + (size_t)L.scan_P * plane;
    } else if (want == Schedule::kFused ? can_fuse : (want == Schedule::kAuto && auto_fuse)) {
        L.fused = true;
        L.flags_off = align_up(L.total, 256);
        L.total = L.flags_off + (size_t)L.max_chunks * H * sizeof(int);
    } else if (want == Schedule::kPipelined ? can_pipe : (want == Schedule::kAuto && auto_pipe)) {
        L.span = 32;
        L.ranges = (int)((nct + L.span - 1) / L.span);
        L.ring = 3;
        L.carry_off = align_up(L.total, 1024);
        L.total = L.carry_off + (size_t)B * H * K * V * sizeof(float);
    }
    return L;
}

}  // namespace kda

using namespace kda;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Size and shape rules shared by kda_fwd and kda_fwd_workspace_bytes.
kda_status check_sizes(int B, int T, int H, int K, int V, int num_seqs, bool packed,
                       int chunk_size, kda_dtype dt) {
    if (B < 1 || T < 0 || H < 1 || K < 1 || V < 1) return KDA_ERR_INVALID_ARG;
    if (dt != KDA_DTYPE_BF16 && dt != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
    // State propagation is defined for K <= 256 (Tokamax design doc, 5.3).
    if (K > 256 || V > 256) return KDA_ERR_INVALID_ARG;
    if (packed && (B != 1 || num_seqs < 1)) return KDA_ERR_INVALID_ARG;
    // every element index must fit the kernels' 64-bit arithmetic and every token
    // index a 32-bit int
    if ((long long)B * T >= INT_MAX) return KDA_ERR_INVALID_ARG;
    if (chunk_size != kChunk) return KDA_ERR_UNSUPPORTED;
    if ((K != 64 && K != 128) || (V != 64 && V != 128)) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

// The library is built for sm_103a only; refuse any other current device up front.
kda_status check_device() {
    // 0 unknown, 1 ok, 2 unusable; host threads may race to fill an entry, and all of
    // them write the same value
    static std::atomic<int> verdict[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return KDA_ERR_DEVICE;
    }
    int v = verdict[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        int major = 0, minor = 0;
        const bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) ==
                            cudaSuccess &&
                        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) ==
                            cudaSuccess &&
                        major == 10 && minor == 3;
        cudaGetLastError();
        v = ok ? 1 : 2;
        verdict[dev].store(v, std::memory_order_relaxed);
    }
    return v == 1 ? KDA_OK : KDA_ERR_DEVICE;
}

}  // namespace

extern "C" {

int kda_abi_version(void) { return 103; }

int kda_fwd_schedule_for(int B, int T, int H, int K, int V, int num_seqs, int chunk_size,
                         kda_dtype dtype, int sm_count) {
    const bool packed = num_seqs > 0;
    if (sm_count < 0) return -1;
    if (check_sizes(B, T, H, K, V, num_seqs, packed, chunk_size, dtype) != KDA_OK) return -1;
    const Layout L = make_layout(B, T, H, K, V, num_seqs, packed, dtype, sm_count);
    if (L.fused) return KDA_SCHEDULE_FUSED;
    if (L.scan) return KDA_SCHEDULE_SCAN;
    if (L.span > 0) return KDA_SCHEDULE_PIPELINED;
    return KDA_SCHEDULE_TWO_KERNELS;
}

int kda_fwd_schedule(int B, int T, int H, int K, int V, int num_seqs, int chunk_size,
                     kda_dtype dtype) {
    return kda_fwd_schedule_for(B, T, H, K, V, num_seqs, chunk_size, dtype, current_sm_count());
}

int kda_fwd_launch_count(int B, int T, int H, int K, int V, int num_seqs, int chunk_size,
                         kda_dtype dtype) {
    const bool packed = num_seqs > 0;
    if (check_sizes(B, T, H, K, V, num_seqs, packed, chunk_size, dtype) != KDA_OK) return -1;
    const Layout L = make_layout(B, T, H, K, V, num_seqs, packed, dtype);
    const int index = L.fixed ? 0 : 1;
    if (L.fused) return 1;
    if (L.scan) return 4;
    if (L.span > 0) return index + 2 * L.ranges;
    return index + (L.max_chunks > 0 ? 1 : 0) + (L.N > 0 ? 1 : 0);
}

const char* kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported configuration";
        case KDA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case KDA_ERR_WORKSPACE: return "workspace missing or too small";
        case KDA_ERR_CUDA: return "CUDA runtime error";
        case KDA_ERR_DEVICE_TIMEOUT: return "device-side bounded wait expired";
        case KDA_ERR_DEVICE: return "no usable sm_103 device";
        default: return "unknown status";
    }
}

size_t kda_fwd_workspace_bytes(int B, int T, int H, int K, int V, int num_seqs, int chunk_size,
                               kda_dtype dtype) {
    const bool packed = num_seqs > 0;
    if (check_sizes(B, T, H, K, V, num_seqs, packed, chunk_size, dtype) != KDA_OK) return 0;
    return make_layout(B, T, H, K, V, num_seqs, packed, dtype).total;
}

kda_status kda_build_chunk_index(const int32_t* cu_seqlens, int num_seqs, int B, int T,
                                 int chunk_size, void* workspace, size_t workspace_bytes,
                                 size_t* chunk_table_offset, size_t* seq_table_offset,
                                 size_t* count_offset, void* stream) {
    const bool packed = cu_seqlens != nullptr;
    if (B < 1 || T < 0 || (packed && (B != 1 || num_seqs < 1))) return KDA_ERR_INVALID_ARG;
    if ((long long)B * T >= INT_MAX) return KDA_ERR_INVALID_ARG;
    if (chunk_size != kChunk) return KDA_ERR_UNSUPPORTED;
    if (!workspace) return KDA_ERR_WORKSPACE;
    if (!aligned16(workspace) || (packed && !aligned4(cu_seqlens))) return KDA_ERR_ALIGNMENT;
    const Layout L = make_layout(B, T, 1, 64, 64, num_seqs, packed, KDA_DTYPE_F32);
    const size_t need = L.inter_off;  // index part only
    if (workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if (chunk_table_offset) *chunk_table_offset = L.chunk_tab_off;
    if (seq_table_offset) *seq_table_offset = L.seq_tab_off;
    if (count_offset) *count_offset = L.count_off;
    if (kda_status d = check_device()) return d;
    char* ws = static_cast<char*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (launch_chunk_index(cu_seqlens, L.N, T, L, ws, s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // extern "C"

namespace {

// kda_gate_options -> the kernels' GateArgs; KDA_OK or the validation failure.
kda_status gate_args(const kda_gate_options* opts, GateArgs* ga) {
    *ga = GateArgs{};
    if (!opts) return KDA_OK;
    if (opts->use_gate_in_kernel) {
        if (!opts->a_log) return KDA_ERR_INVALID_ARG;
        if (!aligned4(opts->a_log) || (opts->dt_bias && !aligned4(opts->dt_bias)))
            return KDA_ERR_ALIGNMENT;
        const float lb = opts->lower_bound;
        // Tokamax design doc 5.3: a lower bound selects the sigmoid form, -5 <= lb < 0
        if (lb != 0.f && !(lb >= -5.f && lb < 0.f)) return KDA_ERR_INVALID_ARG;
        ga->mode = lb == 0.f ? 1 : 2;
        ga->a_log = opts->a_log;
        ga->dt_bias = opts->dt_bias;
        ga->lower_bound = lb;
    }
    ga->qk_l2norm = opts->qk_l2norm ? 1 : 0;
    return KDA_OK;
}

kda_status fwd_impl(const void* q, const void* k, const void* v, const float* g, const float* beta,
                    float scale, int chunk_size, const float* initial_state,
                    const int32_t* cu_seqlens, int num_seqs, void* o, float* final_state, int B,
                    int T, int H, int K, int V, kda_dtype dtype, void* workspace,
                    size_t workspace_bytes, const kda_gate_options* opts, void* stream,
                    void* const* events, int num_events) {
    const bool packed = cu_seqlens != nullptr;
    if (kda_status st = check_sizes(B, T, H, K, V, num_seqs, packed, chunk_size, dtype))
        return st;
    GateArgs ga;
    if (kda_status st = gate_args(opts, &ga)) return st;
    // With T == 0 no token tensor is read or written, so its pointers may be anything.
    const bool tokens = T > 0;
    if (tokens && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (num_events != 0 && (num_events < 4 || !events)) return KDA_ERR_INVALID_ARG;
    if (!workspace) return KDA_ERR_WORKSPACE;
    if ((tokens && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) ||
                    !aligned4(beta) || !aligned16(o))) ||
        !aligned16(workspace) || (initial_state && !aligned16(initial_state)) ||
        (final_state && !aligned16(final_state)) || (packed && !aligned4(cu_seqlens)))
        return KDA_ERR_ALIGNMENT;
    const Layout L = make_layout(B, T, H, K, V, num_seqs, packed, dtype);
    if (workspace_bytes < L.total) return KDA_ERR_WORKSPACE;
    if (kda_status d = check_device()) return d;

    char* ws = static_cast<char*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto mark = [&](int i) {
        return num_events == 0 ||
               cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) == cudaSuccess;
    };
    if (!mark(0)) return KDA_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (!L.fixed && launch_chunk_index(cu_seqlens, L.N, T, L, ws, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (!mark(1)) return KDA_ERR_CUDA;
    const cudaError_t e =
        use_tc_path(K, V, dtype)
            ? launch_tc(q, k, v, g, beta, scale, ga, initial_state, o, final_state, B, T, H, L,
                        ws, s, num_events ? events + 2 : nullptr)
            : launch_simt(q, k, v, g, beta, scale, ga, initial_state, o, final_state, H, K, V,
                          dtype, L, ws, s, num_events ? events + 2 : nullptr);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_fwd_profiled(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, float scale, int chunk_size,
                            const float* initial_state, const int32_t* cu_seqlens, int num_seqs,
                            void* o, float* final_state, int B, int T, int H, int K, int V,
                            kda_dtype dtype, void* workspace, size_t workspace_bytes,
                            void* stream, void* const* events, int num_events) {
    return fwd_impl(q, k, v, g, beta, scale, chunk_size, initial_state, cu_seqlens, num_seqs, o,
                    final_state, B, T, H, K, V, dtype, workspace, workspace_bytes, nullptr, stream,
                    events, num_events);
}

kda_status kda_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                   float scale, int chunk_size, const float* initial_state,
                   const int32_t* cu_seqlens, int num_seqs, void* o, float* final_state, int B,
                   int T, int H, int K, int V, kda_dtype dtype, void* workspace,
                   size_t workspace_bytes, void* stream) {
    return fwd_impl(q, k, v, g, beta, scale, chunk_size, initial_state, cu_seqlens, num_seqs, o,
                    final_state, B, T, H, K, V, dtype, workspace, workspace_bytes, nullptr, stream,
                    nullptr, 0);
}

kda_status kda_fwd_ex(const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float scale, int chunk_size,
                      const float* initial_state, const int32_t* cu_seqlens, int num_seqs,
                      void* o, float* final_state, int B, int T, int H, int K, int V,
                      kda_dtype dtype, void* workspace, size_t workspace_bytes,
                      const kda_gate_options* opts, void* stream) {
    return fwd_impl(q, k, v, g, beta, scale, chunk_size, initial_state, cu_seqlens, num_seqs, o,
                    final_state, B, T, H, K, V, dtype, workspace, workspace_bytes, opts, stream,
                    nullptr, 0);
}

kda_status kda_decode(const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float scale, float* state, void* o, int N, int H, int K,
                      int V, kda_dtype dtype, const kda_gate_options* opts, void* stream) {
    if (N < 0 || H < 1 || K < 1 || V < 1) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
    if (K > 256 || V > 256) return KDA_ERR_INVALID_ARG;
    if ((K != 64 && K != 128) || (V != 64 && V != 128)) return KDA_ERR_UNSUPPORTED;
    GateArgs ga;
    if (kda_status st = gate_args(opts, &ga)) return st;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !state || !o) return KDA_ERR_INVALID_ARG;
    const size_t es = dtype == KDA_DTYPE_BF16 ? 2 : 4;
    auto al = [](const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
    if (!al(q, es) || !al(k, es) || !al(v, es) || !al(o, es) || !aligned4(g) || !aligned4(beta) ||
        !aligned4(state))
        return KDA_ERR_ALIGNMENT;
    if ((long long)N * H * K * V >= (1ll << 40)) return KDA_ERR_INVALID_ARG;
    if (kda_status d = check_device()) return d;
    const cudaError_t e = launch_decode(q, k, v, g, beta, scale, ga, state, o, N, H, K, V, dtype,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_get_device_status(const void* workspace, void* stream) {
    if (!workspace) return KDA_ERR_WORKSPACE;
    int word = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return KDA_ERR_CUDA;
    return word == 0 ? KDA_OK : static_cast<kda_status>(word);
}

}  // extern "C"
