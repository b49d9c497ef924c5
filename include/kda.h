/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention forward library.
 *
 * What is computed (Tokamax "chunk_kda_fwd_design_doc", Appendix 9.1.2, Eq. (1), and
 * "KDA Doesn't Care About the Future", "Chunkwise KDA in Broad Strokes"): for every
 * sequence n and head h, a K x V fp32 state S evolves token by token as
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = scale * S_t^T q_t,
 *
 * starting from initial_state[n,h] (or zero).  The library evaluates it chunk by chunk
 * (chunk size 64) as in Appendix 9.1.3-9.1.6 (Eq. (6)-(9)): a per-chunk gate cumsum, an
 * intra-chunk unit-lower-triangular solve giving the W/U representation and the causal
 * query-key matrix Aqk, the ordered chunk-to-chunk state recurrence and the output.
 * Packed variable-length sequences (cu_seqlens) never share a chunk or a state
 * (Appendix 9.1.7).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are CUDA device pointers owned by the caller; the library
 *     keeps no pointer after a call returns and allocates no device memory.
 *   - Layouts are row-major and token-major:
 *       q, k : [B, T, H, K]    v, o : [B, T, H, V]    g : [B, T, H, K] (fp32)
 *       beta : [B, T, H] (fp32)
 *       initial_state, final_state : [N, H, K, V] (fp32), a state row is a key channel.
 *     N = B for fixed-length input; N = num_seqs for packed input (then B == 1 and
 *     sequence n occupies tokens [cu_seqlens[n], cu_seqlens[n+1]) of the T axis).
 *   - g is the natural-log decay ln(alpha), expected in [-5, 0] (the bound under which
 *     the 16-key rebasing window of the bf16 path cannot overflow); it is not clamped.
 *   - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 *     stream), performs no host synchronisation and no allocation.  Arguments are
 *     validated on the host before anything is enqueued: an error status means that
 *     nothing was launched and no output was written.
 *   - Errors are returned, never printed or thrown.
 *
 * dtype of q, k, v and o: KDA_DTYPE_BF16 or KDA_DTYPE_F32.  fp32 inputs take an exact
 * fp32 path (SIMT forward substitution); bf16 inputs with K = V = 128 take the tcgen05
 * tensor-core path with fp32 accumulation and an fp32 state.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,     /* null required pointer, bad size, B != 1 with cu_seqlens */
    KDA_ERR_UNSUPPORTED = 2,     /* valid but not implemented: chunk_size != 64, K or V not in {64, 128} */
    KDA_ERR_ALIGNMENT = 3,       /* a pointer is misaligned (16 bytes; 4 for beta and cu_seqlens) */
    KDA_ERR_WORKSPACE = 4,       /* workspace null or smaller than kda_fwd_workspace_bytes() */
    KDA_ERR_CUDA = 5,            /* a CUDA runtime call or kernel launch failed */
    KDA_ERR_DEVICE_TIMEOUT = 6,  /* a kernel gave up a bounded wait (read via kda_get_device_status) */
    KDA_ERR_DEVICE = 7           /* no usable sm_103 device is current */
} kda_status;

typedef enum kda_dtype {
    KDA_DTYPE_BF16 = 0,
    KDA_DTYPE_F32 = 1
} kda_dtype;

/* Gate activation and q/k normalisation performed inside the kernels (Tokamax design
 * doc 9.1.3, use_gate_in_kernel; "KDAChunkwise", FP32 core, F.normalize).  Pass NULL
 * (or a zeroed struct) for the plain behaviour: g holds ln(alpha) and q, k are used as
 * given.
 *   use_gate_in_kernel  non-zero: g holds the raw gate x, and with
 *                       lambda_h = exp(a_log[h]) and x' = x + dt_bias[h*K + d]:
 *                         lower_bound == 0:  ln(alpha) = -lambda_h * softplus(x')
 *                         -5 <= lower_bound < 0:  ln(alpha) = lower_bound * sigmoid(lambda_h x')
 *                       (any other lower_bound is KDA_ERR_INVALID_ARG).
 *   a_log               fp32 device [H]; required when use_gate_in_kernel.
 *   dt_bias             nullable fp32 device [H*K].
 *   qk_l2norm           non-zero: q and k are divided by max(||.||_2, 1e-6) along K
 *                       (in fp32) before use.
 * Rows past the end of a sequence are identity steps whatever the raw gate holds, so no
 * -1e4 padding of raw gates (Tokamax design doc 9.1.7) is needed. */
typedef struct kda_gate_options {
    int use_gate_in_kernel;
    const float* a_log;
    const float* dt_bias;
    float lower_bound;
    int qk_l2norm;
} kda_gate_options;

/* Bytes of device workspace kda_fwd needs for these sizes (0 on invalid sizes).
 * Packed input (num_seqs > 0 together with a non-null cu_seqlens at call time) needs
 * room for ceil(T/64) + num_seqs - 1 chunks per head; fixed length for B * ceil(T/64).
 * Pass num_seqs = 0 for fixed-length input.  The workspace holds the chunk table, a
 * device status word, the per-chunk intermediates that the intra-chunk kernel hands to
 * the recurrence kernel (the chunk's affine state map and output operands), and, for
 * pipelined calls (see kda_fwd), the state handed between chunk ranges. */
size_t kda_fwd_workspace_bytes(int B, int T, int H, int K, int V, int num_seqs,
                               int chunk_size, kda_dtype dtype);

/* Chunkwise KDA forward (Tokamax design doc, 9.1.5-9.1.7, Eq. (6)-(9)).
 *
 *   q, k, v        [B,T,H,K], [B,T,H,K], [B,T,H,V] of `dtype`; q and k are used as given
 *                  (callers L2-normalise them when the model does).
 *   g, beta        fp32 [B,T,H,K] natural-log decays, fp32 [B,T,H] write strengths.
 *   scale          output scale (commonly K^-0.5).
 *   chunk_size     must be 64.
 *   initial_state  nullable fp32 [N,H,K,V]; NULL means a zero state.
 *   cu_seqlens     nullable int32 [num_seqs+1] device array, cu_seqlens[0] = 0,
 *                  non-decreasing, cu_seqlens[num_seqs] = T (a precondition: contents
 *                  are not read on the host).  Requires B == 1.  Zero-length sequences
 *                  are allowed and return their initial state.
 *   num_seqs       number of packed sequences (ignored when cu_seqlens is NULL).
 *   o              [B,T,H,V] of `dtype`, written for every token.
 *   final_state    nullable fp32 [N,H,K,V], written when non-NULL.
 *   B,T,H,K,V      sizes; T need not be a multiple of 64 (the last chunk of a sequence
 *                  is shorter).  T == 0 (or all sequences empty) writes only final_state;
 *                  with T == 0 the token tensors are not accessed and may be NULL.
 *   alignment      q, k, v, g, o, the states and the workspace 16 bytes; beta and
 *                  cu_seqlens 4 bytes (so a token slice of any tensor stays valid).
 *   workspace      device memory of at least kda_fwd_workspace_bytes(...) bytes,
 *                  16-byte aligned; contents on entry are ignored.
 *   stream         cudaStream_t to enqueue on.
 *
 * Returns KDA_OK when all launches were enqueued.  Results are deterministic: the
 * same inputs give bit-identical outputs, and o at token t does not depend on any
 * input of a later token of the same sequence.
 *
 * Schedule (bf16, K = V = 128, fixed-length input; everything else launches each kernel
 * once over the whole problem):
 *   fused      at most a third of the SMs' count of (sequence, head) chains: one
 *              cooperative launch, one CTA per SM; some CTAs run the recurrences and poll
 *              per-record flags in the workspace (bounded waits) that the other CTAs set
 *              as they produce the records.  A cudaMemsetAsync of the flags precedes it.
 *              The workspace size then depends on the current device's SM count.
 *   pipelined  otherwise, at most 128 chains and at least 512 chunks per sequence: the
 *              chunks of every sequence are cut into ranges, and the intra-chunk kernel
 *              of the next range runs on `stream` while the recurrence of the current one
 *              runs on a second stream of the library (created once per device with the
 *              events it needs; no device memory is allocated).  The second stream forks
 *              from and joins back into `stream` through events, so the call stays ordered
 *              on `stream` and can be captured into a CUDA graph.
 *   scan       at most an eighth of the SMs' count of chains and at least 128 chunks per
 *              sequence: chunk-parallel state scan (segment summaries, a per-chain merge of
 *              segment start states, then every segment replayed): four launches.
 *              Where both the scan and the fused rule hold, the scan is taken.
 * The environment variable KDA_SCHEDULE ("two", "pipelined", "fused", "scan") forces a schedule
 * where the sizes allow it (read at workspace sizing and at each call, which must agree).
 * kda_fwd_launch_count gives the number of kernel launches. */
kda_status kda_fwd(const void* q, const void* k, const void* v, const float* g,
                   const float* beta, float scale, int chunk_size,
                   const float* initial_state, const int32_t* cu_seqlens, int num_seqs,
                   void* o, float* final_state, int B, int T, int H, int K, int V,
                   kda_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/* kda_fwd with gate activation / q-k normalisation options (`opts` nullable: then this
 * is kda_fwd).  Same arguments, layouts and rules otherwise. */
kda_status kda_fwd_ex(const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float scale, int chunk_size,
                      const float* initial_state, const int32_t* cu_seqlens, int num_seqs,
                      void* o, float* final_state, int B, int T, int H, int K, int V,
                      kda_dtype dtype, void* workspace, size_t workspace_bytes,
                      const kda_gate_options* opts, void* stream);

/* One decode step: every one of N sequences advances by one token, in the recurrent form
 * (Tokamax design doc 9.1.2, Eq. (1) in delta-correction form; "KDA Doesn't Care About
 * the Future", "Chunkwise KDA in Broad Strokes": the recurrence decodes a token at a time):
 *   S <- Diag(exp g) S;  e = v - S^T k;  S <- S + beta k e^T;  o = scale S^T q.
 *   q, k     [N,H,K] of `dtype`;  v, o [N,H,V] of `dtype` (o written);
 *   g        fp32 [N,H,K] (ln(alpha), or the raw gate with opts->use_gate_in_kernel);
 *   beta     fp32 [N,H];  state  fp32 [N,H,K,V], read and updated in place (required);
 *   opts     nullable, as for kda_fwd_ex.
 * K, V in {64, 128}; pointers aligned to their element size; N == 0 is a no-op.  No
 * workspace, no allocation, asynchronous on `stream`. */
kda_status kda_decode(const void* q, const void* k, const void* v, const float* g,
                      const float* beta, float scale, float* state, void* o, int N, int H,
                      int K, int V, kda_dtype dtype, const kda_gate_options* opts,
                      void* stream);

/* kda_fwd, plus CUDA events recorded on `stream` around its stages, for timing each
 * kernel on the stream it runs on.  `events` holds num_events cudaEvent_t handles
 * created by the caller; events[0] is recorded before the first launch and events[i]
 * after stage i, for the stages in order: 1 chunk index, 2 intra-chunk kernel,
 * 3 recurrence/output kernel.  num_events must be 0 (then this is kda_fwd) or at
 * least 4 (KDA_ERR_INVALID_ARG otherwise).  A stage with nothing to do (T == 0)
 * still gets its event recorded (fixed-length bf16 input with K = V = 128 has no
 * chunk-index kernel: its chunk positions are arithmetic).  With events the kernels
 * always run back to back on
 * `stream`, one launch each over the whole problem (never the pipelined or fused
 * schedule), so that each stage is one kernel's time; results agree to the bf16
 * tolerance (bit-identical to the pipelined schedule). */
kda_status kda_fwd_profiled(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, float scale, int chunk_size,
                            const float* initial_state, const int32_t* cu_seqlens,
                            int num_seqs, void* o, float* final_state, int B, int T, int H,
                            int K, int V, kda_dtype dtype, void* workspace,
                            size_t workspace_bytes, void* stream, void* const* events,
                            int num_events);

/* Build only the chunk index of a (possibly packed) input into `workspace`
 * (Tokamax design doc 3.5 and 9.1.7: chunks of 64 tokens that never cross a sequence;
 * the last chunk of a sequence may be shorter).  Writes, at the byte offsets returned
 * through the optional out-pointers:
 *   chunk table  int32x4 per chunk c: {sequence n, first token, length, index in sequence}
 *   seq table    int32x2 per sequence n: {first chunk, number of chunks}
 *   count        one int32: total number of chunks.
 * Entries past `count` are left undefined.  Same validation rules as kda_fwd.
 * kda_fwd performs this step itself; the entry point exists for tests and tools. */
kda_status kda_build_chunk_index(const int32_t* cu_seqlens, int num_seqs, int B, int T,
                                 int chunk_size, void* workspace, size_t workspace_bytes,
                                 size_t* chunk_table_offset, size_t* seq_table_offset,
                                 size_t* count_offset, void* stream);

/* Size of the scratch area compiled into the library for kda_fwd_noalloc (64 MiB). */
#define KDA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* kda_fwd without a caller-provided workspace.  (The KDA pages have no counterpart to
 * this entry point; it exists for callers of this library that cannot allocate.)
 *
 * Who needs it: callers that cannot obtain device memory for the workspace, e.g. a
 * plug-in whose host application owns every device allocation, a request path on which
 * allocating is forbidden because cudaMalloc/cudaFree may synchronise the device, or a
 * binding without any device allocator.  The call allocates nothing: its workspace is a
 * fixed device array of KDA_NOALLOC_SCRATCH_BYTES bytes inside the library.
 *
 * Arguments, layouts and results are those of kda_fwd (minus workspace and its size).
 * Rules specific to this entry point:
 *   - problems with kda_fwd_workspace_bytes(...) > KDA_NOALLOC_SCRATCH_BYTES are
 *     rejected with KDA_ERR_WORKSPACE before anything is launched;
 *   - every GPU on which the library's module is loaded keeps the array until exit;
 *   - all calls on a device share the array and it keeps the previous call's contents
 *     (the call resets what must start at zero); calls whose GPU work overlaps (e.g. on
 *     two unordered streams) race on it and must be serialised by the caller;
 *   - the first call on each device looks up the array's address with that device
 *     current; make it before any stream capture. */
kda_status kda_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                           const float* beta, float scale, int chunk_size,
                           const float* initial_state, const int32_t* cu_seqlens,
                           int num_seqs, void* o, float* final_state, int B, int T, int H,
                           int K, int V, kda_dtype dtype, void* stream);

/* Human-readable name of a kda_status value (static storage, never NULL). */
const char* kda_status_string(int status);

/* Reads the device status word that kernels of the last kda_fwd on this workspace
 * set when they abandon a bounded wait.  Synchronises `stream`.  Returns KDA_OK,
 * KDA_ERR_DEVICE_TIMEOUT, or KDA_ERR_CUDA if the copy failed. */
kda_status kda_get_device_status(const void* workspace, void* stream);

/* Diagnostic: D[128][N] = A[128][K] * B[N][K]^T (bf16 row-major inputs, fp32 row-major
 * output) computed by one CTA with the same tcgen05 MMA, tensor-memory, mbarrier and
 * 128-byte-swizzled operand building blocks as the bf16 kernels.  Mode 0 stages A and B
 * with TMA tensor loads, mode 1 writes them from registers with the software swizzle.
 * N in {16, 32, 64, 128, 256}; K a multiple of 16 in [16, 128].  *status (device int,
 * zeroed by the caller) receives KDA_ERR_DEVICE_TIMEOUT if a bounded wait expires.
 * Used by the tests to check the building blocks in isolation; not part of the
 * forward pass.  Modes 2 and 3 check the MN-major operand form: in mode 2 B is given as
 * its transpose [K][N] (N >= 64), in mode 3 A is given as its transpose [K][128]; the
 * result is the same product.  Mode 4 keeps A in tensor memory (written with
 * tcgen05.st) and B in shared memory. */
kda_status kda_selftest_umma(const void* A, const void* B, float* D, int N, int K, int mode,
                             int* status, void* stream);

/* Number of kernel launches kda_fwd makes for these sizes on the current device: the
 * chunk-index kernel (packed input, and the fp32 / other-shape path), the intra-chunk
 * kernel and the recurrence kernel (pipelined calls launch the last two once per chunk
 * range; fused calls make one launch, scan calls four); -1 for sizes kda_fwd rejects. */
int kda_fwd_launch_count(int B, int T, int H, int K, int V, int num_seqs, int chunk_size,
                         kda_dtype dtype);

/* Schedule kda_fwd takes for these sizes on the current device (see kda_fwd), or -1 for
 * sizes kda_fwd rejects.  kda_fwd_profiled always runs the two-kernel schedule. */
typedef enum {
    KDA_SCHEDULE_TWO_KERNELS = 0,
    KDA_SCHEDULE_PIPELINED = 1,
    KDA_SCHEDULE_FUSED = 2,
    KDA_SCHEDULE_SCAN = 3
} kda_schedule;
int kda_fwd_schedule(int B, int T, int H, int K, int V, int num_seqs, int chunk_size,
                     kda_dtype dtype);

/* The same choice for a device with `sm_count` SMs (152 on a GB300), whichever device is
 * current, e.g. to plan shapes ahead of a call; the environment override KDA_SCHEDULE
 * applies as in kda_fwd.  -1 for sizes kda_fwd rejects or a negative sm_count.  With
 * sm_count 0 neither the fused nor the scan schedule is chosen (both size their grids by
 * the SM count). */
int kda_fwd_schedule_for(int B, int T, int H, int K, int V, int num_seqs, int chunk_size,
                         kda_dtype dtype, int sm_count);

/* Version of this ABI (major * 100 + minor). */
int kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
