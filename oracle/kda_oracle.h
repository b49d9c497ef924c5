/*
 * kda_oracle.h -- fp64 CPU oracle for the forward pass of Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE.  This code exists to check the CUDA library against the
 * method's definition.  Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg use it; the product path never links, loads or calls it, and it
 * shares no code, header, table or helper with the CUDA sources.
 *
 * Sources (web pages, cited by title and section):
 *   [TKD]  Tokamax, "chunk_kda_fwd_design_doc" (KDA forward design document),
 *          Appendix 9.1: Eq. (1) token recurrence and its delta-correction form,
 *          Eq. (2)-(9) chunkwise form, 9.1.7 variable-length sequences.
 *   [KDF]  "KDA Doesn't Care About the Future", section "Chunkwise KDA in Broad
 *          Strokes" (the six-step recurrence, update-before-read) and "Chunkwise Aqk".
 *   [KCW]  Kimi-K3 docs, "KDAChunkwise" (readable chunkwise reference, walk-through).
 *
 * Tensor layouts (row-major, token-major, as the CUDA library uses them):
 *   q, k : [B, T, H, K]     v : [B, T, H, V]     g : [B, T, H, K]   beta : [B, T, H]
 *   o    : [B, T, H, V]     initial_state / final_state : [N, H, K, V]
 * with N = B (fixed length) or N = num_seqs (packed variable length, B == 1,
 * cu_seqlens[0..N] the token offsets).  A state row is a key channel, a column a
 * value channel: S[d][j].
 *
 * g holds natural-log decays, alpha_t = exp(g_t) (g <= 0 in production use).
 * All arithmetic is IEEE fp64 in program order (compiled with -ffp-contract=off).
 *
 * Return value: number of worker threads used (>= 1), or a negative value for
 * invalid arguments (-1) or out-of-memory (-2).
 */
#ifndef KDA_ORACLE_H
#define KDA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Token-by-token recurrence, [TKD] 9.1.2 Eq. (1) in its delta-correction form:
 *   S_bar = Diag(alpha_t) S_{t-1};  e_t = v_t - S_bar^T k_t;
 *   S_t = S_bar + beta_t k_t e_t^T;  o_t = scale * S_t^T q_t.
 * initial_state (nullable) and final_state (nullable) are [N,H,K,V].
 * cu_seqlens (nullable) requires B == 1.  num_threads <= 0 means "all online CPUs". */
int kda_oracle_recurrent(const double* q, const double* k, const double* v,
                         const double* g, const double* beta, double scale,
                         const double* initial_state, const int32_t* cu_seqlens,
                         int num_seqs, int B, int T, int H, int K, int V,
                         double* o, double* final_state, int num_threads);

/* Chunkwise form, [TKD] 9.1.3-9.1.6 (Eq. (6)-(9)) with chunk size C >= 1 and a
 * shorter last chunk where a sequence length is not a multiple of C.  Independent
 * of kda_oracle_recurrent: exact exponentials of gate differences, a dense
 * unit-lower-triangular forward substitution, no rebasing. */
int kda_oracle_chunkwise(const double* q, const double* k, const double* v,
                         const double* g, const double* beta, double scale,
                         const double* initial_state, const int32_t* cu_seqlens,
                         int num_seqs, int B, int T, int H, int K, int V,
                         int chunk_size, double* o, double* final_state,
                         int num_threads);

/* Gate activation of a raw gate, [TKD] 9.1.3 (use_gate_in_kernel):
 *   x' = x + dt_bias[h][d] (dt_bias nullable, [H][K]), lambda_h = exp(a_log[h]);
 *   lower_bound == 0:  ell = -lambda_h * softplus(x'),  softplus(y) = ln(1 + e^y);
 *   otherwise:         ell = lower_bound * sigmoid(lambda_h x'),  sigmoid(y) = 1/(1+e^-y).
 * x and ell are [rows][H][K] (rows = B * T).  Returns 1, or -1 for invalid arguments. */
/* Affine summary of every chunk of fixed-length input ([TKD] context-parallel section):
 * the chunk maps its start state S to Phi S + Psi with Phi = Diag(gamma^C) - K_bar^T W
 * (K x K) and Psi = K_bar^T U (K x V), W, U, K_bar and gamma^C as in the chunkwise form.
 * phi: [B][H][nct][K][K], psi: [B][H][nct][K][V], nct = ceil(T / chunk_size). */
int kda_oracle_chunk_summaries(const double* q, const double* k, const double* v,
                               const double* g, const double* beta, double scale, int B, int T,
                               int H, int K, int V, int chunk_size, double* phi, double* psi,
                               int num_threads);

int kda_oracle_gate(const double* x, const double* a_log, const double* dt_bias,
                    double lower_bound, long rows, int H, int K, double* ell);

/* Row normalisation along the last dimension, [KCW] "FP32 core and log-space decay"
 * (F.normalize): y = x / max(||x||_2, eps).  x, y: [rows][D].  Returns 1 or -1. */
int kda_oracle_l2norm(const double* x, long rows, int D, double eps, double* y);

#ifdef __cplusplus
}
#endif

#endif /* KDA_ORACLE_H */
