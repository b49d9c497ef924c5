/*
 * kda_oracle.c -- fp64 CPU oracle for the forward pass of Kimi Delta Attention.
 *
 * TEST INFRASTRUCTURE: see kda_oracle.h.  Plain, slow, obviously correct; no
 * blocking, fusion or reordering beyond what the cited definitions state.  Worker
 * threads only split independent (sequence, head) units.
 *
 * Parity pins (tests/pins.py) tie both functions to facts outside this file:
 * exact rational evaluation of Eq. (1) in its matrix-product form, textbook causal
 * linear attention (orthogonal keys, no decay), the beta = 0 freeze, the state-norm
 * bound, causality, split-call resume, sequence isolation, and recurrent == chunkwise.
 */
#include "kda_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------- */
/* Shared argument block and (sequence, head) work distribution               */
/* ------------------------------------------------------------------------- */

typedef struct {
    const double *q, *k, *v, *g, *beta;
    double scale;
    const double* initial_state;
    const int32_t* cu_seqlens;
    int N, B, T, H, K, V, C;
    double *o, *final_state;
    int next_unit; /* atomic counter over N*H units */
    int failed;    /* set if a worker could not allocate */
} oracle_job;

/* Token range [begin, end) of sequence n in the flattened B*T token axis
 * ([TKD] 9.1.7: segment n is the interval [p_n, p_{n+1})). */
static void seq_range(const oracle_job* J, int n, long* begin, long* end) {
    if (J->cu_seqlens) {
        *begin = J->cu_seqlens[n];
        *end = J->cu_seqlens[n + 1];
    } else {
        *begin = (long)n * J->T;
        *end = (long)(n + 1) * J->T;
    }
}

static void load_initial_state(const oracle_job* J, int n, int h, double* S) {
    const size_t KV = (size_t)J->K * J->V;
    if (J->initial_state)
        memcpy(S, J->initial_state + ((size_t)n * J->H + h) * KV, KV * sizeof(double));
    else
        memset(S, 0, KV * sizeof(double));
}

static void store_final_state(const oracle_job* J, int n, int h, const double* S) {
    const size_t KV = (size_t)J->K * J->V;
    if (J->final_state)
        memcpy(J->final_state + ((size_t)n * J->H + h) * KV, S, KV * sizeof(double));
}

/* ------------------------------------------------------------------------- */
/* Token recurrence ([TKD] 9.1.2; [KDF] "Chunkwise KDA in Broad Strokes")      */
/* ------------------------------------------------------------------------- */

static int recurrent_unit(const oracle_job* J, int n, int h) {
    const int H = J->H, K = J->K, V = J->V;
    double* S = (double*)malloc((size_t)K * V * sizeof(double));
    double* e = (double*)malloc((size_t)V * sizeof(double));
    if (!S || !e) {
        free(S);
        free(e);
        return -2;
    }
    load_initial_state(J, n, h, S);
    long t0, t1;
    seq_range(J, n, &t0, &t1);
    for (long t = t0; t < t1; ++t) {
        const double* qt = J->q + ((size_t)t * H + h) * K;
        const double* kt = J->k + ((size_t)t * H + h) * K;
        const double* vt = J->v + ((size_t)t * H + h) * V;
        const double* gt = J->g + ((size_t)t * H + h) * K;
        const double bt = J->beta[(size_t)t * H + h];
        double* ot = J->o + ((size_t)t * H + h) * V;

        /* S_bar = Diag(alpha_t) S_{t-1}, alpha_t = exp(g_t): each key-channel row
         * of the state decays by its own factor before the write. */
        for (int d = 0; d < K; ++d) {
            const double alpha = exp(gt[d]);
            for (int j = 0; j < V; ++j) S[(size_t)d * V + j] *= alpha;
        }
        /* e_t = v_t - S_bar^T k_t: the value the decayed state already associates
         * with k_t, subtracted from the new value. */
        for (int j = 0; j < V; ++j) {
            double pred = 0.0;
            for (int d = 0; d < K; ++d) pred += S[(size_t)d * V + j] * kt[d];
            e[j] = vt[j] - pred;
        }
        /* S_t = S_bar + beta_t k_t e_t^T: rank-1 delta correction at key k_t. */
        for (int d = 0; d < K; ++d) {
            const double bk = bt * kt[d];
            for (int j = 0; j < V; ++j) S[(size_t)d * V + j] += bk * e[j];
        }
        /* o_t = scale * S_t^T q_t: the query reads the state after this token's
         * own write (update before read). */
        for (int j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int d = 0; d < K; ++d) acc += S[(size_t)d * V + j] * qt[d];
            ot[j] = J->scale * acc;
        }
    }
    store_final_state(J, n, h, S);
    free(S);
    free(e);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Chunkwise form ([TKD] 9.1.3-9.1.6, Eq. (6)-(9))                             */
/* ------------------------------------------------------------------------- */

typedef struct {
    double *G, *L, *Aqk, *A, *W, *U, *Kbar, *Vnew, *Snew;
} chunk_scratch;

static void free_scratch(chunk_scratch* s) {
    free(s->G);
    free(s->L);
    free(s->Aqk);
    free(s->A);
    free(s->W);
    free(s->U);
    free(s->Kbar);
    free(s->Vnew);
    free(s->Snew);
}

static int alloc_scratch(chunk_scratch* s, int C, int K, int V) {
    memset(s, 0, sizeof(*s));
    s->G = (double*)malloc((size_t)C * K * sizeof(double));
    s->L = (double*)malloc((size_t)C * C * sizeof(double));
    s->Aqk = (double*)malloc((size_t)C * C * sizeof(double));
    s->A = (double*)malloc((size_t)C * C * sizeof(double));
    s->W = (double*)malloc((size_t)C * K * sizeof(double));
    s->U = (double*)malloc((size_t)C * V * sizeof(double));
    s->Kbar = (double*)malloc((size_t)C * K * sizeof(double));
    s->Vnew = (double*)malloc((size_t)C * V * sizeof(double));
    s->Snew = (double*)malloc((size_t)K * V * sizeof(double));
    if (!s->G || !s->L || !s->Aqk || !s->A || !s->W || !s->U || !s->Kbar || !s->Vnew ||
        !s->Snew) {
        free_scratch(s);
        return -2;
    }
    return 0;
}

/* One chunk of c tokens starting at flattened token t0, head h; S is the
 * chunk-start state S_c^0 on entry and S_{c+1}^0 on exit. */
static void chunk_step(const oracle_job* J, int h, long t0, int c, double* S, chunk_scratch* s) {
    const int H = J->H, K = J->K, V = J->V;
    const double inv_ln2 = 1.0 / log(2.0);
#define Q_(r, d) J->q[((size_t)(t0 + (r)) * H + h) * K + (d)]
#define K_(r, d) J->k[((size_t)(t0 + (r)) * H + h) * K + (d)]
#define V_(r, j) J->v[((size_t)(t0 + (r)) * H + h) * V + (j)]
#define GATE(r, d) J->g[((size_t)(t0 + (r)) * H + h) * K + (d)]
#define BETA(r) J->beta[(size_t)(t0 + (r)) * H + h]
#define G_(r, d) s->G[(size_t)(r) * K + (d)]

    /* 9.1.3: G^r = (1/ln 2) * sum_{m <= r} l^m, chunk-local, inclusive of token r;
     * gamma^r = 2^{G^r}, rho^{i->r} = 2^{G^r - G^i}. */
    for (int d = 0; d < K; ++d) {
        double acc = 0.0;
        for (int r = 0; r < c; ++r) {
            acc += GATE(r, d);
            G_(r, d) = acc * inv_ln2;
        }
    }

    /* 9.1.5: L = StrictTril(D_beta K+ (K-)^T), entries beta_i sum_d k_i k_j 2^{G_i-G_j};
     *        Aqk = Tril((Gamma . Q~)(K-)^T), entries scale sum_d q_i k_j 2^{G_i-G_j}.
     * The gate ratio is evaluated directly as exp2 of the difference (exact math,
     * no split into separately scaled operands). */
    for (int i = 0; i < c; ++i) {
        for (int j = 0; j < c; ++j) {
            double lij = 0.0, aij = 0.0;
            if (j <= i) {
                for (int d = 0; d < K; ++d) {
                    const double rho = exp2(G_(i, d) - G_(j, d));
                    lij += K_(i, d) * K_(j, d) * rho;
                    aij += Q_(i, d) * K_(j, d) * rho;
                }
            }
            s->L[(size_t)i * c + j] = (j < i) ? BETA(i) * lij : 0.0;
            s->Aqk[(size_t)i * c + j] = (j <= i) ? J->scale * aij : 0.0;
        }
    }

    /* 9.1.5 Eq. (6): A = (I + L)^{-1}, by forward substitution on the identity:
     * row r of A solves A[r,:] = e_r - sum_{j<r} L[r,j] A[j,:]. */
    for (int r = 0; r < c; ++r) {
        for (int col = 0; col < c; ++col) {
            double x = (r == col) ? 1.0 : 0.0;
            for (int j = 0; j < r; ++j) x -= s->L[(size_t)r * c + j] * s->A[(size_t)j * c + col];
            s->A[(size_t)r * c + col] = x;
        }
    }

    /* 9.1.5 Eq. (7): W = A (D_beta K+), U = A (D_beta V), K+ = Gamma . K. */
    for (int r = 0; r < c; ++r) {
        for (int d = 0; d < K; ++d) {
            double acc = 0.0;
            for (int j = 0; j < c; ++j)
                acc += s->A[(size_t)r * c + j] * BETA(j) * exp2(G_(j, d)) * K_(j, d);
            s->W[(size_t)r * K + d] = acc;
        }
        for (int jv = 0; jv < V; ++jv) {
            double acc = 0.0;
            for (int j = 0; j < c; ++j) acc += s->A[(size_t)r * c + j] * BETA(j) * V_(j, jv);
            s->U[(size_t)r * V + jv] = acc;
        }
    }

    /* 9.1.5: K_bar^r = k^r . 2^{G^C - G^r} (each key carried to the chunk end). */
    for (int r = 0; r < c; ++r)
        for (int d = 0; d < K; ++d)
            s->Kbar[(size_t)r * K + d] = K_(r, d) * exp2(G_(c - 1, d) - G_(r, d));

    /* 9.1.6: V_new = U - W S. */
    for (int r = 0; r < c; ++r) {
        for (int jv = 0; jv < V; ++jv) {
            double acc = 0.0;
            for (int d = 0; d < K; ++d) acc += s->W[(size_t)r * K + d] * S[(size_t)d * V + jv];
            s->Vnew[(size_t)r * V + jv] = s->U[(size_t)r * V + jv] - acc;
        }
    }

    /* 9.1.6 Eq. (9): O = (Gamma . Q~) S + Aqk V_new, Q~ = scale * Q. */
    for (int r = 0; r < c; ++r) {
        double* orow = J->o + ((size_t)(t0 + r) * H + h) * V;
        for (int jv = 0; jv < V; ++jv) {
            double inter = 0.0, intra = 0.0;
            for (int d = 0; d < K; ++d)
                inter += J->scale * Q_(r, d) * exp2(G_(r, d)) * S[(size_t)d * V + jv];
            for (int j = 0; j < c; ++j) intra += s->Aqk[(size_t)r * c + j] * s->Vnew[(size_t)j * V + jv];
            orow[jv] = inter + intra;
        }
    }

    /* 9.1.6 Eq. (8): S' = Diag(gamma^C) S + K_bar^T V_new. */
    for (int d = 0; d < K; ++d) {
        const double gammaC = exp2(G_(c - 1, d));
        for (int jv = 0; jv < V; ++jv) {
            double acc = 0.0;
            for (int r = 0; r < c; ++r) acc += s->Kbar[(size_t)r * K + d] * s->Vnew[(size_t)r * V + jv];
            s->Snew[(size_t)d * V + jv] = gammaC * S[(size_t)d * V + jv] + acc;
        }
    }
    memcpy(S, s->Snew, (size_t)K * V * sizeof(double));
#undef Q_
#undef K_
#undef V_
#undef GATE
#undef BETA
#undef G_
}

static int chunkwise_unit(const oracle_job* J, int n, int h) {
    chunk_scratch s;
    if (alloc_scratch(&s, J->C, J->K, J->V)) return -2;
    double* S = (double*)malloc((size_t)J->K * J->V * sizeof(double));
    if (!S) {
        free_scratch(&s);
        return -2;
    }
    load_initial_state(J, n, h, S);
    long t0, t1;
    seq_range(J, n, &t0, &t1);
    /* 9.1.7: chunks never cross a sequence; the last one may be shorter. */
    for (long c0 = t0; c0 < t1; c0 += J->C) {
        const int c = (int)((t1 - c0) < J->C ? (t1 - c0) : J->C);
        chunk_step(J, h, c0, c, S, &s);
    }
    store_final_state(J, n, h, S);
    free(S);
    free_scratch(&s);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Affine chunk summaries ([TKD] context-parallel section: each chunk maps its */
/* start state affinely, S' = Phi S + Psi)                                    */
/* ------------------------------------------------------------------------- */

/* The summary job reuses oracle_job: o points at a scratch output the chunk steps may
 * overwrite, final_state at Phi [N][H][nct][K][K] and initial_state at Psi
 * [N][H][nct][K][V] (both written; cast away const for Psi). */
static int summary_unit(const oracle_job* J, int n, int h) {
    const int K = J->K, V = J->V;
    chunk_scratch s;
    if (alloc_scratch(&s, J->C, K, V)) return -2;
    double* S = (double*)malloc((size_t)K * V * sizeof(double));
    if (!S) {
        free_scratch(&s);
        return -2;
    }
    long t0, t1;
    seq_range(J, n, &t0, &t1);
    const long nct = ((long)J->T + J->C - 1) / J->C;
    double* Phi = J->final_state;
    double* Psi = (double*)J->initial_state;
    long j = 0;
    for (long c0 = t0; c0 < t1; c0 += J->C, ++j) {
        const int c = (int)((t1 - c0) < J->C ? (t1 - c0) : J->C);
        /* the chunk's W, U, K_bar and G do not depend on the state it starts from */
        memset(S, 0, (size_t)K * V * sizeof(double));
        chunk_step(J, h, c0, c, S, &s);
        double* phi = Phi + (((size_t)n * J->H + h) * nct + j) * K * K;
        double* psi = Psi + (((size_t)n * J->H + h) * nct + j) * K * V;
        /* Phi = Diag(gamma^C) - K_bar^T W;  Psi = K_bar^T U  (gamma^C = 2^{G^{C-1}}) */
        for (int d = 0; d < K; ++d) {
            for (int e = 0; e < K; ++e) {
                double acc = 0.0;
                for (int r = 0; r < c; ++r) acc += s.Kbar[(size_t)r * K + d] * s.W[(size_t)r * K + e];
                phi[(size_t)d * K + e] = (d == e ? exp2(s.G[(size_t)(c - 1) * K + d]) : 0.0) - acc;
            }
            for (int jv = 0; jv < V; ++jv) {
                double acc = 0.0;
                for (int r = 0; r < c; ++r) acc += s.Kbar[(size_t)r * K + d] * s.U[(size_t)r * V + jv];
                psi[(size_t)d * V + jv] = acc;
            }
        }
    }
    free(S);
    free_scratch(&s);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Threading and argument checks                                              */
/* ------------------------------------------------------------------------- */

typedef struct {
    oracle_job* job;
    int (*unit)(const oracle_job*, int, int);
} worker_arg;

static void* worker(void* p) {
    worker_arg* w = (worker_arg*)p;
    oracle_job* J = w->job;
    const int units = J->N * J->H;
    for (;;) {
        const int u = __atomic_fetch_add(&J->next_unit, 1, __ATOMIC_RELAXED);
        if (u >= units) break;
        if (w->unit(J, u / J->H, u % J->H)) __atomic_store_n(&J->failed, 1, __ATOMIC_RELAXED);
    }
    return NULL;
}

static int run(oracle_job* J, int (*unit)(const oracle_job*, int, int), int num_threads) {
    const int units = J->N * J->H;
    if (num_threads <= 0) {
        const long ncpu = sysconf(_SC_NPROCESSORS_ONLN);
        num_threads = ncpu > 0 ? (int)ncpu : 1;
    }
    if (num_threads > units) num_threads = units > 0 ? units : 1;
    worker_arg wa = {J, unit};
    if (num_threads == 1) {
        worker(&wa);
    } else {
        pthread_t* th = (pthread_t*)malloc((size_t)num_threads * sizeof(pthread_t));
        if (!th) return -2;
        int started = 0;
        for (int i = 0; i < num_threads; ++i)
            if (pthread_create(&th[i], NULL, worker, &wa) == 0) ++started;
        if (started == 0) worker(&wa);
        for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
        free(th);
        num_threads = started > 0 ? started : 1;
    }
    return J->failed ? -2 : num_threads;
}

static int fill_job(oracle_job* J, const double* q, const double* k, const double* v,
                    const double* g, const double* beta, double scale,
                    const double* initial_state, const int32_t* cu_seqlens, int num_seqs,
                    int B, int T, int H, int K, int V, int C, double* o, double* final_state) {
    if (!q || !k || !v || !g || !beta || !o) return -1;
    if (B < 1 || T < 0 || H < 1 || K < 1 || V < 1 || C < 1) return -1;
    if (cu_seqlens) {
        if (B != 1 || num_seqs < 0) return -1;
        if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != T) return -1;
        for (int n = 0; n < num_seqs; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    }
    memset(J, 0, sizeof(*J));
    J->q = q;
    J->k = k;
    J->v = v;
    J->g = g;
    J->beta = beta;
    J->scale = scale;
    J->initial_state = initial_state;
    J->cu_seqlens = cu_seqlens;
    J->N = cu_seqlens ? num_seqs : B;
    J->B = B;
    J->T = T;
    J->H = H;
    J->K = K;
    J->V = V;
    J->C = C;
    J->o = o;
    J->final_state = final_state;
    return 0;
}

int kda_oracle_recurrent(const double* q, const double* k, const double* v,
                         const double* g, const double* beta, double scale,
                         const double* initial_state, const int32_t* cu_seqlens,
                         int num_seqs, int B, int T, int H, int K, int V,
                         double* o, double* final_state, int num_threads) {
    oracle_job J;
    if (fill_job(&J, q, k, v, g, beta, scale, initial_state, cu_seqlens, num_seqs, B, T, H, K, V,
                 1, o, final_state))
        return -1;
    return run(&J, recurrent_unit, num_threads);
}

int kda_oracle_chunk_summaries(const double* q, const double* k, const double* v,
                               const double* g, const double* beta, double scale, int B, int T,
                               int H, int K, int V, int chunk_size, double* phi, double* psi,
                               int num_threads) {
    oracle_job J;
    if (!phi || !psi) return -1;
    double* o_scratch = (double*)malloc(((size_t)B * T * H * V + 1) * sizeof(double));
    if (!o_scratch) return -2;
    const int rc = fill_job(&J, q, k, v, g, beta, scale, psi, NULL, 0, B, T, H, K, V, chunk_size,
                            o_scratch, phi);
    int out = rc ? -1 : run(&J, summary_unit, num_threads);
    free(o_scratch);
    return out;
}

int kda_oracle_chunkwise(const double* q, const double* k, const double* v,
                         const double* g, const double* beta, double scale,
                         const double* initial_state, const int32_t* cu_seqlens,
                         int num_seqs, int B, int T, int H, int K, int V,
                         int chunk_size, double* o, double* final_state,
                         int num_threads) {
    oracle_job J;
    if (fill_job(&J, q, k, v, g, beta, scale, initial_state, cu_seqlens, num_seqs, B, T, H, K, V,
                 chunk_size, o, final_state))
        return -1;
    return run(&J, chunkwise_unit, num_threads);
}

/* ------------------------------------------------------------------------------------
 * Gate activation and row normalisation (the inputs of use_gate_in_kernel / q-k
 * normalisation; applied before the recurrence, which then takes ell = ln(alpha)).
 * ------------------------------------------------------------------------------------ */

/* softplus(y) = ln(1 + e^y), evaluated as max(y, 0) + ln(1 + e^{-|y|}) (the same value,
 * without overflow of e^y for large y). */
static double softplus(double y) {
    const double a = y > 0.0 ? y : -y;
    return (y > 0.0 ? y : 0.0) + log1p(exp(-a));
}

/* sigmoid(y) = 1 / (1 + e^{-y}). */
static double sigmoid(double y) { return 1.0 / (1.0 + exp(-y)); }

int kda_oracle_gate(const double* x, const double* a_log, const double* dt_bias,
                    double lower_bound, long rows, int H, int K, double* ell) {
    if (!x || !a_log || !ell || rows < 0 || H < 1 || K < 1) return -1;
    for (long r = 0; r < rows; ++r) {
        for (int h = 0; h < H; ++h) {
            const double lam = exp(a_log[h]);
            for (int d = 0; d < K; ++d) {
                const size_t i = ((size_t)r * H + h) * K + d;
                double xb = x[i];
                if (dt_bias) xb += dt_bias[(size_t)h * K + d];
                ell[i] = lower_bound == 0.0 ? -lam * softplus(xb) : lower_bound * sigmoid(lam * xb);
            }
        }
    }
    return 1;
}

int kda_oracle_l2norm(const double* x, long rows, int D, double eps, double* y) {
    if (!x || !y || rows < 0 || D < 1) return -1;
    for (long r = 0; r < rows; ++r) {
        const double* xr = x + (size_t)r * D;
        double ss = 0.0;
        for (int d = 0; d < D; ++d) ss += xr[d] * xr[d];
        double n = sqrt(ss);
        if (n < eps) n = eps;
        for (int d = 0; d < D; ++d) y[(size_t)r * D + d] = xr[d] / n;
    }
    return 1;
}
