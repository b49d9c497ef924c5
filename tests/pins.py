"""Pins of the fp64 oracle to facts outside the oracle itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with the fact.  ``tests/test_oracle_pins.py`` runs them on the committed
oracle; ``tests/test_oracle_mutants.py`` runs them on copies of the oracle with one
planted mistake each and requires that some pin fails for every copy.

Sources (web pages, by title and section):
  Tokamax "chunk_kda_fwd_design_doc", Appendix 9.1.2 (Eq. (1) and its delta-correction
  form), 9.1.3-9.1.6 (chunkwise Eq. (6)-(9)), 9.1.7 (variable-length sequences);
  "KDA Doesn't Care About the Future", "Chunkwise KDA in Broad Strokes" and
  "Decisions Decisions" (causality); Kimi-K3 "KDAChunkwise", "Verification and
  boundaries" (chunkwise-vs-recurrent test idea, chunk sizes 1, 2, 4, 8) and "FP32 core
  and log-space decay" (q/k normalisation); Tokamax 9.1.3 and 5.3 (raw-gate forms).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

RECURRENT = "recurrent"


def run(oracle, form, *args, chunk_size=None, **kw):
    """Call one oracle form; ``form`` is "recurrent" or a chunk size (int)."""
    if form == RECURRENT:
        return oracle.recurrent(*args, **kw)
    return oracle.chunkwise(*args[:6], chunk_size=form, **kw)


FORMS = (RECURRENT, 1, 2, 3, 16, 64)


def _rand_inputs(rng, B, T, H, K, V, unit_keys=True, g_max=5.0, beta_range=(0.0, 1.0)):
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    if unit_keys:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    g = -g_max * rng.random((B, T, H, K))
    beta = rng.uniform(*beta_range, size=(B, T, H))
    return q, k, v, g, beta


# ---------------------------------------------------------------------------
# P-1: exact rational evaluation of Eq. (1) in its matrix-product form
# ---------------------------------------------------------------------------

def _eq1_exact(q, k, v, alpha, beta, scale, S0, seqs, H, K, V):
    """S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = S_t^T (scale q_t), evaluated with Fractions (Tokamax design doc 9.1.2,
    Eq. (1)); each sequence restarts from its own initial state (9.1.7)."""
    T = len(q)
    o = [[[Fraction(0)] * V for _ in range(H)] for _ in range(T)]
    finals = []
    for n, (t0, t1) in enumerate(seqs):
        fin_n = []
        for h in range(H):
            S = [[S0[n][h][d][j] for j in range(V)] for d in range(K)]
            for t in range(t0, t1):
                kt, vt, qt, at, bt = k[t][h], v[t][h], q[t][h], alpha[t][h], beta[t][h]
                # M = (I - b k k^T) Diag(a): M[d][e] = (delta_de - b k_d k_e) a_e
                M = [[((1 if d == e else 0) - bt * kt[d] * kt[e]) * at[e] for e in range(K)]
                     for d in range(K)]
                S = [[sum(M[d][e] * S[e][j] for e in range(K)) + bt * kt[d] * vt[j]
                      for j in range(V)] for d in range(K)]
                o[t][h] = [sum(S[d][j] * scale * qt[d] for d in range(K)) for j in range(V)]
            fin_n.append(S)
        finals.append(fin_n)
    return o, finals


def pin_eq1_exact_rational(oracle, forms=FORMS):
    rng = np.random.default_rng(11)
    H, K, V = 2, 3, 2
    lens = [4, 0, 5, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, N = int(cu[-1]), len(lens)
    seqs = [(int(cu[i]), int(cu[i + 1])) for i in range(N)]

    def rat(lo, hi, den, shape):
        return [[[Fraction(int(x), den) for x in row] for row in block]
                for block in rng.integers(lo, hi + 1, size=shape)]

    q = rat(-8, 8, 8, (T, H, K))
    k = rat(-8, 8, 8, (T, H, K))
    v = rat(-8, 8, 4, (T, H, V))
    alpha_choices = [Fraction(1, 2), Fraction(3, 4), Fraction(7, 8), Fraction(1), Fraction(5, 8)]
    alpha = [[[alpha_choices[int(rng.integers(0, 5))] for _ in range(K)] for _ in range(H)]
             for _ in range(T)]
    beta = [[Fraction(int(rng.integers(1, 5)), 4) for _ in range(H)] for _ in range(T)]
    S0 = [[[[Fraction(int(rng.integers(-4, 5)), 4) for _ in range(V)] for _ in range(K)]
           for _ in range(H)] for _ in range(N)]
    scale = Fraction(3, 4)
    o_ex, fin_ex = _eq1_exact(q, k, v, alpha, beta, scale, S0, seqs, H, K, V)

    f = lambda x: np.array(x, dtype=np.float64)
    qa, ka, va = f(q)[None], f(k)[None], f(v)[None]
    ga = np.log(f(alpha))[None]
    ba = f(beta)[None]
    s0 = f(S0)
    o_ex, fin_ex = f(o_ex)[None], f(fin_ex)
    for form in forms:
        o, fin = run(oracle, form, qa, ka, va, ga, ba, float(scale), initial_state=s0,
                     cu_seqlens=cu)
        assert np.allclose(o, o_ex, rtol=0, atol=1e-12), f"Eq.(1) output mismatch ({form})"
        assert np.allclose(fin, fin_ex, rtol=0, atol=1e-12), f"Eq.(1) state mismatch ({form})"


# ---------------------------------------------------------------------------
# P-3: orthogonal keys, no decay -> (beta-weighted) causal linear attention
# ---------------------------------------------------------------------------

def pin_linear_attention(oracle, forms=FORMS):
    """With g = 0, S_0 = 0 and mutually orthonormal keys, S_{t-1}^T k_t = 0 before each
    write, so o_t = scale * sum_{j<=t} beta_j (q_t . k_j) v_j; with beta = 1 this is the
    textbook causal linear attention sum (brute force, O(T^2))."""
    rng = np.random.default_rng(12)
    B, T, H, K, V = 2, 24, 2, 32, 8
    q = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, H, V))
    k = np.empty((B, T, H, K))
    for b in range(B):
        for h in range(H):
            Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
            k[b, :, h, :] = Qm[:T]          # T orthonormal rows
    g = np.zeros((B, T, H, K))
    scale = 0.37
    for beta in (np.ones((B, T, H)), rng.uniform(0.1, 0.9, (B, T, H))):
        ref = np.zeros((B, T, H, V))
        for b in range(B):
            for h in range(H):
                for t in range(T):
                    acc = np.zeros(V)
                    for j in range(t + 1):
                        acc += beta[b, j, h] * np.dot(q[b, t, h], k[b, j, h]) * v[b, j, h]
                    ref[b, t, h] = scale * acc
        for form in forms:
            o, _ = run(oracle, form, q, k, v, g, beta, scale)
            assert np.allclose(o, ref, rtol=0, atol=1e-11), f"linear attention mismatch ({form})"


# ---------------------------------------------------------------------------
# Delta-rule retrieval: a full-strength write is read back exactly
# ---------------------------------------------------------------------------

def pin_delta_rule_retrieval(oracle, forms=FORMS):
    """With beta_t = 1 and a unit key, the write replaces what the decayed state held at
    k_t: S_t^T k_t = (Diag(alpha_t) S_{t-1})^T (I - k_t k_t^T) k_t + v_t (k_t . k_t) = v_t,
    whatever S_0 and the decays are (Tokamax 9.1.2, the delta-correction form of Eq. (1):
    the correction v_t - S^T k_t is written back in full).  So querying with q_t = k_t
    gives o_t = scale * v_t at every token."""
    rng = np.random.default_rng(21)
    B, T, H, K, V = 2, 40, 2, 16, 8
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    g = -5.0 * rng.random((B, T, H, K))
    beta = np.ones((B, T, H))
    s0 = rng.standard_normal((B, H, K, V))
    scale = 0.61
    for form in forms:
        o, fin = run(oracle, form, k.copy(), k, v, g, beta, scale, initial_state=s0)
        assert np.allclose(o, scale * v, rtol=0, atol=1e-10), f"retrieval mismatch ({form})"
        last = np.einsum("bhkv,bhk->bhv", fin, k[:, -1])
        assert np.allclose(last, v[:, -1], rtol=0, atol=1e-10), f"final-state retrieval ({form})"


# ---------------------------------------------------------------------------
# P-2: beta = 0 freezes the state up to its decay
# ---------------------------------------------------------------------------

def pin_beta_zero_freeze(oracle, forms=FORMS):
    """beta = 0 removes every write: S_t = Diag(exp(sum_{m<=t} g_m)) S_0 and
    o_t = scale * S_t^T q_t (Eq. (1) with beta_t = 0)."""
    rng = np.random.default_rng(13)
    B, T, H, K, V = 2, 37, 2, 16, 12
    q, k, v, g, _ = _rand_inputs(rng, B, T, H, K, V, g_max=0.3)
    beta = np.zeros((B, T, H))
    s0 = rng.standard_normal((B, H, K, V))
    scale = 0.25
    cum = np.cumsum(g, axis=1)                       # [B,T,H,K]
    St = np.exp(cum)[..., None] * s0[:, None]        # [B,T,H,K,V]
    ref_o = scale * np.einsum("bthkv,bthk->bthv", St, q)
    ref_f = St[:, -1]
    for form in forms:
        o, fin = run(oracle, form, q, k, v, g, beta, scale, initial_state=s0)
        assert np.allclose(o, ref_o, rtol=0, atol=1e-12), f"beta=0 output mismatch ({form})"
        assert np.allclose(fin, ref_f, rtol=0, atol=1e-12), f"beta=0 state mismatch ({form})"


# ---------------------------------------------------------------------------
# P-5: recurrent form == chunkwise form for several chunk sizes
# ---------------------------------------------------------------------------

def pin_recurrent_equals_chunkwise(oracle):
    """The chunkwise rewrite (Eq. (6)-(9)) reaches the token recurrence exactly up to
    rounding, for any chunk size, a short last chunk, packed sequences and an
    initial state (Kimi-K3 "KDAChunkwise" compares chunk sizes 1, 2, 4, 8)."""
    rng = np.random.default_rng(14)
    H, K, V = 2, 24, 20
    lens = [70, 1, 0, 64, 129]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v, g, beta = _rand_inputs(rng, 1, T, H, K, V)
    s0 = 0.1 * rng.standard_normal((len(lens), H, K, V))
    o_r, f_r = oracle.recurrent(q, k, v, g, beta, 0.3, initial_state=s0, cu_seqlens=cu)
    for C in (1, 2, 4, 8, 16, 33, 64):
        o_c, f_c = oracle.chunkwise(q, k, v, g, beta, 0.3, C, initial_state=s0, cu_seqlens=cu)
        assert np.max(np.abs(o_c - o_r)) <= 1e-10, f"chunkwise C={C} output differs"
        assert np.max(np.abs(f_c - f_r)) <= 1e-10, f"chunkwise C={C} state differs"


# ---------------------------------------------------------------------------
# P-6: state-norm bound for unit keys, beta in (0,1), g <= 0
# ---------------------------------------------------------------------------

def pin_state_norm_bound(oracle, forms=(RECURRENT, 4)):
    """||I - beta k k^T||_2 = 1 for unit k and beta in [0, 2], ||Diag(alpha)||_2 <= 1,
    so ||S_t||_2 <= ||S_{t-1}||_2 + beta_t ||v_t||_2 at every step."""
    rng = np.random.default_rng(15)
    T, H, K, V = 30, 1, 12, 10
    q, k, v, g, beta = _rand_inputs(rng, 1, T, H, K, V, g_max=0.05, beta_range=(0.05, 0.95))
    s0 = rng.standard_normal((1, H, K, V))
    for form in forms:
        prev = np.linalg.norm(s0[0, 0], 2)
        for t in range(1, T + 1):
            _, fin = run(oracle, form, q[:, :t], k[:, :t], v[:, :t], g[:, :t], beta[:, :t],
                         1.0, initial_state=s0)
            cur = np.linalg.norm(fin[0, 0], 2)
            bound = prev + beta[0, t - 1, 0] * np.linalg.norm(v[0, t - 1, 0])
            assert cur <= bound + 1e-12, f"state norm bound violated at t={t} ({form})"
            prev = cur


# ---------------------------------------------------------------------------
# P-7: causality
# ---------------------------------------------------------------------------

def pin_causality(oracle, forms=(RECURRENT, 16, 64)):
    """Perturbing q/k/v/g/beta after position n leaves o_{<=n} bit-identical ("KDA
    Doesn't Care About the Future", "Decisions Decisions")."""
    rng = np.random.default_rng(16)
    B, T, H, K, V = 1, 100, 2, 16, 16
    base = _rand_inputs(rng, B, T, H, K, V)
    for form in forms:
        o0, _ = run(oracle, form, *base, 0.5)
        for n in (0, 15, 16, 37, 63, 64, 98):
            pert = [x.copy() for x in base]
            for x in pert:
                x[:, n + 1:] = x[:, n + 1:] * 0.5 + 0.25
            pert[3] = np.minimum(pert[3], 0.0)
            o1, _ = run(oracle, form, *pert, 0.5)
            assert np.array_equal(o0[:, :n + 1], o1[:, :n + 1]), f"future leak at n={n} ({form})"
            assert not np.array_equal(o0[:, n + 1:], o1[:, n + 1:])


# ---------------------------------------------------------------------------
# P-8: split-call resume through final_state -> initial_state
# ---------------------------------------------------------------------------

def pin_split_resume(oracle, forms=(RECURRENT, 8)):
    rng = np.random.default_rng(17)
    B, T, H, K, V = 2, 90, 2, 8, 12
    q, k, v, g, beta = _rand_inputs(rng, B, T, H, K, V)
    s0 = rng.standard_normal((B, H, K, V))
    for form in forms:
        o_full, f_full = run(oracle, form, q, k, v, g, beta, 0.7, initial_state=s0)
        for a in (1, 37, 64):
            o1, f1 = run(oracle, form, q[:, :a], k[:, :a], v[:, :a], g[:, :a], beta[:, :a], 0.7,
                         initial_state=s0)
            o2, f2 = run(oracle, form, q[:, a:], k[:, a:], v[:, a:], g[:, a:], beta[:, a:], 0.7,
                         initial_state=f1)
            assert np.allclose(np.concatenate([o1, o2], axis=1), o_full, rtol=0, atol=1e-12)
            assert np.allclose(f2, f_full, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# P-11: packed sequences are isolated
# ---------------------------------------------------------------------------

def pin_varlen_isolation(oracle, forms=(RECURRENT, 64)):
    """Packing sequences with cu_seqlens equals running each one alone: state never
    crosses a sequence boundary (Tokamax design doc 9.1.7).  An empty sequence returns
    its initial state unchanged."""
    rng = np.random.default_rng(18)
    H, K, V = 2, 16, 8
    lens = [5, 0, 77, 64, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v, g, beta = _rand_inputs(rng, 1, T, H, K, V)
    s0 = rng.standard_normal((len(lens), H, K, V))
    for form in forms:
        o, fin = run(oracle, form, q, k, v, g, beta, 0.4, initial_state=s0, cu_seqlens=cu)
        for n, L in enumerate(lens):
            a, b = int(cu[n]), int(cu[n + 1])
            if L == 0:
                assert np.array_equal(fin[n], s0[n]), "empty sequence changed its state"
                continue
            o1, f1 = run(oracle, form, q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b],
                         beta[:, a:b], 0.4, initial_state=s0[n:n + 1])
            assert np.array_equal(o[:, a:b], o1), f"sequence {n} output differs when packed"
            assert np.array_equal(fin[n:n + 1], f1), f"sequence {n} state differs when packed"


def pin_gate_softplus(oracle):
    """Raw-gate softplus form (Tokamax design doc 9.1.3): ell = -exp(a_log) softplus(x + b).
    Facts of the mathematics: softplus(y) - softplus(-y) = y exactly in value, softplus(0)
    = ln 2, softplus(y) -> 0 for y -> -inf (the design doc's -1e4 raw-gate padding gives
    an identity decay), ell <= 0, ell is linear in exp(a_log), and dt_bias shifts x."""
    rng = np.random.default_rng(11)
    H, K = 3, 5
    x = rng.standard_normal((4, H, K)) * 3.0
    a_log = np.array([0.0, math.log(2.0), -0.7])
    b = rng.standard_normal(H * K)
    lam = np.exp(a_log)[None, :, None]
    e_pos = oracle.gate(x, a_log, None, 0.0)
    e_neg = oracle.gate(-x, a_log, None, 0.0)
    # -ell / lam = softplus(x): softplus(x) - softplus(-x) = x
    assert np.allclose(-e_pos / lam + e_neg / lam, x, rtol=0, atol=1e-13)
    assert np.all(e_pos <= 0.0)
    z = oracle.gate(np.zeros((1, H, K)), a_log, None, 0.0)
    assert np.allclose(z, -np.exp(a_log)[None, :, None] * math.log(2.0), rtol=0, atol=1e-15)
    pad = oracle.gate(np.full((1, H, K), -1e4), a_log, None, 0.0)
    assert np.all(np.abs(pad) < 1e-300)
    # exp(a_log) = 2 doubles the decay of exp(a_log) = 1
    assert np.allclose(e_pos[:, 1], 2.0 * oracle.gate(x, np.zeros(H), None, 0.0)[:, 1], atol=1e-14)
    # dt_bias adds to x before the activation
    shifted = x + b.reshape(H, K)[None]
    assert np.allclose(oracle.gate(x, a_log, b, 0.0), oracle.gate(shifted, a_log, None, 0.0),
                       rtol=0, atol=1e-14)


def pin_gate_sigmoid(oracle):
    """Lower-bound form (Tokamax design doc 9.1.3, 5.3): ell = a sigmoid(exp(a_log)(x + b))
    with -5 <= a < 0.  Facts: sigmoid(y) + sigmoid(-y) = 1, sigmoid(0) = 1/2, so ell lies in
    (a, 0), ell(x) + ell(-x) = a, ell(0) = a / 2, ell decreases with x, and exp(a_log)
    scales x."""
    rng = np.random.default_rng(12)
    H, K, a = 2, 6, -3.5
    x = rng.standard_normal((5, H, K)) * 2.0
    a_log = np.array([0.3, -1.2])
    e = oracle.gate(x, a_log, None, a)
    assert np.all((e < 0.0) & (e > a))
    assert np.allclose(e + oracle.gate(-x, a_log, None, a), a, rtol=0, atol=1e-14)
    assert np.allclose(oracle.gate(np.zeros((1, H, K)), a_log, None, a), a / 2, rtol=0, atol=1e-15)
    xs = np.sort(x, axis=0)
    es = oracle.gate(xs, a_log, None, a)
    assert np.all(np.diff(es, axis=0) <= 0.0)
    lam = np.exp(a_log)[None, :, None]
    assert np.allclose(e, oracle.gate(x * lam, np.zeros(H), None, a), rtol=0, atol=1e-14)
    b = rng.standard_normal(H * K)
    assert np.allclose(oracle.gate(x, a_log, b, a),
                       oracle.gate(x + b.reshape(H, K)[None], a_log, None, a), rtol=0, atol=1e-14)


def pin_l2norm(oracle):
    """x / max(||x||_2, eps) ("KDAChunkwise", F.normalize with eps 1e-6): rows of norm
    >= eps come out with norm 1 and the direction of x, a 3-4-5 row is exact, rows below
    eps are divided by eps, the zero row stays zero."""
    rng = np.random.default_rng(13)
    x = rng.standard_normal((7, 9)) * rng.uniform(0.1, 10.0, (7, 1))
    y = oracle.l2norm(x)
    assert np.allclose(np.linalg.norm(y, axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.allclose(y * np.linalg.norm(x, axis=1, keepdims=True), x, rtol=1e-14, atol=0)
    assert np.array_equal(oracle.l2norm(np.array([[3.0, 4.0]])), np.array([[0.6, 0.8]]))
    tiny = np.array([[3e-8, 4e-8], [0.0, 0.0]])
    assert np.allclose(oracle.l2norm(tiny), [[3e-2, 4e-2], [0.0, 0.0]], rtol=1e-14, atol=0)


# ---------------------------------------------------------------------------
# Affine chunk summaries (Tokamax design doc, context-parallel section)
# ---------------------------------------------------------------------------

def pin_affine_summaries_replay(oracle):
    """Each chunk maps its start state affinely (S' = Phi S + Psi): composing the chunk
    summaries in order and applying them to S_0 reaches the token recurrence's final
    state, and the merged segment start states are the recurrence's states at the
    segment boundaries (prefixes of the sequence)."""
    from oracle import compose_summaries, segment_start_states
    rng = np.random.default_rng(21)
    B, T, H, K, V, C = 2, 157, 2, 16, 12, 16
    q, k, v, g, beta = _rand_inputs(rng, B, T, H, K, V, g_max=0.8)
    s0 = rng.standard_normal((B, H, K, V))
    scale = 0.3
    phi, psi = oracle.chunk_summaries(q, k, v, g, beta, scale, chunk_size=C)
    nct = -(-T // C)
    assert phi.shape == (B, H, nct, K, K) and psi.shape == (B, H, nct, K, V)
    Pall, Qall = compose_summaries(phi, psi, 0, nct)
    _, fin = oracle.recurrent(q, k, v, g, beta, scale, initial_state=s0)
    assert np.allclose(Pall @ s0 + Qall, fin, rtol=0, atol=1e-10), "summaries do not replay the recurrence"
    seg = 3
    starts, last = segment_start_states(phi, psi, s0, seg)
    assert np.allclose(last, fin, rtol=0, atol=1e-10)
    for si in range(1, starts.shape[-3]):
        t_end = si * seg * C
        _, fin_p = oracle.recurrent(q[:, :t_end], k[:, :t_end], v[:, :t_end], g[:, :t_end],
                                    beta[:, :t_end], scale, initial_state=s0)
        assert np.allclose(starts[..., si, :, :], fin_p, rtol=0, atol=1e-10), f"segment {si} start"


def pin_affine_beta_zero(oracle):
    """With beta = 0 no chunk writes: Phi_j = Diag(exp(sum of g over chunk j)) and
    Psi_j = 0 (Eq. (1) with beta_t = 0)."""
    rng = np.random.default_rng(22)
    B, T, H, K, V, C = 1, 50, 2, 8, 6, 16
    q, k, v, g, _ = _rand_inputs(rng, B, T, H, K, V, g_max=0.5)
    beta = np.zeros((B, T, H))
    phi, psi = oracle.chunk_summaries(q, k, v, g, beta, 0.5, chunk_size=C)
    for j in range(-(-T // C)):
        gam = np.exp(g[:, j * C:(j + 1) * C].sum(axis=1))       # [B,H,K]
        ref = np.zeros((B, H, K, K))
        for d in range(K):
            ref[..., d, d] = gam[..., d]
        assert np.allclose(phi[:, :, j], ref, rtol=1e-13, atol=1e-15), f"Phi of chunk {j}"
        assert np.array_equal(psi[:, :, j], np.zeros((B, H, K, V))), f"Psi of chunk {j}"


ALL_PINS = [
    pin_eq1_exact_rational,
    pin_linear_attention,
    pin_delta_rule_retrieval,
    pin_beta_zero_freeze,
    pin_recurrent_equals_chunkwise,
    pin_state_norm_bound,
    pin_causality,
    pin_split_resume,
    pin_varlen_isolation,
    pin_gate_softplus,
    pin_gate_sigmoid,
    pin_l2norm,
    pin_affine_summaries_replay,
    pin_affine_beta_zero,
]
