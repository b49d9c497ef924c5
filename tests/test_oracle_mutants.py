"""Planted-mistake check of the oracle pins (CPU only).

Each mutant is a copy of ``oracle/kda_oracle.c`` with one plausible mistake (a wrong
sign, a dropped term, a wrong index or operand, a moved step).  The test compiles the
copy and requires that at least one pin of ``tests/pins.py`` fails on it, which shows
that the pins would catch that mistake in the real oracle.
"""
import os

import pytest

import oracle
from tests import pins

_WRITE = ("        for (int d = 0; d < K; ++d) {\n"
          "            const double bk = bt * kt[d];\n"
          "            for (int j = 0; j < V; ++j) S[(size_t)d * V + j] += bk * e[j];\n"
          "        }\n")
_READ = ("        for (int j = 0; j < V; ++j) {\n"
         "            double acc = 0.0;\n"
         "            for (int d = 0; d < K; ++d) acc += S[(size_t)d * V + j] * qt[d];\n"
         "            ot[j] = J->scale * acc;\n"
         "        }\n")
_DECAY = ("        for (int d = 0; d < K; ++d) {\n"
          "            const double alpha = exp(gt[d]);\n"
          "            for (int j = 0; j < V; ++j) S[(size_t)d * V + j] *= alpha;\n"
          "        }\n")

MUTANTS = {
    # token recurrence
    "gate_sign": [("exp(gt[d])", "exp(-gt[d])")],
    "delta_sign": [("e[j] = vt[j] - pred;", "e[j] = vt[j] + pred;")],
    "predict_with_query": [("pred += S[(size_t)d * V + j] * kt[d];",
                            "pred += S[(size_t)d * V + j] * qt[d];")],
    "write_without_beta": [("const double bk = bt * kt[d];", "const double bk = kt[d];")],
    "output_without_scale": [("ot[j] = J->scale * acc;", "ot[j] = acc;")],
    "read_with_key": [("acc += S[(size_t)d * V + j] * qt[d];",
                       "acc += S[(size_t)d * V + j] * kt[d];")],
    "read_before_write": [(_READ, ""), (_WRITE, _READ + _WRITE)],
    "decay_after_write": [(_DECAY, ""), (_WRITE, _WRITE + _DECAY)],
    "previous_token_gate": [("const double* gt = J->g + ((size_t)t * H + h) * K;",
                             "const double* gt = J->g + ((size_t)(t > t0 ? t - 1 : t) * H + h) * K;")],
    "ignore_initial_state": [("    if (J->initial_state)\n", "    if (0)\n")],
    "no_sequence_reset": [("*begin = J->cu_seqlens[n];", "*begin = J->cu_seqlens[0];")],
    "beta_of_head0": [("const double bt = J->beta[(size_t)t * H + h];",
                       "const double bt = J->beta[(size_t)t * H];")],
    # chunkwise form
    "L_without_beta": [("(j < i) ? BETA(i) * lij : 0.0", "(j < i) ? lij : 0.0")],
    "L_beta_of_column": [("(j < i) ? BETA(i) * lij : 0.0", "(j < i) ? BETA(j) * lij : 0.0")],
    "Aqk_strict": [("(j <= i) ? J->scale * aij : 0.0", "(j < i) ? J->scale * aij : 0.0")],
    "exclusive_cumsum": [("            acc += GATE(r, d);\n            G_(r, d) = acc * inv_ln2;\n",
                          "            G_(r, d) = acc * inv_ln2;\n            acc += GATE(r, d);\n")],
    "decay_ratio_sign": [("const double rho = exp2(G_(i, d) - G_(j, d));",
                          "const double rho = exp2(G_(j, d) - G_(i, d));")],
    "solve_sign": [("x -= s->L[(size_t)r * c + j]", "x += s->L[(size_t)r * c + j]")],
    "W_without_gate": [("BETA(j) * exp2(G_(j, d)) * K_(j, d)", "BETA(j) * K_(j, d)")],
    "U_without_beta": [("acc += s->A[(size_t)r * c + j] * BETA(j) * V_(j, jv);",
                        "acc += s->A[(size_t)r * c + j] * V_(j, jv);")],
    "Kbar_from_chunk_start": [("K_(r, d) * exp2(G_(c - 1, d) - G_(r, d))",
                               "K_(r, d) * exp2(-G_(r, d))")],
    # affine chunk summaries
    "phi_plus": [("d == e ? exp2(s.G[(size_t)(c - 1) * K + d]) : 0.0) - acc;",
                  "d == e ? exp2(s.G[(size_t)(c - 1) * K + d]) : 0.0) + acc;")],
    "phi_transposed": [("acc += s.Kbar[(size_t)r * K + d] * s.W[(size_t)r * K + e];",
                        "acc += s.Kbar[(size_t)r * K + e] * s.W[(size_t)r * K + d];")],
    "phi_gamma_first_row": [("(d == e ? exp2(s.G[(size_t)(c - 1) * K + d]) : 0.0)",
                             "(d == e ? exp2(s.G[d]) : 0.0)")],
    "psi_without_kbar": [("acc += s.Kbar[(size_t)r * K + d] * s.U[(size_t)r * V + jv];",
                          "acc += s.U[(size_t)r * V + jv];")],
    "Vnew_sign": [("s->U[(size_t)r * V + jv] - acc;", "s->U[(size_t)r * V + jv] + acc;")],
    "O_without_inter": [("orow[jv] = inter + intra;", "orow[jv] = intra;")],
    "inter_without_gate": [("J->scale * Q_(r, d) * exp2(G_(r, d)) * S[(size_t)d * V + jv]",
                            "J->scale * Q_(r, d) * S[(size_t)d * V + jv]")],
    "state_without_decay": [("= gammaC * S[(size_t)d * V + jv] + acc;",
                             "= S[(size_t)d * V + jv] + acc;")],
    # raw-gate activation and row normalisation
    "softplus_sign": [("log1p(exp(-a))", "log1p(exp(a))")],
    "softplus_no_linear_part": [("return (y > 0.0 ? y : 0.0) + log1p", "return log1p")],
    "sigmoid_sign": [("1.0 / (1.0 + exp(-y))", "1.0 / (1.0 + exp(y))")],
    "gate_without_lambda": [("-lam * softplus(xb)", "-softplus(xb)")],
    "sigmoid_without_lambda": [("lower_bound * sigmoid(lam * xb)", "lower_bound * sigmoid(xb)")],
    "gate_without_bias": [("if (dt_bias) xb += dt_bias[(size_t)h * K + d];", "")],
    "l2norm_without_eps": [("if (n < eps) n = eps;", "")],
    "l2norm_without_sqrt": [("double n = sqrt(ss);", "double n = ss;")],
}


@pytest.fixture(scope="module")
def source_text():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source_text, tmp_path):
    text = source_text
    for old, new in MUTANTS[name]:
        assert text.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
        text = text.replace(old, new)
    src = tmp_path / "kda_oracle.c"
    src.write_text(text)
    # the header travels with the copy
    with open(os.path.join(oracle.HERE, "kda_oracle.h")) as f:
        (tmp_path / "kda_oracle.h").write_text(f.read())
    lib = oracle.build_oracle(str(src), str(tmp_path / "libmutant.so"), force=True)
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError) as exc:
            caught.append(f"{pin.__name__}: {exc}")
            break
    assert caught, f"no pin catches mutant {name}"
