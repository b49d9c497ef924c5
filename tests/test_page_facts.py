"""The pages' printed scalar facts against closed forms (tests/golden/page_facts.json).

These pin the design constants of the CUDA path: the 16-key rebasing window that keeps
rescaled bf16 operands finite at the -5 gate bound, and the tolerance reasoning."""
import json
import math
import os

import numpy as np
import torch

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def test_strongest_decay():
    f = GOLD["strongest_decay"]
    assert round(math.exp(-5.0), f["digits"]) == f["value"]


def test_overflow_window():
    f = GOLD["overflow_after_18_steps_log2"]
    grow = lambda steps: 5.0 * steps * math.log2(math.e)   # log2 of e^{5 steps}
    assert round(grow(18), f["digits"]) == f["value"]
    assert grow(18) > 128.0                                 # beyond the fp32/bf16 range
    w = GOLD["key_window"]["value"]
    assert grow(w - 1) < 128.0 <= grow(w + 8 - 1)           # 16 keys fit, 24 do not
    assert w % 8 == 0


def test_reference_choice_bound():
    u = 2.0 ** -8
    assert 4 * u == GOLD["reference_choice_bound"]["value"]


def test_underflow_loss_bound():
    f = GOLD["underflow_loss_bound"]
    bound = math.sqrt(f["D"]) * 2.0 ** f["tau_log2"] * math.exp(f["boost_ln"])
    assert abs(bound - f["value"]) / f["value"] < 0.01


def test_diagonal_block_counts():
    f = GOLD["diagonal_block_kept"]
    for key, w in (("w16", 16), ("w32", 32)):
        assert [w * (w + 1) // 2, w * w] == f[key]


def test_tcgen05_ratio():
    f = GOLD["tcgen05_shape_speedup"]
    assert round(f["n32_tflops"] / f["n16_tflops"], 2) == f["ratio"]


def test_alignment_padding_bound():
    C = 64
    rng = np.random.default_rng(0)
    for _ in range(100):
        L = rng.integers(0, 500, size=rng.integers(1, 20))
        pad = int(np.sum(C * np.ceil(L / C) - L))
        assert 0 <= pad <= len(L) * (C - 1)
    L = np.full(7, 65)
    assert int(np.sum(C * np.ceil(L / C) - L)) == 7 * (C - 1)


def test_reference_choice_bound_in_bf16_simulation():
    """First-row vs midpoint rebasing of one Aqk entry, with bf16-rounded operands and
    exact accumulation, differ by at most 4u for unit q, k ("Why is it hard to extract
    the future signal?")."""
    gen = torch.Generator().manual_seed(3)
    D = 128
    worst = 0.0
    for _ in range(200):
        q = torch.randn(D, generator=gen, dtype=torch.float64)
        k = torch.randn(D, generator=gen, dtype=torch.float64)
        q, k = q / q.norm(), k / k.norm()
        # cumulative log2 gates of a 16-token window at the -5 bound region
        gl = -5.0 * torch.rand(16, D, generator=gen, dtype=torch.float64) / math.log(2.0)
        G = torch.cumsum(gl, 0)
        i, j = 5, 2

        def entry(r):
            a = (q * torch.exp2(G[i] - r)).to(torch.bfloat16).double()
            b = (k * torch.exp2(r - G[j])).to(torch.bfloat16).double()
            return float((a * b).sum())

        worst = max(worst, abs(entry(G[0]) - entry(G[8])))
    assert worst <= GOLD["reference_choice_bound"]["value"]
