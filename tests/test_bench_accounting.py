"""The benchmark's algorithmic work counts against the measurement plan's printed figures
(per chunk of 64 tokens with K = V = 128: 9,024,832 flops, i.e. 141,013 per token-head;
46,613 per token-head for K = V = 64; 1540 bytes per bf16 token-head plus the states),
and the counting rules for short chunks and packed sequences."""
import torch

import bench
from workloads import WORKLOADS, custom, make_inputs


def test_flops_per_chunk_plan_figures():
    assert bench.flops_per_chunk(64, 128, 128) == 9_024_832
    assert bench.flops_per_chunk(64, 128, 128) == 141_013 * 64
    assert bench.flops_per_chunk(64, 64, 64) == 46_613 * 64


def test_flops_small_chunks_by_counting():
    # count the multiply-adds of each product of one chunk of c tokens element by element
    # (2 flops each); the solve's forward substitution takes one multiply-add per
    # (i, j, m) with j <= m < i, (c-1)c(c+1)/6 of them
    for c in (1, 2, 3, 5, 16):
        for K, V in ((2, 3), (4, 4)):
            aqk = sum(K for i in range(c) for j in range(i + 1))          # j <= i
            ell = sum(K for i in range(c) for j in range(i))              # j < i
            w = sum(K for i in range(c) for j in range(i + 1))            # lower incl. diagonal
            u = sum(V for i in range(c) for j in range(i + 1))
            state = 3 * c * K * V                                         # W S, Qg S, K_bar^T V_new
            av = sum(V for i in range(c) for j in range(i + 1))           # Aqk V_new
            solve = sum(1 for i in range(c) for j in range(i) for m in range(j, i))
            assert 2 * (aqk + ell + w + u + state + av + solve) == bench.flops_per_chunk(c, K, V), (c, K, V)


def test_dense_bytes_and_flops():
    inp = make_inputs(WORKLOADS["dense_bf16"])
    a = bench.algorithmic(inp)
    th = 2 * 4096 * 16
    assert a["token_heads"] == th
    assert a["in_bytes"] + a["out_bytes"] == 1540 * th
    assert a["state_out"] == 2 * 16 * 128 * 128 * 4 and a["state_in"] == 0
    assert a["bytes"] == 203_948_032
    assert a["flops"] == 2 * 16 * 64 * 9_024_832


def test_short_chunks_and_packed_sequences():
    inp = make_inputs(custom(B=1, T=64 * 3 + 5, H=2, K=64, V=64, dtype=torch.float32, seed=5))
    a = bench.algorithmic(inp)
    assert a["flops"] == 2 * (3 * bench.flops_per_chunk(64, 64, 64) + bench.flops_per_chunk(5, 64, 64))
    assert a["in_bytes"] + a["out_bytes"] == 1284 * (64 * 3 + 5) * 2      # fp32: 4(2K+V)+4K+4+4V
    cu = torch.tensor([0, 70, 70, 200], dtype=torch.int32)
    inp["cu_seqlens"], inp["N"], inp["T"] = cu, 3, 200
    inp["B"] = 1
    a = bench.algorithmic(inp)
    per = lambda L: (L // 64) * bench.flops_per_chunk(64, 64, 64) + (bench.flops_per_chunk(L % 64, 64, 64) if L % 64 else 0)
    assert a["flops"] == 2 * (per(70) + per(0) + per(130))
    assert a["state_out"] == 3 * 2 * 64 * 64 * 4


def test_decode_reference_rate_runs_the_oracle():
    spec = dict(N=2, H=2, K=64, V=64, dtype=torch.float32, init_std=0.1, seed=3)
    rate, threads, desc, dt = bench.oracle_decode_rate(spec, 0.0)
    assert rate > 0 and dt > 0 and threads >= 1
    assert "2 sequences x 2 heads" in desc
