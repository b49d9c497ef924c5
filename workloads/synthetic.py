"""Seeded synthetic inputs for the KDA forward workloads.

This module only draws random tensors; it holds none of the method's arithmetic.
Both the CUDA-library tests/benchmark and the oracle tests take their inputs from here.

Recipe (shared by all workloads unless a workload overrides it):
  * q, k, v ~ N(0, 1) drawn in fp32; q and k L2-normalised along the key dimension as
    ``x / max(||x||_2, 1e-6)`` in fp32, then cast to the workload dtype (bf16 or fp32);
  * beta = sigmoid(N(mu_beta, 1)) per (token, head), fp32;
  * g = -g_max * sigmoid(N(0, 1)) per (token, head, key channel), fp32 natural-log decay;
  * scale = K ** -0.5;
  * initial_state ~ N(0, init_std^2) fp32 when the workload has one, else absent.
Random numbers come from a CPU ``torch.Generator`` seeded per workload, so the same
seed gives the same tensors on every host.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    dtype: torch.dtype
    chunk_size: int = 64
    g_max: float = 5.0          # g = -g_max * sigmoid(N(0,1))
    beta_mean: float = 0.0      # beta = sigmoid(N(beta_mean, 1))
    init_std: Optional[float] = None  # None: zero initial state (argument omitted)
    varlen: Optional[Tuple[int, int, int]] = None  # (num_seqs, min_len, max_len)
    seed: int = 0

    @property
    def dtype_name(self) -> str:
        return {torch.bfloat16: "bf16", torch.float32: "f32"}[self.dtype]


# The five workloads of the KDA forward measurement plan (sizes and distributions), and
# one for the scan schedule.
WORKLOADS: Dict[str, Workload] = {
    "tiny_f32": Workload("tiny_f32", B=1, T=256, H=2, K=64, V=64, dtype=torch.float32,
                         seed=1001),
    "dense_bf16": Workload("dense_bf16", B=2, T=4096, H=16, K=128, V=128,
                           dtype=torch.bfloat16, seed=1002),
    "varlen_bf16": Workload("varlen_bf16", B=1, T=0, H=32, K=128, V=128,
                            dtype=torch.bfloat16, init_std=0.1, varlen=(8, 300, 9000),
                            seed=1003),
    "long_bf16": Workload("long_bf16", B=1, T=131072, H=32, K=128, V=128,
                          dtype=torch.bfloat16, g_max=0.5, init_std=0.1, seed=1004),
    "serving_bf16": Workload("serving_bf16", B=32, T=2048, H=32, K=128, V=128,
                             dtype=torch.bfloat16, beta_mean=2.0, seed=1005),
    # Few, very long chains (the case the chunk-parallel state scan serves): 2 heads of
    # one 262144-token sequence.
    "few_long_bf16": Workload("few_long_bf16", B=1, T=262144, H=2, K=128, V=128,
                              dtype=torch.bfloat16, g_max=0.5, init_std=0.1, seed=1007),
}


# Decode-step workload: one token for each of N sequences against an existing state (the
# serving batch of the measurement plan, 32 sequences x 32 heads).
DECODE_WORKLOADS: Dict[str, dict] = {
    "decode_bf16": dict(N=32, H=32, K=128, V=128, dtype=torch.bfloat16, init_std=0.1, seed=1006),
}


def make_decode_inputs(N: int, H: int, K: int, V: int, dtype: torch.dtype, init_std: float,
                       seed: int, device: str = "cpu") -> Dict[str, object]:
    """q, k [N,H,K] (unit rows), v [N,H,V], g [N,H,K] = -5 sigmoid(N(0,1)), beta [N,H] =
    sigmoid(N(0,1)), state [N,H,K,V] ~ N(0, init_std^2), by the shared recipe."""
    gen = torch.Generator().manual_seed(seed)

    def unit_rows(shape):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-6)

    out = dict(q=unit_rows((N, H, K)).to(dtype), k=unit_rows((N, H, K)).to(dtype),
               v=torch.randn((N, H, V), generator=gen).to(dtype),
               g=(-5.0 * torch.sigmoid(torch.randn((N, H, K), generator=gen))).contiguous(),
               beta=torch.sigmoid(torch.randn((N, H), generator=gen)).contiguous(),
               state=(init_std * torch.randn((N, H, K, V), generator=gen)).contiguous(),
               scale=K ** -0.5, N=N, H=H, K=K, V=V, dtype=dtype)
    if device != "cpu":
        for key in ("q", "k", "v", "g", "beta", "state"):
            out[key] = out[key].to(device)
    return out


def custom(name: str = "custom", **kw) -> Workload:
    """A workload with the shared recipe and explicit sizes (for small test cases)."""
    base = dict(B=1, T=128, H=1, K=64, V=64, dtype=torch.float32, seed=7)
    base.update(kw)
    return Workload(name=name, **base)


def varlen_lengths(w: Workload) -> torch.Tensor:
    """Sequence lengths of a packed workload, uniform in [min_len, max_len]."""
    n, lo, hi = w.varlen
    gen = torch.Generator().manual_seed(w.seed + 7919)
    return torch.randint(lo, hi + 1, (n,), generator=gen, dtype=torch.int64)


def make_inputs(w: Workload, device: str = "cpu") -> Dict[str, object]:
    """Draw one seeded input set. Returns a dict with q, k, v, g, beta, scale,
    initial_state (or None), cu_seqlens (int32 or None) and the shape numbers."""
    gen = torch.Generator().manual_seed(w.seed)
    if w.varlen is not None:
        lens = varlen_lengths(w)
        cu = torch.zeros(lens.numel() + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
        B, T, N = 1, int(cu[-1]), lens.numel()
    else:
        cu = None
        B, T, N = w.B, w.T, w.B
    H, K, V = w.H, w.K, w.V

    def unit_rows(shape):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-6)

    q = unit_rows((B, T, H, K)).to(w.dtype)
    k = unit_rows((B, T, H, K)).to(w.dtype)
    v = torch.randn((B, T, H, V), generator=gen, dtype=torch.float32).to(w.dtype)
    beta = torch.sigmoid(torch.randn((B, T, H), generator=gen) + w.beta_mean)
    g = -w.g_max * torch.sigmoid(torch.randn((B, T, H, K), generator=gen))
    s0 = None
    if w.init_std is not None:
        s0 = w.init_std * torch.randn((N, H, K, V), generator=gen, dtype=torch.float32)

    out = dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta.contiguous(), scale=K ** -0.5,
               initial_state=s0, cu_seqlens=cu, B=B, T=T, H=H, K=K, V=V, N=N,
               chunk_size=w.chunk_size, dtype=w.dtype)
    if device != "cpu":
        for key in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens"):
            if out[key] is not None:
                out[key] = out[key].to(device)
    return out


def token_heads(inp: Dict[str, object]) -> int:
    """Number of (token, head) pairs of an input set."""
    return int(inp["B"]) * int(inp["T"]) * int(inp["H"])
