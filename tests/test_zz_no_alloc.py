"""kda_fwd_noalloc: the forward pass for callers that cannot allocate device memory.

It runs kda_fwd's kernels with the library's own fixed scratch array as workspace.
Checked through the C ABI against kda_fwd (which gets a workspace from the caller) on
two calls in a row with different shapes, so that the second call also shows that the
contents the first call left in the shared array do not leak into its results."""
import ctypes

import numpy as np
import pytest
import torch

from workloads import custom, make_inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
SCRATCH_BYTES = 64 * 1024 * 1024


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(lib, inp, o, fin):
    cu = inp["cu_seqlens"]
    st = lib.kda_fwd_noalloc(
        _p(inp["q"]), _p(inp["k"]), _p(inp["v"]), _p(inp["g"]), _p(inp["beta"]),
        float(inp["scale"]), 64, _p(inp["initial_state"]), _p(cu),
        (cu.numel() - 1) if cu is not None else 0, _p(o), _p(fin), inp["B"], inp["T"],
        inp["H"], inp["K"], inp["V"], 0 if inp["dtype"] == torch.bfloat16 else 1,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_matches_kda_fwd_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kimi_delta_attention_11_gb300 as kda
    lib = kda.load_library()
    lens = [70, 0, 129, 64, 1]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    cases = []
    a = make_inputs(custom(B=2, T=300, H=3, K=128, V=128, dtype=torch.bfloat16, init_std=0.1,
                           seed=71), device="cuda")
    cases.append(a)
    b = make_inputs(custom(B=1, T=int(cu[-1]), H=2, K=64, V=64, dtype=torch.float32, seed=72),
                    device="cuda")
    b["cu_seqlens"] = cu.cuda()
    b["N"] = len(lens)
    b["initial_state"] = 0.2 * torch.randn((len(lens), 2, 64, 64), device="cuda")
    cases.append(b)
    for inp in cases:
        need = kda.workspace_bytes(inp["B"], inp["T"], inp["H"], inp["K"], inp["V"],
                                   len(lens) if inp["cu_seqlens"] is not None else 0,
                                   inp["dtype"])
        assert need <= SCRATCH_BYTES
        ref_o, ref_f = kda.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                               inp["scale"], initial_state=inp["initial_state"],
                               cu_seqlens=inp["cu_seqlens"])
        o = torch.full_like(ref_o, float("nan"))
        fin = torch.full_like(ref_f, float("nan"))
        assert _call_noalloc(lib, inp, o, fin) == 0
        torch.cuda.synchronize()
        tol = TOL[inp["dtype"]]
        assert (o.float() - ref_o.float()).abs().max().item() <= tol
        assert (fin - ref_f).abs().max().item() <= tol


def test_noalloc_rejects_problems_larger_than_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kimi_delta_attention_11_gb300 as kda
    lib = kda.load_library()
    inp = make_inputs(custom(B=1, T=16384, H=8, K=128, V=128, dtype=torch.bfloat16, seed=73),
                      device="cuda")
    assert kda.workspace_bytes(1, 16384, 8, 128, 128, 0, torch.bfloat16) > SCRATCH_BYTES
    o = torch.zeros((1, 16384, 8, 128), dtype=torch.bfloat16, device="cuda")
    fin = torch.zeros((1, 8, 128, 128), device="cuda")
    assert _call_noalloc(lib, inp, o, fin) == 4   # KDA_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert o.abs().max().item() == 0 and fin.abs().max().item() == 0
