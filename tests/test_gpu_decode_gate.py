"""GPU parity of the decode step and of the in-kernel gate activation / q-k
normalisation against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from workloads import custom, make_inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kimi_delta_attention_11_gb300 as k
    k.load_library()
    return k


@pytest.fixture(scope="module")
def orc():
    return oracle.default_oracle()


def _decode_inputs(N, H, K, V, dtype, seed, raw=False):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((N, H, K), generator=g)
    k = torch.randn((N, H, K), generator=g)
    if not raw:  # unit rows, as the pre-normalised path expects
        q = q / q.norm(dim=-1, keepdim=True)
        k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn((N, H, V), generator=g)
    gate = torch.randn((N, H, K), generator=g) if raw else -5.0 * torch.sigmoid(
        torch.randn((N, H, K), generator=g))
    beta = torch.sigmoid(torch.randn((N, H), generator=g))
    state = 0.3 * torch.randn((N, H, K, V), generator=g)
    return (q.to(dtype), k.to(dtype), v.to(dtype), gate.float().contiguous(),
            beta.float().contiguous(), state.float().contiguous())


def _oracle_step(orc, q, k, v, g, beta, state, scale):
    """One token per sequence through the fp64 token recurrence: B = N, T = 1."""
    return orc.recurrent(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None], scale,
                         initial_state=state)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("KV", [(64, 64), (128, 128), (64, 128), (128, 64)],
                         ids=lambda kv: f"K{kv[0]}V{kv[1]}")
def test_decode_step(kda, orc, dtype, KV):
    K, V = KV
    q, k, v, g, beta, s0 = _decode_inputs(6, 3, K, V, dtype, seed=K * 7 + V)
    state = s0.cuda()
    o = kda.decode(q.cuda(), k.cuda(), v.cuda(), g.cuda(), beta.cuda(), state)
    torch.cuda.synchronize()
    o_ref, s_ref = _oracle_step(orc, q, k, v, g, beta, s0, K ** -0.5)
    eo = np.abs(o.float().cpu().numpy() - o_ref[:, 0]).max()
    es = np.abs(state.cpu().numpy() - s_ref).max()
    assert eo <= TOL[dtype] and es <= TOL[dtype], (eo, es)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_decode_steps_continue_prefill(kda, dtype):
    """A prefill of 100 tokens followed by 37 decode steps equals one prefill of 137."""
    K = V = 128 if dtype == torch.bfloat16 else 64
    inp = make_inputs(custom(B=2, T=137, H=2, K=K, V=V, dtype=dtype, init_std=0.2, seed=91),
                      device="cuda")
    o_all, f_all = kda.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                           initial_state=inp["initial_state"])
    sl = lambda x, a, b: x[:, a:b].contiguous()
    o1, f1 = kda.fwd(sl(inp["q"], 0, 100), sl(inp["k"], 0, 100), sl(inp["v"], 0, 100),
                     sl(inp["g"], 0, 100), sl(inp["beta"], 0, 100), inp["scale"],
                     initial_state=inp["initial_state"])
    state = f1.clone()
    outs = []
    for t in range(100, 137):
        outs.append(kda.decode(inp["q"][:, t].contiguous(), inp["k"][:, t].contiguous(),
                               inp["v"][:, t].contiguous(), inp["g"][:, t].contiguous(),
                               inp["beta"][:, t].contiguous(), state, inp["scale"]))
    torch.cuda.synchronize()
    o_dec = torch.stack(outs, 1)
    tol = TOL[dtype]
    assert (o_dec.float() - o_all[:, 100:].float()).abs().max().item() <= tol
    assert (torch.cat([o1, o_dec], 1).float() - o_all.float()).abs().max().item() <= tol
    assert (state - f_all).abs().max().item() <= tol


GATES = {
    "softplus": dict(lower_bound=0.0),
    "sigmoid": dict(lower_bound=-4.0),
}


def _gate_dict(H, K, form, seed, qk_norm):
    g = torch.Generator().manual_seed(seed)
    # exp(a_log) = 0.5 keeps -ln(alpha) = 0.5 softplus(x) under the -5 bound for |x| < 9
    a_log = (torch.full((H,), np.log(0.5)) + 0.1 * torch.randn((H,), generator=g)).float()
    dt_bias = 0.3 * torch.randn((H * K,), generator=g).float()
    return dict(a_log=a_log, dt_bias=dt_bias, qk_l2norm=qk_norm, **GATES[form])


def _activated(orc, gd, graw, q, k):
    ell = orc.gate(graw, gd["a_log"], gd["dt_bias"], gd["lower_bound"])
    if gd["qk_l2norm"]:
        q, k = orc.l2norm(q), orc.l2norm(k)
    return ell, q, k


@pytest.mark.parametrize("form", list(GATES))
@pytest.mark.parametrize("path", ["tc_bf16", "tc_bf16_many_chains", "tc_bf16_two", "tc_bf16_scan",
                                  "simt_f32"])
def test_gate_activation_fwd(kda, orc, form, path, monkeypatch):
    """In-kernel gate activation and q/k normalisation on every path and schedule:
    fused (tc_bf16), per-chain two kernels (many chains), value-sliced two kernels (forced),
    scan (forced), and the exact CUDA-core path."""
    dtype, K = (torch.float32, 64) if path == "simt_f32" else (torch.bfloat16, 128)
    B, T, H = (2, 150, 3) if path != "tc_bf16_many_chains" else (6, 90, 14)
    if path == "tc_bf16_two":
        monkeypatch.setenv("KDA_SCHEDULE", "two")
    if path == "tc_bf16_scan":
        B, T, H = 1, 64 * 9 + 11, 2
        monkeypatch.setenv("KDA_SCHEDULE", "scan")
        assert kda.schedule(B, T, H, K, K) == "scan"
    g = torch.Generator().manual_seed(5 + len(form) + K)
    q = torch.randn((B, T, H, K), generator=g).to(dtype)   # not normalised: the kernel does it
    k = torch.randn((B, T, H, K), generator=g).to(dtype)
    v = torch.randn((B, T, H, K), generator=g).to(dtype)
    graw = torch.randn((B, T, H, K), generator=g).float()
    beta = torch.sigmoid(torch.randn((B, T, H), generator=g)).float()
    s0 = 0.1 * torch.randn((B, H, K, K), generator=g).float()
    gd = _gate_dict(H, K, form, seed=3, qk_norm=True)
    gdev = {k_: (v_.cuda() if torch.is_tensor(v_) else v_) for k_, v_ in gd.items()}
    o, fin = kda.fwd(q.cuda(), k.cuda(), v.cuda(), graw.cuda(), beta.cuda(), K ** -0.5,
                     initial_state=s0.cuda(), gate=gdev)
    torch.cuda.synchronize()
    ell, qn, kn = _activated(orc, gd, graw, q, k)
    assert ell.min() >= -5.0   # the activated gate respects the kernel's precondition
    o_ref, f_ref = orc.recurrent(qn, kn, v, ell, beta, K ** -0.5, initial_state=s0)
    eo = np.abs(o.float().cpu().numpy() - o_ref).max()
    es = np.abs(fin.cpu().numpy() - f_ref).max()
    assert eo <= TOL[dtype] and es <= TOL[dtype], (eo, es)


@pytest.mark.parametrize("form", list(GATES))
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_gate_activation_decode(kda, orc, form, dtype):
    N, H, K, V = 4, 2, 128, 128
    q, k, v, graw, beta, s0 = _decode_inputs(N, H, K, V, dtype, seed=77, raw=True)
    gd = _gate_dict(H, K, form, seed=4, qk_norm=True)
    gdev = {k_: (v_.cuda() if torch.is_tensor(v_) else v_) for k_, v_ in gd.items()}
    state = s0.cuda()
    o = kda.decode(q.cuda(), k.cuda(), v.cuda(), graw.cuda(), beta.cuda(), state, gate=gdev)
    torch.cuda.synchronize()
    ell, qn, kn = _activated(orc, gd, graw, q, k)
    o_ref, s_ref = _oracle_step(orc, qn, kn, v, ell, beta, s0, K ** -0.5)
    eo = np.abs(o.float().cpu().numpy() - o_ref[:, 0]).max()
    es = np.abs(state.cpu().numpy() - s_ref).max()
    assert eo <= TOL[dtype] and es <= TOL[dtype], (eo, es)


def test_gate_option_validation(kda):
    inp = make_inputs(custom(B=1, T=64, H=2, K=128, V=128, dtype=torch.bfloat16, seed=3),
                      device="cuda")
    a_log = torch.zeros(2, device="cuda")
    with pytest.raises(kda.KdaError):     # lower bound outside [-5, 0)
        kda.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                gate=dict(a_log=a_log, lower_bound=-6.0))
    with pytest.raises(ValueError):       # a_log of the wrong size
        kda.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                gate=dict(a_log=torch.zeros(3, device="cuda")))
