"""GPU parity of the CUDA library (through the C ABI) against the fp64 oracle.

Tolerances (max absolute error on o and on final_state): 1e-4 for fp32 inputs and
2e-2 for bf16 inputs.  Small cases compare every element; the full-size workloads
compare every output of a sample of (sequence, head) chains, which the oracle
evaluates one by one.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, custom, make_inputs

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


def run_gpu(kda, inp, **kw):
    o, fin = kda.fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                     initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    return o, fin


def run_oracle(orc, inp):
    return orc.recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["scale"],
                         initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"])


def errors(o, fin, o_ref, f_ref):
    eo = float(np.max(np.abs(o.float().cpu().numpy() - o_ref))) if o.numel() else 0.0
    ef = float(np.max(np.abs(fin.cpu().numpy() - f_ref))) if fin.numel() else 0.0
    return eo, ef


def check(kda, orc, inp, tol=None):
    tol = tol or TOL[inp["dtype"]]
    o, fin = run_gpu(kda, inp)
    o_ref, f_ref = run_oracle(orc, inp)
    eo, ef = errors(o, fin, o_ref, f_ref)
    assert np.isfinite(o.float().cpu().numpy()).all()
    assert eo <= tol, f"max|o - oracle| = {eo:.3e} > {tol}"
    assert ef <= tol, f"max|S - oracle| = {ef:.3e} > {tol}"
    return eo, ef


def test_tiny_f32_workload(kda, orc):
    check(kda, orc, make_inputs(WORKLOADS["tiny_f32"], device="cuda"))


SHAPES = [(1, 1, 1), (1, 63, 2), (2, 64, 1), (1, 65, 2), (2, 200, 3), (1, 257, 1)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("KV", [(64, 64), (128, 128), (64, 128), (128, 64)],
                         ids=lambda kv: f"K{kv[0]}V{kv[1]}")
@pytest.mark.parametrize("BTH", SHAPES, ids=lambda s: "B{}T{}H{}".format(*s))
@pytest.mark.parametrize("init", [None, 0.3], ids=["zero_state", "init_state"])
def test_small_shapes(kda, orc, dtype, KV, BTH, init):
    B, T, H = BTH
    K, V = KV
    w = custom(B=B, T=T, H=H, K=K, V=V, dtype=dtype, init_std=init, seed=B * 1000 + T + H)
    check(kda, orc, make_inputs(w, device="cuda"))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_varlen_edges(kda, orc, dtype):
    """Packed sequences of length 0, 1, 63, 64, 65, 129 with per-sequence initial states."""
    lens = [1, 63, 0, 64, 65, 129, 2, 0]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    inp = make_inputs(custom(B=1, T=int(cu[-1]), H=2, K=128, V=128, dtype=dtype, seed=32))
    inp["cu_seqlens"] = cu
    inp["N"] = len(lens)
    inp["initial_state"] = 0.2 * torch.randn((len(lens), 2, 128, 128),
                                             generator=torch.Generator().manual_seed(3))
    for key in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens"):
        inp[key] = inp[key].cuda()
    check(kda, orc, inp)


def test_empty_input_returns_initial_state(kda):
    dev = "cuda"
    H, K, V = 2, 64, 64
    z = lambda *s, dt=torch.float32: torch.zeros(s, dtype=dt, device=dev)
    s0 = torch.randn((3, H, K, V), device=dev)
    cu = torch.zeros(4, dtype=torch.int32, device=dev)
    o, fin = kda.fwd(z(1, 0, H, K), z(1, 0, H, K), z(1, 0, H, V), z(1, 0, H, K), z(1, 0, H),
                     initial_state=s0, cu_seqlens=cu)
    torch.cuda.synchronize()
    assert o.shape == (1, 0, H, V) and torch.equal(fin, s0)


def test_binding_rejects_mismatched_tensors(kda):
    # the library trusts the sizes it is given, so the binding checks every tensor's shape,
    # contiguity and device against them before anything is enqueued
    inp = _base_bf16(T=96, H=2)
    q, k, v, g, beta = (inp[x] for x in ("q", "k", "v", "g", "beta"))
    bad = {
        "k": dict(k=k[:, :64].contiguous()),
        "v": dict(v=v[:, :64].contiguous()),
        "g": dict(g=g[:, :, :1].contiguous()),
        "beta": dict(beta=beta[:, :64].contiguous()),
        "q non-contiguous": dict(q=q.transpose(1, 2).contiguous().transpose(1, 2)),
        "initial_state": dict(initial_state=torch.zeros((2, 2, 128, 128), device="cuda")),
        "out": dict(out=torch.empty((1, 96, 2, 64), dtype=q.dtype, device="cuda")),
        "final_state": dict(final_state=torch.empty((1, 2, 128, 64), device="cuda")),
        "cu_seqlens on the host": dict(cu_seqlens=torch.tensor([0, 96], dtype=torch.int32)),
    }
    for what, change in bad.items():
        args = dict(q=q, k=k, v=v, g=g, beta=beta)
        args.update(change)
        with pytest.raises(ValueError):
            kda.fwd(args.pop("q"), args.pop("k"), args.pop("v"), args.pop("g"), args.pop("beta"),
                    **args)
    N, H, K, V = 2, 2, 128, 128
    st = torch.zeros((N, H, K, V), device="cuda")
    dq = torch.zeros((N, H, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        kda.decode(dq, dq, torch.zeros((N, H, V), dtype=torch.bfloat16, device="cuda"),
                   torch.zeros((N, H, K), device="cuda"), torch.zeros((N, 1), device="cuda"), st)
    torch.cuda.synchronize()


def _base_bf16(T=200, H=2, seed=41):
    return make_inputs(custom(B=1, T=T, H=H, K=128, V=128, dtype=torch.bfloat16, init_std=0.1,
                              seed=seed), device="cuda")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_causality_bit_exact(kda, dtype):
    """Perturbing any input after position n leaves o[:n+1] bit-identical ("KDA Doesn't
    Care About the Future": the first-row reference keeps the kernel causal)."""
    inp = make_inputs(custom(B=1, T=200, H=2, K=128, V=128, dtype=dtype, init_std=0.1, seed=42),
                      device="cuda")
    o0, _ = run_gpu(kda, inp)
    for n in (0, 15, 16, 37, 63, 64, 100, 150, 198):
        pert = dict(inp)
        for key in ("q", "k", "v", "g", "beta"):
            x = inp[key].clone()
            x[:, n + 1:] = (x[:, n + 1:].float() * 0.5 - 0.3).to(x.dtype)
            pert[key] = x
        pert["g"] = pert["g"].clamp(-5.0, 0.0)
        pert["beta"] = pert["beta"].clamp(0.0, 1.0)
        o1, _ = run_gpu(kda, pert)
        assert torch.equal(o0[:, :n + 1], o1[:, :n + 1]), f"future leak at n={n}"


def test_deterministic(kda):
    inp = _base_bf16()
    o0, f0 = run_gpu(kda, inp)
    for _ in range(3):
        o1, f1 = run_gpu(kda, inp)
        assert torch.equal(o0, o1) and torch.equal(f0, f1)


@pytest.mark.parametrize("shape", [(1, 64 * 512, 2, 0.1), (2, 64 * 600 + 37, 1, None)],
                         ids=["512chunks_init", "601chunks_tail"])
def test_pipelined_schedule(kda, orc, shape, monkeypatch):
    """The pipelined schedule (chunk ranges on two streams, state handed over in fp32)
    gives bit-identical results to the whole-problem schedule, and matches the oracle."""
    B, T, H, init = shape
    inp = make_inputs(custom(B=B, T=T, H=H, K=128, V=128, dtype=torch.bfloat16,
                             init_std=init, seed=T + H), device="cuda")
    monkeypatch.setenv("KDA_SCHEDULE", "pipelined")
    assert kda.launch_count(B, T, H, 128, 128) > 3   # really pipelined
    o_p, f_p = run_gpu(kda, inp)
    monkeypatch.delenv("KDA_SCHEDULE")
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in evs:
        e.record()
    o_w, f_w = run_gpu(kda, inp, events=evs)         # whole-problem schedule
    assert torch.equal(o_p, o_w) and torch.equal(f_p, f_w)
    o_ref, f_ref = run_oracle(orc, inp)
    eo, ef = errors(o_p, f_p, o_ref, f_ref)
    assert eo <= 2e-2 and ef <= 2e-2, (eo, ef)


@pytest.mark.parametrize("shape", [(6, 200, 14, 0.2), (1, 130, 80, None)],
                         ids=["84chains_init", "80chains"])
def test_per_chain_recurrence_form(kda, orc, shape):
    """With more chains than two CTAs per chain fit in one wave, the recurrence runs one CTA
    per (sequence, head) on the transposed record form; it must agree with the oracle like
    the value-sliced form the small cases use."""
    B, T, H, init = shape
    inp = make_inputs(custom(B=B, T=T, H=H, K=128, V=128, dtype=torch.bfloat16, init_std=init,
                             seed=B + T + H), device="cuda")
    check(kda, orc, inp)


@pytest.mark.parametrize("shape", [(2, 4096, 4, None), (3, 64 * 37 + 29, 2, 0.1), (1, 64, 3, 0.1),
                                   (1, 1, 2, None), (2, 63, 1, 0.1)],
                         ids=["dense_like", "tail_init", "one_chunk", "one_token", "short"])
def test_fused_schedule(kda, orc, shape, monkeypatch):
    """Few chains of fixed-length sequences run fused: one cooperative launch in which
    some CTAs run the per-chain recurrences while the others produce the records.  It
    matches the oracle, and the two-kernel schedule (value-sliced recurrence, other
    operand rounding) to the bf16 tolerance."""
    B, T, H, init = shape
    inp = make_inputs(custom(B=B, T=T, H=H, K=128, V=128, dtype=torch.bfloat16,
                             init_std=init, seed=T * 7 + H), device="cuda")
    assert kda.launch_count(B, T, H, 128, 128) == 1   # fused
    o_f, f_f = run_gpu(kda, inp)
    o_ref, f_ref = run_oracle(orc, inp)
    eo, ef = errors(o_f, f_f, o_ref, f_ref)
    assert eo <= 2e-2 and ef <= 2e-2, (eo, ef)
    monkeypatch.setenv("KDA_SCHEDULE", "two")
    assert kda.launch_count(B, T, H, 128, 128) == 2
    o_t, f_t = run_gpu(kda, inp)
    monkeypatch.delenv("KDA_SCHEDULE")
    eo, ef = errors(o_t, f_t, o_ref, f_ref)
    assert eo <= 2e-2 and ef <= 2e-2, (eo, ef)
    assert (o_f.float() - o_t.float()).abs().max().item() <= 2e-2
    assert (f_f - f_t).abs().max().item() <= 2e-2
    o_2, f_2 = run_gpu(kda, inp)                     # repeatable (flags reset per call)
    assert torch.equal(o_2, o_f) and torch.equal(f_2, f_f)


@pytest.mark.parametrize("shape", [(1, 64 * 40 + 17, 2, 0.1), (2, 64 * 9, 3, None), (1, 64 * 4, 1, 0.1)],
                         ids=["tail_init", "batch2", "four_chunks"])
def test_scan_schedule(kda, orc, shape, monkeypatch):
    """The chunk-parallel scan (segment summaries Phi, Psi from S = I with U = 0 and from
    S = 0, a per-chain fp32 merge, then every segment replayed from its merged start)
    matches the oracle and the two-kernel schedule to the bf16 tolerance."""
    B, T, H, init = shape
    inp = make_inputs(custom(B=B, T=T, H=H, K=128, V=128, dtype=torch.bfloat16,
                             init_std=init, seed=T * 3 + H), device="cuda")
    monkeypatch.setenv("KDA_SCHEDULE", "scan")
    assert kda.launch_count(B, T, H, 128, 128) == 4   # intra, summaries, merge, replay
    o_s, f_s = run_gpu(kda, inp)
    monkeypatch.setenv("KDA_SCHEDULE", "two")
    o_t, f_t = run_gpu(kda, inp)
    monkeypatch.delenv("KDA_SCHEDULE")
    o_ref, f_ref = run_oracle(orc, inp)
    for o_x, f_x in ((o_s, f_s), (o_t, f_t)):
        eo, ef = errors(o_x, f_x, o_ref, f_ref)
        assert eo <= 2e-2 and ef <= 2e-2, (eo, ef)
    assert (o_s.float() - o_t.float()).abs().max().item() <= 2e-2


def test_scan_schedule_automatic(kda, orc):
    """Two chains of 128 chunks take the scan schedule by themselves; the plan's
    workloads take theirs."""
    inp = make_inputs(custom(B=1, T=64 * 128, H=2, K=128, V=128, dtype=torch.bfloat16,
                             init_std=0.1, seed=77), device="cuda")
    assert kda.launch_count(1, 64 * 128, 2, 128, 128) == 4
    assert kda.schedule(1, 64 * 128, 2, 128, 128) == "scan"
    assert kda.schedule(2, 4096, 16, 128, 128) == "fused"           # dense
    assert kda.schedule(1, 131072, 32, 128, 128) == "fused"         # long
    assert kda.schedule(32, 2048, 32, 128, 128) == "two_kernels"    # serving
    check(kda, orc, inp)


@pytest.mark.parametrize("mode", ["two", "fused"])
def test_forced_schedules_dense(kda, orc, mode, monkeypatch):
    """The dense workload's shape under each schedule, checked on a sample of chains."""
    w = WORKLOADS["dense_bf16"]
    inp = make_inputs(w, device="cuda")
    monkeypatch.setenv("KDA_SCHEDULE", mode)
    o, fin = run_gpu(kda, inp)
    monkeypatch.delenv("KDA_SCHEDULE")
    for b, h in ((0, 0), (1, 15), (1, 7)):
        one = {k_: (v_[b:b + 1, :, h:h + 1].contiguous() if k_ in ("q", "k", "v", "g", "beta") else v_)
               for k_, v_ in inp.items()}
        one["initial_state"] = None
        one["cu_seqlens"] = None
        o_ref, f_ref = run_oracle(orc, {**one, "T": one["q"].shape[1]})
        eo = float(np.max(np.abs(o[b:b + 1, :, h:h + 1].float().cpu().numpy() - o_ref)))
        ef = float(np.max(np.abs(fin[b:b + 1, h:h + 1].cpu().numpy() - f_ref)))
        assert eo <= 2e-2 and ef <= 2e-2, (b, h, eo, ef)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_split_call_resume(kda, dtype):
    inp = make_inputs(custom(B=2, T=300, H=2, K=128, V=128, dtype=dtype, init_std=0.1, seed=43),
                      device="cuda")
    o, fin = run_gpu(kda, inp)
    for a in (64, 100):
        part1 = {k_: (v_[:, :a].contiguous() if k_ in ("q", "k", "v", "g", "beta") else v_)
                 for k_, v_ in inp.items()}
        o1, f1 = run_gpu(kda, part1)
        part2 = {k_: (v_[:, a:].contiguous() if k_ in ("q", "k", "v", "g", "beta") else v_)
                 for k_, v_ in inp.items()}
        part2["initial_state"] = f1
        o2, f2 = run_gpu(kda, part2)
        tol = TOL[dtype]
        assert (torch.cat([o1, o2], 1).float() - o.float()).abs().max().item() <= tol
        assert (f2 - fin).abs().max().item() <= tol
        if a % 64 == 0:   # the chunk grid is the same, so the result is bit-identical
            assert torch.equal(torch.cat([o1, o2], 1), o) and torch.equal(f2, fin)


def test_varlen_isolation_bit_exact(kda):
    lens = [5, 77, 64, 1, 130]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    inp = make_inputs(custom(B=1, T=int(cu[-1]), H=2, K=128, V=128, dtype=torch.bfloat16,
                             seed=44), device="cuda")
    inp["cu_seqlens"] = cu
    inp["initial_state"] = 0.1 * torch.randn((len(lens), 2, 128, 128), device="cuda")
    o, fin = run_gpu(kda, inp)
    for n in range(len(lens)):
        a, b = int(cu[n]), int(cu[n + 1])
        one = {k_: (v_[:, a:b].contiguous() if k_ in ("q", "k", "v", "g", "beta") else v_)
               for k_, v_ in inp.items()}
        one["cu_seqlens"] = None
        one["initial_state"] = inp["initial_state"][n:n + 1].contiguous()
        o1, f1 = run_gpu(kda, one)
        assert torch.equal(o[:, a:b], o1) and torch.equal(fin[n:n + 1], f1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_gate_floor_stress(kda, orc, dtype):
    """Every gate at the -5 bound: the rescaled operands of a 16-key window stay finite
    (the validation gap named in the Tokamax design doc, 6.4)."""
    inp = make_inputs(custom(B=1, T=256, H=2, K=128, V=128, dtype=dtype, seed=45), device="cuda")
    inp["g"] = torch.full_like(inp["g"], -5.0)
    check(kda, orc, inp)


def test_chunk_index_matches_definition(kda):
    lens = [0, 1, 64, 65, 300, 0, 128, 7]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    ctab, stab, count = kda.build_chunk_index(cu, 1, int(cu[-1]))
    exp_c, exp_s = [], []
    for n, L in enumerate(lens):
        exp_s.append([len(exp_c), (L + 63) // 64])
        for j in range((L + 63) // 64):
            exp_c.append([n, int(cu[n]) + 64 * j, min(64, L - 64 * j), j])
    assert count == len(exp_c)
    assert ctab.tolist() == exp_c and stab.tolist() == exp_s
    ctab, stab, count = kda.build_chunk_index(None, 3, 130)
    assert count == 9 and stab.tolist() == [[0, 3], [3, 3], [6, 3]]
    assert ctab[4].tolist() == [1, 130 + 64, 64, 1] and ctab[8].tolist() == [2, 260 + 128, 2, 2]


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times
# ---------------------------------------------------------------------------

def _slice(inp, batches=None, heads=None):
    """CPU copy of the inputs restricted to some batch rows and heads."""
    out = dict(inp)
    for key in ("q", "k", "v", "g", "beta"):
        x = inp[key].cpu()
        if batches is not None:
            x = x[batches]
        if heads is not None:
            x = x[:, :, heads]
        out[key] = x.contiguous()
    if inp["initial_state"] is not None:
        s = inp["initial_state"].cpu()
        if batches is not None and inp["cu_seqlens"] is None:
            s = s[batches]
        if heads is not None:
            s = s[:, heads]
        out["initial_state"] = s.contiguous()
    if inp["cu_seqlens"] is not None:
        out["cu_seqlens"] = inp["cu_seqlens"].cpu()
    return out


SAMPLES = {
    "dense_bf16": (None, None),
    "varlen_bf16": (None, [0, 13, 31]),
    "long_bf16": (None, [0, 21]),
    "serving_bf16": ([0, 17, 31], [0, 9, 31]),
    "few_long_bf16": (None, [1]),
}


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_size_workload(kda, orc, name):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    gpu = {k_: (v_.cuda() if torch.is_tensor(v_) else v_) for k_, v_ in inp.items()}
    o, fin = run_gpu(kda, gpu)
    batches, heads = SAMPLES[name]
    ref_in = _slice(inp, batches, heads)
    o_ref, f_ref = run_oracle(orc, ref_in)
    o_s, f_s = o.cpu(), fin.cpu()
    if batches is not None:
        o_s, f_s = o_s[batches], f_s[batches]
    if heads is not None:
        o_s, f_s = o_s[:, :, heads], f_s[:, heads]
    eo, ef = errors(o_s, f_s, o_ref, f_ref)
    assert np.isfinite(o.float().cpu().numpy()).all()
    assert eo <= 2e-2 and ef <= 2e-2, f"{name}: max|o-ref|={eo:.3e} max|S-ref|={ef:.3e}"
