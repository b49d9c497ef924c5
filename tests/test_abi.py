"""C-ABI contract checks that need no GPU: the library loads, exports every function
that include/kda.h declares, and rejects invalid arguments before launching anything."""
import ctypes
import os
import re

import pytest
import torch

import kimi_delta_attention_11_gb300 as kda
from kimi_delta_attention_11_gb300 import _native

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "kda.h")

OK, INVALID, UNSUPPORTED, ALIGN, WORKSPACE, CUDA, TIMEOUT, DEVICE = range(8)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return kda.load_library()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "kda_fwd" in names and len(names) >= 6
    for n in names:
        assert hasattr(lib, n), f"{n} declared in kda.h but not exported"
        assert n in _native._SIGNATURES, f"{n} has no binding signature"


def test_status_strings(lib):
    for s in range(8):
        assert lib.kda_status_string(s).decode()
    assert lib.kda_status_string(99).decode() == "unknown status"
    assert lib.kda_abi_version() == 103


def test_launch_count(lib):
    """bf16 K = V = 128 fixed length: no index kernel, intra + recurrence (once per range
    of 32 chunks when pipelined: <= 128 chains, >= 512 chunks per sequence); packed input
    and the other paths: index + intra + recurrence.  (Without a device the SM count is
    unknown, so no call is fused or scanned; tests/test_gpu_parity.py covers those.)"""
    lc = lambda *a: lib.kda_fwd_launch_count(*a)
    bf16, f32 = 0, 1
    assert lc(2, 4096, 16, 128, 128, 0, 64, bf16) == 2             # 64 chunks
    assert lc(1, 131072, 32, 128, 128, 0, 64, bf16) == 2 * 64      # 2048 chunks
    assert lc(1, 512 * 64, 2, 128, 128, 0, 64, bf16) == 2 * 16
    assert lc(1, 511 * 64, 2, 128, 128, 0, 64, bf16) == 2          # 511 chunks
    assert lc(1, 600 * 64 + 5, 2, 128, 128, 0, 64, bf16) == 2 * 19
    assert lc(32, 2048, 32, 128, 128, 0, 64, bf16) == 2            # 1024 chains
    assert lc(1, 37000, 32, 128, 128, 8, 64, bf16) == 3            # packed
    assert lc(1, 131072, 32, 128, 128, 0, 64, f32) == 3            # fp32 path
    assert lc(1, 131072, 32, 64, 64, 0, 64, bf16) == 3             # other shapes
    assert lc(2, 4096, 16, 128, 128, 0, 32, bf16) == -1            # rejected sizes


def test_schedule_query(lib):
    """kda_fwd_schedule names the schedule kda_fwd_launch_count counts."""
    sc = lambda *a: lib.kda_fwd_schedule(*a)
    bf16, f32 = 0, 1
    assert sc(1, 131072, 32, 128, 128, 0, 64, bf16) == 1            # pipelined
    assert sc(32, 2048, 32, 128, 128, 0, 64, bf16) == 0             # two kernels
    assert sc(1, 37000, 32, 128, 128, 8, 64, bf16) == 0             # packed
    assert sc(1, 131072, 32, 128, 128, 0, 64, f32) == 0             # fp32 path
    assert sc(2, 4096, 16, 128, 128, 0, 32, bf16) == -1             # rejected sizes


@pytest.mark.parametrize("sizes,sms,expected", [
    ((2, 4096, 16, 0), 152, "fused"),          # dense: 32 chains, a fifth of the SMs
    ((1, 131072, 32, 0), 152, "fused"),        # long: 32 chains of 2048 chunks
    ((1, 262144, 2, 0), 152, "scan"),          # two chains of 4096 chunks
    ((1, 64 * 100, 2, 0), 152, "fused"),       # few chains, too short to scan
    ((32, 2048, 32, 0), 152, "two_kernels"),   # serving: 1024 chains
    ((1, 37000, 32, 8), 152, "two_kernels"),   # packed sequences
    ((1, 131072, 32, 0), 0, "pipelined"),      # no SM count: neither fused nor scanned
    ((2, 4096, 16, 0), 64, "two_kernels"),     # 32 chains need three times as many SMs
    ((2, 4096, 16, 0), 96, "fused"),
    ((1, 262144, 2, 0), 15, "fused"),          # the scan wants eight SMs per chain
    ((1, 262144, 2, 0), 16, "scan"),
])
def test_schedule_rules_for_a_given_sm_count(sizes, sms, expected, monkeypatch):
    """The host's choice of schedule (kda_fwd_schedule_for), which kda_fwd makes with the
    current device's SM count."""
    monkeypatch.delenv("KDA_SCHEDULE", raising=False)
    B, T, H, nseq = sizes
    assert kda.schedule(B, T, H, 128, 128, nseq, sm_count=sms) == expected


def test_schedule_override_and_rejections(lib, monkeypatch):
    sc = lambda *a: lib.kda_fwd_schedule_for(*a)
    bf16, f32 = 0, 1
    monkeypatch.setenv("KDA_SCHEDULE", "two")
    assert sc(2, 4096, 16, 128, 128, 0, 64, bf16, 152) == 0
    monkeypatch.setenv("KDA_SCHEDULE", "fused")             # forced where it can run
    assert sc(2, 4096, 16, 128, 128, 0, 64, bf16, 64) == 2
    assert sc(2, 4096, 16, 128, 128, 0, 64, bf16, 63) == 0  # 32 chains need 64 SMs
    monkeypatch.setenv("KDA_SCHEDULE", "scan")
    assert sc(2, 4096, 16, 128, 128, 0, 64, bf16, 152) == 3
    monkeypatch.delenv("KDA_SCHEDULE")
    assert sc(1, 131072, 32, 128, 128, 0, 64, f32, 152) == 0  # fp32 path
    assert sc(2, 4096, 16, 128, 128, 0, 32, bf16, 152) == -1  # rejected sizes
    assert sc(2, 4096, 16, 128, 128, 0, 64, bf16, -1) == -1   # negative SM count


def test_workspace_bytes_rules(lib):
    ws = lambda *a: lib.kda_fwd_workspace_bytes(*a)
    bf16, f32 = 0, 1
    assert ws(2, 4096, 16, 128, 128, 0, 64, bf16) > 0
    assert ws(2, 4096, 16, 128, 128, 0, 32, bf16) == 0        # chunk size
    assert ws(2, 4096, 16, 96, 128, 0, 64, bf16) == 0         # K unsupported
    assert ws(2, 4096, 16, 512, 128, 0, 64, bf16) == 0        # K > 256
    assert ws(0, 4096, 16, 128, 128, 0, 64, bf16) == 0        # B
    assert ws(1, 5000, 4, 64, 64, 3, 64, f32) >= ws(1, 5000, 4, 64, 64, 1, 64, f32)
    assert ws(2, 0, 1, 64, 64, 0, 64, f32) > 0                # T = 0 is valid
    assert ws(1, 1000, 8, 128, 128, 2, 64, bf16) >= ws(1, 1000, 8, 128, 128, 1, 64, bf16)


FAKE = 0x10000  # an aligned address that is never dereferenced: calls fail validation


def call_fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=0.1, chunk=64, s0=None, cu=None,
             nseq=0, o=FAKE, fin=None, B=1, T=64, H=1, K=64, V=64, dt=1, ws=FAKE,
             wsb=1 << 40, stream=None)
    a.update(kw)
    return lib.kda_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["chunk"], a["s0"],
                       a["cu"], a["nseq"], a["o"], a["fin"], a["B"], a["T"], a["H"], a["K"],
                       a["V"], a["dt"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), INVALID), (dict(beta=None), INVALID), (dict(o=None), INVALID),
    (dict(B=0), INVALID), (dict(T=-1), INVALID), (dict(H=0), INVALID),
    (dict(K=512), INVALID), (dict(V=300), INVALID), (dict(dt=7), INVALID),
    (dict(cu=FAKE, nseq=2, B=2), INVALID), (dict(cu=FAKE, nseq=0), INVALID),
    (dict(chunk=32), UNSUPPORTED), (dict(K=96), UNSUPPORTED), (dict(V=32), UNSUPPORTED),
    (dict(q=FAKE + 8), ALIGN), (dict(o=FAKE + 4), ALIGN), (dict(s0=FAKE + 2), ALIGN),
    (dict(beta=FAKE + 2), ALIGN), (dict(g=FAKE + 4), ALIGN),
    (dict(fin=FAKE + 12), ALIGN), (dict(cu=FAKE + 2, nseq=1), ALIGN), (dict(ws=FAKE + 8), ALIGN),
    (dict(ws=None), WORKSPACE), (dict(wsb=16), WORKSPACE),
])
def test_fwd_rejects_before_launch(lib, kw, status):
    assert call_fwd(lib, **kw) == status


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
def test_valid_call_without_gpu_reports_device(lib):
    assert call_fwd(lib) == DEVICE
    assert call_fwd(lib, beta=FAKE + 4) == DEVICE          # beta needs 4-byte alignment only
    assert call_fwd(lib, q=None, k=None, v=None, g=None, beta=None, o=None, T=0) == DEVICE


def test_profiled_rejects_short_event_list(lib):
    a = [FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, 64, None, None, 0, FAKE, None, 1, 64, 1, 64, 64, 1,
         FAKE, 1 << 40, None]
    evs = (ctypes.c_void_p * 2)()
    assert lib.kda_fwd_profiled(*a, evs, 2) == INVALID
    assert lib.kda_fwd_profiled(*a, None, 4) == INVALID
    a[0] = None
    assert lib.kda_fwd_profiled(*a, None, 0) == INVALID


def test_chunk_index_rejects(lib):
    off = ctypes.c_size_t(0)
    f = lib.kda_build_chunk_index
    assert f(None, 0, 0, 10, 64, FAKE, 1 << 30, None, None, None, None) == INVALID
    assert f(FAKE, 2, 2, 10, 64, FAKE, 1 << 30, None, None, None, None) == INVALID
    assert f(None, 0, 1, 10, 32, FAKE, 1 << 30, None, None, None, None) == UNSUPPORTED
    assert f(None, 0, 1, 10, 64, None, 1 << 30, None, None, None, None) == WORKSPACE
    assert f(None, 0, 1, 10, 64, FAKE, 8, ctypes.byref(off), None, None, None) == WORKSPACE


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(kda.KdaLibraryMissing):
        _native.load_library(str(tmp_path / "missing.so"))


def test_binding_refuses_host_tensors(lib):
    # there is no CPU path: host tensors are rejected before the library is called
    B, T, H, K, V = 1, 64, 2, 64, 64
    q = torch.zeros((B, T, H, K))
    with pytest.raises(ValueError, match="CUDA"):
        kda.fwd(q, q, torch.zeros((B, T, H, V)), q, torch.zeros((B, T, H)))
    s = torch.zeros((2, H, K, V))
    d = torch.zeros((2, H, K))
    with pytest.raises(ValueError, match="CUDA"):
        kda.decode(d, d, torch.zeros((2, H, V)), d, torch.zeros((2, H)), s)


def call_decode(lib, opts=None, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, scale=0.1, state=FAKE, o=FAKE, N=2, H=1,
             K=64, V=64, dt=1, stream=None)
    a.update(kw)
    return lib.kda_decode(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["state"],
                          a["o"], a["N"], a["H"], a["K"], a["V"], a["dt"],
                          None if opts is None else ctypes.byref(opts), a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), INVALID), (dict(state=None), INVALID), (dict(o=None), INVALID),
    (dict(N=-1), INVALID), (dict(H=0), INVALID), (dict(dt=5), INVALID), (dict(K=512), INVALID),
    (dict(K=96), UNSUPPORTED), (dict(V=32), UNSUPPORTED),
    (dict(q=FAKE + 2), ALIGN), (dict(state=FAKE + 2), ALIGN), (dict(beta=FAKE + 1), ALIGN),
    (dict(N=0, q=None, state=None), OK),      # nothing to do
])
def test_decode_rejects_before_launch(lib, kw, status):
    assert call_decode(lib, **kw) == status


@pytest.mark.parametrize("fields,status", [
    (dict(use_gate_in_kernel=1, a_log=None), INVALID),              # a_log required
    (dict(use_gate_in_kernel=1, a_log=FAKE, lower_bound=-6.0), INVALID),
    (dict(use_gate_in_kernel=1, a_log=FAKE, lower_bound=0.5), INVALID),
    (dict(use_gate_in_kernel=1, a_log=FAKE + 2), ALIGN),
    (dict(use_gate_in_kernel=1, a_log=FAKE, dt_bias=FAKE + 1), ALIGN),
])
def test_gate_options_validated(lib, fields, status):
    opts = _native._GateOptions(**{"use_gate_in_kernel": 0, "a_log": None, "dt_bias": None,
                                   "lower_bound": 0.0, "qk_l2norm": 0, **fields})
    assert call_decode(lib, opts) == status
    a = [FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, 64, None, None, 0, FAKE, None, 1, 64, 1, 64, 64, 1,
         FAKE, 1 << 40]
    assert lib.kda_fwd_ex(*a, ctypes.byref(opts), None) == status
