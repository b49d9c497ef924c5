"""ctypes binding of libkda_gb300.so (the C ABI in include/kda.h).

Argument marshalling only: tensors are passed as raw device pointers with the current
CUDA stream; every step of the computation runs in the library's CUDA kernels.  There
is no fallback: without the built library every call raises ``KdaLibraryMissing``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

KDA_OK = 0
STATUS_NAMES = {
    0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_ALIGNMENT",
    4: "KDA_ERR_WORKSPACE", 5: "KDA_ERR_CUDA", 6: "KDA_ERR_DEVICE_TIMEOUT", 7: "KDA_ERR_DEVICE",
}
DTYPE_CODES = {torch.bfloat16: 0, torch.float32: 1}


class KdaLibraryMissing(RuntimeError):
    """The CUDA library has not been built (run __graft_entry__.build())."""


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} "
                         f"({status_string(status)})")


_LIB = None
_LOCK = threading.Lock()


class _GateOptions(ctypes.Structure):
    """kda_gate_options of include/kda.h."""
    _fields_ = [("use_gate_in_kernel", ctypes.c_int), ("a_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p), ("lower_bound", ctypes.c_float),
                ("qk_l2norm", ctypes.c_int)]

_vp, _sz, _i, _f = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
_SIGNATURES = {
    "kda_fwd_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "kda_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _f, _i, _vp, _vp, _i, _vp, _vp,
                     _i, _i, _i, _i, _i, _i, _vp, _sz, _vp]),
    "kda_fwd_profiled": (_i, [_vp, _vp, _vp, _vp, _vp, _f, _i, _vp, _vp, _i, _vp, _vp,
                              _i, _i, _i, _i, _i, _i, _vp, _sz, _vp,
                              ctypes.POINTER(ctypes.c_void_p), _i]),
    "kda_fwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _f, _i, _vp, _vp, _i, _vp, _vp,
                             _i, _i, _i, _i, _i, _i, _vp]),
    "kda_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _f, _i, _vp, _vp, _i, _vp, _vp,
                        _i, _i, _i, _i, _i, _i, _vp, _sz, ctypes.POINTER(_GateOptions), _vp]),
    "kda_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _f, _vp, _vp, _i, _i, _i, _i, _i,
                        ctypes.POINTER(_GateOptions), _vp]),
    "kda_build_chunk_index": (_i, [_vp, _i, _i, _i, _i, _vp, _sz, ctypes.POINTER(_sz),
                                   ctypes.POINTER(_sz), ctypes.POINTER(_sz), _vp]),
    "kda_selftest_umma": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp]),
    "kda_status_string": (ctypes.c_char_p, [_i]),
    "kda_get_device_status": (_i, [_vp, _vp]),
    "kda_abi_version": (_i, []),
    "kda_fwd_launch_count": (_i, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "kda_fwd_schedule": (_i, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "kda_fwd_schedule_for": (_i, [_i, _i, _i, _i, _i, _i, _i, _i, _i]),
}


def library_path() -> str:
    return _build.LIBRARY


def load_library(path: Optional[str] = None):
    """Load (once) and return the ctypes handle of libkda_gb300.so."""
    global _LIB
    with _LOCK:
        if _LIB is not None and path is None:
            return _LIB
        p = path or library_path()
        if not os.path.exists(p):
            raise KdaLibraryMissing(
                f"{p} not found: build the CUDA library first (__graft_entry__.build())")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _LIB = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load_library().kda_status_string(int(status)).decode()
    except KdaLibraryMissing:
        return STATUS_NAMES.get(status, "unknown")


def _check(name: str, t: torch.Tensor, shape: tuple, device: torch.device) -> None:
    """The library reads and writes through raw pointers with the sizes it is given, so
    every tensor must have the shape those sizes imply, be contiguous and live on the
    calling device."""
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def workspace_bytes(B: int, T: int, H: int, K: int, V: int, num_seqs: int = 0,
                    dtype: torch.dtype = torch.bfloat16, chunk_size: int = 64) -> int:
    n = load_library().kda_fwd_workspace_bytes(B, T, H, K, V, num_seqs, chunk_size,
                                               DTYPE_CODES[dtype])
    if n == 0:
        raise KdaError(1, "kda_fwd_workspace_bytes")
    return int(n)


def launch_count(B: int, T: int, H: int, K: int, V: int, num_seqs: int = 0,
                 dtype: torch.dtype = torch.bfloat16, chunk_size: int = 64) -> int:
    """Number of kernel launches one kda_fwd makes for these sizes."""
    n = load_library().kda_fwd_launch_count(B, T, H, K, V, num_seqs, chunk_size,
                                            DTYPE_CODES[dtype])
    if n < 0:
        raise KdaError(1, "kda_fwd_launch_count")
    return int(n)


SCHEDULES = {0: "two_kernels", 1: "pipelined", 2: "fused", 3: "scan"}


def schedule(B: int, T: int, H: int, K: int, V: int, num_seqs: int = 0,
             dtype: torch.dtype = torch.bfloat16, chunk_size: int = 64,
             sm_count: Optional[int] = None) -> str:
    """Schedule one kda_fwd takes for these sizes on the current device, or on a device
    with `sm_count` SMs."""
    lib = load_library()
    if sm_count is None:
        n = lib.kda_fwd_schedule(B, T, H, K, V, num_seqs, chunk_size, DTYPE_CODES[dtype])
    else:
        n = lib.kda_fwd_schedule_for(B, T, H, K, V, num_seqs, chunk_size, DTYPE_CODES[dtype],
                                     int(sm_count))
    if n < 0:
        raise KdaError(1, "kda_fwd_schedule")
    return SCHEDULES[int(n)]


def _gate_struct(gate: Optional[dict], H: int, K: int):
    """Validated kda_gate_options from a dict with keys a_log ([H] fp32 CUDA),
    dt_bias (optional [H*K] fp32 CUDA), lower_bound (float, 0 = softplus form),
    use_gate_in_kernel (default True when a_log is given) and qk_l2norm (bool)."""
    if gate is None:
        return None
    a_log, dt_bias = gate.get("a_log"), gate.get("dt_bias")
    use = bool(gate.get("use_gate_in_kernel", a_log is not None))
    for name, t, n in (("a_log", a_log, H), ("dt_bias", dt_bias, H * K)):
        if t is not None and (not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous()
                              or t.numel() != n):
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor of {n} elements")
    opts = _GateOptions(int(use), None if a_log is None else a_log.data_ptr(),
                        None if dt_bias is None else dt_bias.data_ptr(),
                        float(gate.get("lower_bound", 0.0)), int(bool(gate.get("qk_l2norm", False))))
    return opts


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
        beta: torch.Tensor, scale: Optional[float] = None,
        initial_state: Optional[torch.Tensor] = None,
        cu_seqlens: Optional[torch.Tensor] = None, output_final_state: bool = True,
        chunk_size: int = 64, workspace: Optional[torch.Tensor] = None,
        out: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
        events=None, gate: Optional[dict] = None):
    """Chunkwise KDA forward on the current CUDA stream (no host synchronisation).

    q, k: [B,T,H,K]; v: [B,T,H,V] (bf16 or fp32, all the same dtype); g: [B,T,H,K] fp32;
    beta: [B,T,H] fp32; initial_state: optional [N,H,K,V] fp32; cu_seqlens: optional
    int32 [N+1] (then B == 1).  Returns (o [B,T,H,V] in q.dtype, final_state [N,H,K,V]
    fp32 or None).  ``workspace``/``out``/``final_state`` may be passed to reuse memory.
    ``events``: optional list of >= 4 ``torch.cuda.Event`` recorded around the stages
    (chunk index, intra-chunk kernel, recurrence kernel) for per-kernel timing; with
    events the kernels run back to back, one launch each (see include/kda.h).
    ``gate``: optional in-kernel gate activation / q-k normalisation (kda_fwd_ex):
    dict(a_log=[H] fp32, dt_bias=[H*K] fp32 or None, lower_bound=0.0 (softplus form) or
    in [-5, 0) (sigmoid form), qk_l2norm=bool); g then holds raw gates when a_log is set.
    """
    lib = load_library()
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, g must be [B,T,H,K] and v [B,T,H,V]")
    B, T, H, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = K ** -0.5
    dev = q.device
    if k.dtype != q.dtype or v.dtype != q.dtype or q.dtype not in DTYPE_CODES:
        raise ValueError("q, k, v must share one dtype, bf16 or fp32")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise ValueError("g and beta must be fp32")
    _check("q", q, (B, T, H, K), dev)
    _check("k", k, (B, T, H, K), dev)
    _check("v", v, (B, T, H, V), dev)
    _check("g", g, (B, T, H, K), dev)
    _check("beta", beta, (B, T, H), dev)
    num_seqs = 0
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
            raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
        _check("cu_seqlens", cu_seqlens, tuple(cu_seqlens.shape), dev)
        num_seqs = cu_seqlens.numel() - 1
    N = num_seqs if cu_seqlens is not None else B
    if initial_state is not None:
        if initial_state.dtype != torch.float32:
            raise ValueError("initial_state must be fp32")
        _check("initial_state", initial_state, (N, H, K, V), dev)
    need = workspace_bytes(B, T, H, K, V, num_seqs, q.dtype, chunk_size)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    else:
        _check("workspace", workspace, tuple(workspace.shape), dev)
    if out is not None:
        if out.dtype != q.dtype:
            raise ValueError("out must have q's dtype")
        _check("out", out, (B, T, H, V), dev)
    o = out if out is not None else torch.empty((B, T, H, V), dtype=q.dtype, device=dev)
    fin = final_state
    if fin is not None:
        if fin.dtype != torch.float32:
            raise ValueError("final_state must be fp32")
        _check("final_state", fin, (N, H, K, V), dev)
    if fin is None and output_final_state:
        fin = torch.empty((N, H, K, V), dtype=torch.float32, device=dev)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), chunk_size,
            _ptr(initial_state), _ptr(cu_seqlens), num_seqs, _ptr(o), _ptr(fin),
            B, T, H, K, V, DTYPE_CODES[q.dtype], _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream_handle(dev))
    opts = _gate_struct(gate, H, K)
    if opts is not None:
        if events is not None:
            raise ValueError("events and gate options cannot be combined")
        st = lib.kda_fwd_ex(*args[:-1], ctypes.byref(opts), args[-1])
    elif events is None:
        st = lib.kda_fwd(*args)
    else:
        if any(e.cuda_event == 0 for e in events):
            raise ValueError("events must have been created (record each once before use)")
        handles = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        st = lib.kda_fwd_profiled(*args, handles, len(events))
    if st != KDA_OK:
        raise KdaError(st, "kda_fwd")
    return o, fin


def decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
           beta: torch.Tensor, state: torch.Tensor, scale: Optional[float] = None,
           out: Optional[torch.Tensor] = None, gate: Optional[dict] = None) -> torch.Tensor:
    """One decode step on the current CUDA stream: q, k [N,H,K], v [N,H,V] (bf16 or fp32),
    g [N,H,K] fp32, beta [N,H] fp32, state [N,H,K,V] fp32 updated in place.  Returns o
    [N,H,V] in q.dtype.  ``gate`` as for fwd."""
    lib = load_library()
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, g must be [N,H,K] and v [N,H,V]")
    N, H, K = q.shape
    V = v.shape[-1]
    if scale is None:
        scale = K ** -0.5
    dev = q.device
    if k.dtype != q.dtype or v.dtype != q.dtype or q.dtype not in DTYPE_CODES:
        raise ValueError("q, k, v must share one dtype, bf16 or fp32")
    if g.dtype != torch.float32 or beta.dtype != torch.float32 or state.dtype != torch.float32:
        raise ValueError("g, beta and state must be fp32")
    for name, t, shape in (("q", q, (N, H, K)), ("k", k, (N, H, K)), ("v", v, (N, H, V)),
                           ("g", g, (N, H, K)), ("beta", beta, (N, H)),
                           ("state", state, (N, H, K, V))):
        _check(name, t, shape, dev)
    if out is not None:
        if out.dtype != q.dtype:
            raise ValueError("out must have q's dtype")
        _check("out", out, (N, H, V), dev)
    o = out if out is not None else torch.empty((N, H, V), dtype=q.dtype, device=dev)
    opts = _gate_struct(gate, H, K)
    st = lib.kda_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                        _ptr(state), _ptr(o), N, H, K, V, DTYPE_CODES[q.dtype],
                        None if opts is None else ctypes.byref(opts), _stream_handle(q.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode")
    return o


def build_chunk_index(cu_seqlens: Optional[torch.Tensor], B: int, T: int,
                      device: Optional[torch.device] = None, chunk_size: int = 64):
    """Run the chunk-index kernel alone. Returns (chunk_table [n,4], seq_table [N,2],
    count) as int32 tensors read back to the host (this synchronises)."""
    lib = load_library()
    num_seqs = cu_seqlens.numel() - 1 if cu_seqlens is not None else 0
    dev = device or (cu_seqlens.device if cu_seqlens is not None else torch.device("cuda"))
    need = workspace_bytes(B, T, 1, 64, 64, num_seqs, torch.float32, chunk_size)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    offs = [ctypes.c_size_t(0) for _ in range(3)]
    st = lib.kda_build_chunk_index(_ptr(cu_seqlens), num_seqs, B, T, chunk_size, _ptr(ws), need,
                                   ctypes.byref(offs[0]), ctypes.byref(offs[1]),
                                   ctypes.byref(offs[2]), _stream_handle(dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_build_chunk_index")
    wsh = ws.cpu()
    count = int(wsh[offs[2].value:offs[2].value + 4].view(torch.int32)[0])
    N = num_seqs if cu_seqlens is not None else B
    ctab = wsh[offs[0].value:offs[0].value + 16 * count].view(torch.int32).view(count, 4)
    stab = wsh[offs[1].value:offs[1].value + 8 * N].view(torch.int32).view(N, 2)
    return ctab.clone(), stab.clone(), count


def selftest_umma(A: torch.Tensor, B: torch.Tensor, mode: int = 0) -> torch.Tensor:
    """Diagnostic tcgen05 GEMM: returns A[128,K] @ B[N,K]^T in fp32 (synchronises)."""
    lib = load_library()
    if mode == 2:      # B given transposed: [K, N]
        K, N = B.shape
    else:
        N, K = B.shape
    D = torch.empty((128, N), dtype=torch.float32, device=A.device)
    status = torch.zeros(1, dtype=torch.int32, device=A.device)
    st = lib.kda_selftest_umma(_ptr(A), _ptr(B), _ptr(D), N, K, mode, _ptr(status),
                               _stream_handle(A.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_selftest_umma")
    torch.cuda.synchronize(A.device)
    if int(status.item()) != 0:
        raise KdaError(int(status.item()), "kda_selftest_umma (device)")
    return D


def get_device_status(workspace: torch.Tensor) -> int:
    """Status word the kernels of the last kda_fwd on `workspace` left (synchronises)."""
    return int(load_library().kda_get_device_status(_ptr(workspace),
                                                    _stream_handle(workspace.device)))
