"""fp64 CPU oracle for the Kimi Delta Attention forward pass.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` import this package.  The CUDA library never calls it and shares no
code with it: ``kda_oracle.c`` is a plain C restatement of the token recurrence
(Tokamax "chunk_kda_fwd_design_doc", Appendix 9.1.2, Eq. (1)), of the chunkwise form
(same document, 9.1.3-9.1.6, Eq. (6)-(9)), of the raw-gate activation (9.1.3) and of the
q/k row normalisation (Kimi-K3 docs, "KDAChunkwise", FP32 core).

Every function here is pinned by ``tests/pins.py``; ``tests/test_oracle_mutants.py``
plants single mistakes in a copy of the C source and checks that a pin catches each.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "kda_oracle.c")
LIBRARY = os.path.join(HERE, "libkda_oracle.so")

# -ffp-contract=off: no fused multiply-add contraction, so x86 and Arm hosts
# evaluate the same expressions in the same fp64 operations.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off"]


def build_oracle(source: str = SOURCE, output: str = LIBRARY, force: bool = False) -> str:
    """Compile the C oracle with gcc into a shared library and return its path."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    cmd = ["gcc", *CFLAGS, "-I", HERE, "-o", output, source, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return output


def _f64(x) -> np.ndarray:
    """Exact widening of an input tensor (bf16/fp32/fp64 torch or numpy) to fp64."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: bf16 -> fp32 is exact, numpy has no bf16
        x = x.detach().to("cpu")
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: Optional[np.ndarray], ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, lib_path: Optional[str] = None):
        self.path = lib_path or build_oracle()
        self.lib = ctypes.CDLL(self.path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        common = [dp, dp, dp, dp, dp, ctypes.c_double, dp, ip, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        self.lib.kda_oracle_recurrent.argtypes = common + [dp, dp, ctypes.c_int]
        self.lib.kda_oracle_recurrent.restype = ctypes.c_int
        self.lib.kda_oracle_chunkwise.argtypes = common + [ctypes.c_int, dp, dp, ctypes.c_int]
        self.lib.kda_oracle_chunkwise.restype = ctypes.c_int
        self.lib.kda_oracle_gate.argtypes = [dp, dp, dp, ctypes.c_double, ctypes.c_long,
                                             ctypes.c_int, ctypes.c_int, dp]
        self.lib.kda_oracle_gate.restype = ctypes.c_int
        self.lib.kda_oracle_l2norm.argtypes = [dp, ctypes.c_long, ctypes.c_int, ctypes.c_double, dp]
        self.lib.kda_oracle_l2norm.restype = ctypes.c_int
        self.lib.kda_oracle_chunk_summaries.argtypes = [dp, dp, dp, dp, dp, ctypes.c_double,
                                                        ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                        ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                        dp, dp, ctypes.c_int]
        self.lib.kda_oracle_chunk_summaries.restype = ctypes.c_int
        self.threads_used = 0

    def gate(self, x, a_log, dt_bias=None, lower_bound=0.0):
        """ln(alpha) from a raw gate x [..., H, K] (Tokamax design doc 9.1.3)."""
        xa = _f64(x)
        H, K = xa.shape[-2], xa.shape[-1]
        rows = xa.size // (H * K)
        al = _f64(a_log).reshape(H)
        db = None if dt_bias is None else _f64(dt_bias).reshape(H * K)
        out = np.empty_like(xa)
        rc = self.lib.kda_oracle_gate(_ptr(xa), _ptr(al), _ptr(db), float(lower_bound), rows, H, K,
                                      _ptr(out))
        if rc < 0:
            raise ValueError("kda_oracle_gate: invalid arguments")
        return out

    def l2norm(self, x, eps=1e-6):
        """x / max(||x||_2, eps) along the last dimension ("KDAChunkwise", F.normalize)."""
        xa = _f64(x)
        D = xa.shape[-1]
        out = np.empty_like(xa)
        rc = self.lib.kda_oracle_l2norm(_ptr(xa), xa.size // D, D, float(eps), _ptr(out))
        if rc < 0:
            raise ValueError("kda_oracle_l2norm: invalid arguments")
        return out

    def _prepare(self, q, k, v, g, beta, initial_state, cu_seqlens):
        q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
        B, T, H, K = q.shape
        V = v.shape[-1]
        if cu_seqlens is not None:
            cu = np.ascontiguousarray(np.asarray(
                cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                dtype=np.int32))
            N = cu.shape[0] - 1
        else:
            cu, N = None, B
        s0 = _f64(initial_state)
        o = np.empty((B, T, H, V), dtype=np.float64)
        fin = np.empty((N, H, K, V), dtype=np.float64)
        return q, k, v, g, beta, s0, cu, N, B, T, H, K, V, o, fin

    def recurrent(self, q, k, v, g, beta, scale, initial_state=None, cu_seqlens=None,
                  num_threads: int = 0):
        """Token recurrence in fp64. Returns (o [B,T,H,V], final_state [N,H,K,V])."""
        q, k, v, g, beta, s0, cu, N, B, T, H, K, V, o, fin = self._prepare(
            q, k, v, g, beta, initial_state, cu_seqlens)
        rc = self.lib.kda_oracle_recurrent(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(s0),
            _ptr(cu, ctypes.c_int32), N, B, T, H, K, V, _ptr(o), _ptr(fin), int(num_threads))
        if rc < 0:
            raise ValueError(f"kda_oracle_recurrent failed with code {rc}")
        self.threads_used = rc
        return o, fin

    def chunkwise(self, q, k, v, g, beta, scale, chunk_size, initial_state=None,
                  cu_seqlens=None, num_threads: int = 0):
        """Chunkwise form in fp64 with any chunk size. Returns (o, final_state)."""
        q, k, v, g, beta, s0, cu, N, B, T, H, K, V, o, fin = self._prepare(
            q, k, v, g, beta, initial_state, cu_seqlens)
        rc = self.lib.kda_oracle_chunkwise(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(s0),
            _ptr(cu, ctypes.c_int32), N, B, T, H, K, V, int(chunk_size), _ptr(o), _ptr(fin),
            int(num_threads))
        if rc < 0:
            raise ValueError(f"kda_oracle_chunkwise failed with code {rc}")
        self.threads_used = rc
        return o, fin

    def chunk_summaries(self, q, k, v, g, beta, scale, chunk_size: int = 64,
                        num_threads: int = 0):
        """Affine summary of every chunk of fixed-length input (Tokamax design doc,
        context-parallel section): chunk j maps its start state S to Phi_j S + Psi_j.
        Returns (phi [B,H,nct,K,K], psi [B,H,nct,K,V]) in fp64."""
        q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
        B, T, H, K = q.shape
        V = v.shape[-1]
        nct = -(-T // chunk_size)
        phi = np.empty((B, H, nct, K, K), dtype=np.float64)
        psi = np.empty((B, H, nct, K, V), dtype=np.float64)
        rc = self.lib.kda_oracle_chunk_summaries(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), B, T, H, K, V,
            int(chunk_size), _ptr(phi), _ptr(psi), int(num_threads))
        if rc < 0:
            raise ValueError(f"kda_oracle_chunk_summaries failed with code {rc}")
        self.threads_used = rc
        return phi, psi


def compose_summaries(phi, psi, lo: int, hi: int):
    """Summary of chunks lo .. hi-1 taken in order, from the per-chunk summaries
    [..., nct, K, K] / [..., nct, K, V]: applying chunk a then chunk b gives
    (Phi_b Phi_a, Phi_b Psi_a + Psi_b) (Tokamax design doc, context-parallel section)."""
    K = phi.shape[-1]
    P = np.broadcast_to(np.eye(K), phi.shape[:-3] + (K, K)).copy()
    Q = np.zeros(psi.shape[:-3] + psi.shape[-2:])
    for j in range(lo, hi):
        P = phi[..., j, :, :] @ P
        Q = phi[..., j, :, :] @ Q + psi[..., j, :, :]
    return P, Q


def segment_start_states(phi, psi, initial_state, segment_chunks: int):
    """Start states of the segments of `segment_chunks` chunks, merged in order from the
    segments' composed summaries: X_0 = S_0, X_{s+1} = Phi_s X_s + Psi_s.  Returns
    [..., n_segments, K, V] and the state after the last segment."""
    nct = phi.shape[-3]
    X = np.zeros(psi.shape[:-3] + psi.shape[-2:]) if initial_state is None else _f64(initial_state).copy()
    starts = []
    for lo in range(0, nct, segment_chunks):
        starts.append(X.copy())
        P, Q = compose_summaries(phi, psi, lo, min(lo + segment_chunks, nct))
        X = P @ X + Q
    return np.stack(starts, axis=-3), X


_DEFAULT: Optional[Oracle] = None


def default_oracle() -> Oracle:
    """The oracle built from the committed source (built on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
