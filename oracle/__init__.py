"""fp64 CPU oracle for the Kimi Delta Attention forward recurrence.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The CUDA library never calls it and shares no
code with it; it is the slow, obviously-correct definition the kernels are checked against.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, OpenMP over (sequence, head) units):
the token loop forget / erase-and-write / read of flash-linear-attention's ``naive.py`` as
shown on "How Kimi K3 Engineered Its Way to the Frontier", section "How KDA updates its
state".  This module only builds the shared object with gcc and marshals arrays to it.

The input prologue (raw projections -> q, k, v, g, beta) is plain numpy fp64 in
``input_prologue.py``, exported here as ``prologue``.

The gradients of the recurrence (``recurrence_backward``) come from reverse-mode automatic
differentiation of the same token loop written in torch float64 (``backward.py``).

Every function here is pinned by ``tests/test_oracle_pins.py``, ``tests/test_oracle_prologue.py``
and ``tests/test_oracle_backward.py``; there is no unpinned entry.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .input_prologue import prologue  # noqa: F401  (re-exported)
from .backward import recurrence_backward  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

F64, F32, BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE fp64, no fused multiply-add contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def load_variant(path: str):
    """Load another build of the same C source (used by the planted-mistake tests)."""
    lib = ctypes.CDLL(path)
    _declare(lib)
    return lib


def _declare(lib):
    lib.kda_oracle_recurrence.restype = ctypes.c_int
    lib.kda_oracle_recurrence.argtypes = [
        ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_int32,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            _declare(lib)
            _lib = lib
    return _lib


def _as_host_array(x):
    """Return (contiguous numpy array, format code) for a torch tensor or numpy array.

    bf16 tensors are passed as their raw 16-bit patterns; the C side widens them exactly."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float32:
                return x.numpy(), F32
            if x.dtype == torch.float64:
                return x.numpy(), F64
            raise TypeError(f"oracle: unsupported dtype {x.dtype}")
    except ImportError:  # pragma: no cover - torch is always present in this project
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.float32:
        return x, F32
    raise TypeError(f"oracle: unsupported dtype {x.dtype}")


def recurrence(q, k, v, g, beta, cu_seqlens, state_in=None, windows=None,
               want_out: bool = True, want_state: bool = True, threads: int = 0, lib=None):
    """Run the KDA token loop for every (sequence, head) unit of a packed batch.

    q, k, g: [T_tot, H, d_k]; v: [T_tot, H, d_v]; beta: [T_tot, H] — all the same dtype
    (float64, float32 or bfloat16).  cu_seqlens: [N+1] int.  state_in: [N, H, d_k, d_v]
    (any float dtype, widened to fp64) or None for zeros.  windows: list of (lo, hi) global
    token ranges whose outputs are recorded (None: every token).

    Returns (out [rows, H, d_v] float64 or None, state_out [N, H, d_k, d_v] float64 or None).
    """
    lib = _load() if lib is None else lib
    arrs = [_as_host_array(x) for x in (q, k, v, g, beta)]
    fmts = {f for _, f in arrs}
    if len(fmts) != 1:
        raise TypeError("oracle: q, k, v, g, beta must share one dtype")
    fmt = fmts.pop()
    (qa, _), (ka, _), (va, _), (ga, _), (ba, _) = arrs
    T, H, dk = qa.shape
    dv = va.shape[-1]
    if ka.shape != (T, H, dk) or ga.shape != (T, H, dk) or va.shape != (T, H, dv) \
            or ba.shape != (T, H):
        raise ValueError("oracle: inconsistent shapes")
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    if int(cu[-1]) != T:
        raise ValueError("oracle: cu_seqlens[-1] != T_tot")
    s_in = None
    if state_in is not None:
        s_in = state_in
        if hasattr(s_in, "cpu"):
            s_in = s_in.detach().cpu().double().numpy()
        s_in = np.ascontiguousarray(s_in, dtype=np.float64)
        if s_in.shape != (N, H, dk, dv):
            raise ValueError("oracle: state_in shape")
    win = None
    rows = T
    if windows is not None:
        win = np.ascontiguousarray(np.asarray(windows, dtype=np.int64).reshape(-1, 2))
        rows = int(sum(hi - lo for lo, hi in win))
    out = np.zeros((rows, H, dv), dtype=np.float64) if want_out else None
    s_out = np.zeros((N, H, dk, dv), dtype=np.float64) if want_state else None

    def p(a):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    rc = lib.kda_oracle_recurrence(
        T, N, H, dk, dv, p(cu), fmt, p(qa), p(ka), p(va), p(ga), p(ba), p(s_in), p(out),
        0 if win is None else int(win.shape[0]), p(win), p(s_out), int(threads))
    if rc != 0:
        raise ValueError(f"oracle: kda_oracle_recurrence returned {rc}")
    return out, s_out


def decode_step(q, k, v, g, beta, state, threads: int = 0):
    """One decode token per (sequence, head): the recurrence with every sequence of length 1.

    q, k, g: [N, H, d_k]; v: [N, H, d_v]; beta: [N, H]; state: [N, H, d_k, d_v].
    Returns (out [N, H, d_v], new state [N, H, d_k, d_v]) in float64."""
    n = (q.shape[0])
    cu = np.arange(n + 1, dtype=np.int32)
    return recurrence(q, k, v, g, beta, cu, state_in=state, threads=threads)
