"""ctypes binding of the KDA C ABI (``include/kda.h``).

Argument marshalling only: shapes and dtypes are checked, missing output buffers are
allocated with torch (PyTorch is the plumbing for device memory and streams), and the call
goes straight to the library.  Every step of the operator runs in the library's kernels.
If the library is missing the calls raise; there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libkda_gb300.so")
_lock = threading.Lock()
_lib = None

KDA_OK = 0
_DTYPES = {torch.bfloat16: 0, torch.float32: 1}
_STATUS = {0: "KDA_OK", -1: "KDA_ERR_INVALID_ARG", -2: "KDA_ERR_UNSUPPORTED",
           -3: "KDA_ERR_WORKSPACE", -4: "KDA_ERR_CUDA", -5: "KDA_ERR_TIMEOUT",
           -6: "KDA_ERR_DECAY_RANGE"}


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {_STATUS.get(int(status), status)}")


class KdaDesc(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("total_tokens", ctypes.c_int64), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("host_seqlens", ctypes.POINTER(ctypes.c_int32))]


class KdaPlanInfo(ctypes.Structure):
    _fields_ = [("chunks", ctypes.c_int64), ("work_items", ctypes.c_int64),
                ("split_sequences", ctypes.c_int32), ("chunk_size", ctypes.c_int32),
                ("segment_chunks", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t)]


class KdaPrologueParams(ctypes.Structure):
    _fields_ = [("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("lower_bound", ctypes.c_float), ("q_scale", ctypes.c_float)]


class KdaConvParams(ctypes.Structure):
    _fields_ = [("w_q", ctypes.c_void_p), ("w_k", ctypes.c_void_p), ("w_v", ctypes.c_void_p),
                ("cache_in", ctypes.c_void_p), ("cache_out", ctypes.c_void_p)]


# exported symbol -> (restype, argtypes)
_P = ctypes.c_void_p
SIGNATURES = {
    "kda_fwd_plan": (ctypes.c_int, [ctypes.POINTER(KdaDesc), ctypes.POINTER(KdaPlanInfo)]),
    "kda_fwd_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(KdaDesc)]),
    "kda_fwd_chunked": (ctypes.c_int, [ctypes.POINTER(KdaDesc), _P, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _P, ctypes.c_size_t, _P]),
    "kda_fwd_chunked_noalloc": (ctypes.c_int, [ctypes.POINTER(KdaDesc), _P, _P, _P, _P, _P, _P,
                                               _P, _P, _P, _P]),
    "kda_fwd_host_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(KdaDesc), ctypes.c_int32]),
    "kda_fwd_chunked_host": (ctypes.c_int, [ctypes.POINTER(KdaDesc), _P, _P, _P, _P, _P, _P, _P,
                                            _P, ctypes.c_int32, _P, ctypes.c_size_t, _P]),
    "kda_fwd_checkpoint_count": (ctypes.c_int64, [ctypes.POINTER(KdaDesc), ctypes.c_int32]),
    "kda_fwd_chunked_ckpt": (ctypes.c_int, [ctypes.POINTER(KdaDesc), _P, _P, _P, _P, _P, _P, _P,
                                            _P, _P, ctypes.c_int32, _P, _P, ctypes.c_size_t, _P]),
    "kda_prologue": (ctypes.c_int, [ctypes.POINTER(KdaDesc), ctypes.POINTER(KdaPrologueParams),
                                    _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "kda_fwd_chunked_prologue": (ctypes.c_int, [ctypes.POINTER(KdaDesc),
                                                ctypes.POINTER(KdaPrologueParams), _P, _P, _P,
                                                _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "kda_prologue_conv": (ctypes.c_int, [ctypes.POINTER(KdaDesc),
                                         ctypes.POINTER(KdaPrologueParams),
                                         ctypes.POINTER(KdaConvParams), _P, _P, _P, _P, _P, _P,
                                         _P, _P, _P, _P, _P, _P]),
    "kda_decode_step": (ctypes.c_int, [ctypes.POINTER(KdaDesc), _P, _P, _P, _P, _P, _P, _P, _P]),
    "kda_decode_step_prologue": (ctypes.c_int, [ctypes.POINTER(KdaDesc),
                                                ctypes.POINTER(KdaPrologueParams), _P, _P, _P,
                                                _P, _P, _P, _P, _P]),
    "kda_decode_window_prologue": (ctypes.c_int, [ctypes.POINTER(KdaDesc),
                                                  ctypes.POINTER(KdaPrologueParams), _P, _P, _P,
                                                  _P, _P, _P, _P, _P, _P, _P]),
    "kda_decode_window": (ctypes.c_int, [ctypes.POINTER(KdaDesc), _P, _P, _P, _P, _P, _P, _P, _P,
                                         _P, _P]),
    "kda_read_device_status": (ctypes.c_int, [_P]),
    "kda_selftest_wait_timeout": (ctypes.c_int, [_P]),
    "kda_bwd_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(KdaDesc)]),
    "kda_bwd": (ctypes.c_int, [ctypes.POINTER(KdaDesc), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                               _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "kda_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kda_launch_count": (ctypes.c_uint64, []),
    "kda_version": (ctypes.c_int32, []),
}


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load ``libkda_gb300.so`` (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"KDA CUDA library not built ({_LIB_PATH} missing); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def make_desc(seqlens, num_heads: int, dtype: torch.dtype, d: int = 128):
    lens = (ctypes.c_int32 * len(seqlens))(*[int(x) for x in seqlens])
    desc = KdaDesc(len(seqlens), int(num_heads), int(sum(int(x) for x in seqlens)), d, d,
                   _DTYPES.get(dtype, 99), 0, lens)
    desc._lens = lens  # keep the host array alive with the struct
    return desc


def fwd_plan(seqlens, num_heads: int, dtype: torch.dtype = torch.bfloat16) -> dict:
    lib = load_library()
    info = KdaPlanInfo()
    st = lib.kda_fwd_plan(ctypes.byref(make_desc(seqlens, num_heads, dtype)), ctypes.byref(info))
    if st != KDA_OK:
        raise KdaError(st, "kda_fwd_plan")
    return {f: getattr(info, f) for f, _ in KdaPlanInfo._fields_ if f != "reserved"}


def fwd_workspace_bytes(seqlens, num_heads: int, dtype: torch.dtype = torch.bfloat16) -> int:
    lib = load_library()
    return int(lib.kda_fwd_workspace_bytes(ctypes.byref(make_desc(seqlens, num_heads, dtype))))


def _check_io(name, t, shape, dtype, device):
    if t.device != device or t.dtype != dtype or tuple(t.shape) != tuple(shape) \
            or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)} on {device}, got "
                         f"{t.dtype} {tuple(t.shape)} on {t.device}")


def fwd_chunked(q, k, v, log_alpha, beta, cu_seqlens, seqlens, init_state=None, out=None,
                final_state=None, want_final_state: bool = True, workspace=None, stream=None):
    """Chunked KDA prefill.  q, k, log_alpha, v: [T, H, 128]; beta: [T, H]; cu_seqlens: int32
    [N+1] on the device; seqlens: the same lengths on the host.  Returns (out, final_state)."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("fwd_chunked needs CUDA tensors")
    T, H, d = q.shape
    N = len(seqlens)
    dt = q.dtype
    for name, t, shp in (("k", k, (T, H, d)), ("v", v, (T, H, d)),
                         ("log_alpha", log_alpha, (T, H, d)), ("beta", beta, (T, H))):
        _check_io(name, t, shp, dt, dev)
    _check_io("cu_seqlens", cu_seqlens, (N + 1,), torch.int32, dev)
    if init_state is not None:
        _check_io("init_state", init_state, (N, H, d, d), torch.float32, dev)
    if out is None:
        out = torch.empty((T, H, d), dtype=dt, device=dev)
    _check_io("out", out, (T, H, d), dt, dev)
    if final_state is None and want_final_state:
        final_state = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    if final_state is not None:
        _check_io("final_state", final_state, (N, H, d, d), torch.float32, dev)
    desc = make_desc(seqlens, H, dt, d)
    need = int(lib.kda_fwd_workspace_bytes(ctypes.byref(desc)))
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.kda_fwd_chunked(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                             _ptr(beta), _ptr(init_state), _ptr(cu_seqlens), _ptr(out),
                             _ptr(final_state), _ptr(workspace), ws_bytes,
                             _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_fwd_chunked")
    return out, final_state


def _prologue_params(A_log, dt_bias, lower_bound, q_scale, H, d, dev):
    _check_io("A_log", A_log, (H,), torch.float32, dev)
    if dt_bias is not None:
        _check_io("dt_bias", dt_bias, (H, d), torch.float32, dev)
    return KdaPrologueParams(A_log.data_ptr(), None if dt_bias is None else dt_bias.data_ptr(),
                             float(lower_bound), float(q_scale))


def prologue(q_raw, k_raw, v_raw, g_raw, beta_logit, A_log, dt_bias=None,
             lower_bound: float = -5.0, q_scale: float = 128 ** -0.5, stream=None):
    """The input prologue alone: raw bf16 projections q_raw, k_raw, g_raw, v_raw [T, H, 128] and
    beta_logit [T, H] -> (q, k, v, log_alpha, beta), bf16.  A_log: fp32 [H]; dt_bias: fp32
    [H, 128] or None."""
    lib = load_library()
    dev = q_raw.device
    if dev.type != "cuda":
        raise ValueError("prologue needs CUDA tensors")
    T, H, d = q_raw.shape
    dt = q_raw.dtype
    for name, t, shp in (("k_raw", k_raw, (T, H, d)), ("v_raw", v_raw, (T, H, d)),
                         ("g_raw", g_raw, (T, H, d)), ("beta_logit", beta_logit, (T, H))):
        _check_io(name, t, shp, dt, dev)
    prm = _prologue_params(A_log, dt_bias, lower_bound, q_scale, H, d, dev)
    outs = [torch.empty((T, H, d), dtype=dt, device=dev) for _ in range(4)]
    beta = torch.empty((T, H), dtype=dt, device=dev)
    desc = make_desc([T], H, dt, d)
    st = lib.kda_prologue(ctypes.byref(desc), ctypes.byref(prm), _ptr(q_raw), _ptr(k_raw),
                          _ptr(v_raw), _ptr(g_raw), _ptr(beta_logit), _ptr(outs[0]),
                          _ptr(outs[1]), _ptr(outs[2]), _ptr(outs[3]), _ptr(beta),
                          _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_prologue")
    return outs[0], outs[1], outs[2], outs[3], beta


def fwd_chunked_prologue(q_raw, k_raw, v_raw, g_raw, beta_logit, cu_seqlens, seqlens, A_log,
                         dt_bias=None, lower_bound: float = -5.0, q_scale: float = 128 ** -0.5,
                         init_state=None, out=None, final_state=None,
                         want_final_state: bool = True, workspace=None, stream=None):
    """Chunked KDA prefill on raw projections, the prologue fused into the kernel (arguments
    as ``prologue`` and ``fwd_chunked``).  Returns (out, final_state)."""
    lib = load_library()
    dev = q_raw.device
    if dev.type != "cuda":
        raise ValueError("fwd_chunked_prologue needs CUDA tensors")
    T, H, d = q_raw.shape
    N = len(seqlens)
    dt = q_raw.dtype
    for name, t, shp in (("k_raw", k_raw, (T, H, d)), ("v_raw", v_raw, (T, H, d)),
                         ("g_raw", g_raw, (T, H, d)), ("beta_logit", beta_logit, (T, H))):
        _check_io(name, t, shp, dt, dev)
    _check_io("cu_seqlens", cu_seqlens, (N + 1,), torch.int32, dev)
    prm = _prologue_params(A_log, dt_bias, lower_bound, q_scale, H, d, dev)
    if init_state is not None:
        _check_io("init_state", init_state, (N, H, d, d), torch.float32, dev)
    if out is None:
        out = torch.empty((T, H, d), dtype=dt, device=dev)
    _check_io("out", out, (T, H, d), dt, dev)
    if final_state is None and want_final_state:
        final_state = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    if final_state is not None:
        _check_io("final_state", final_state, (N, H, d, d), torch.float32, dev)
    desc = make_desc(seqlens, H, dt, d)
    need = int(lib.kda_fwd_workspace_bytes(ctypes.byref(desc)))
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.kda_fwd_chunked_prologue(ctypes.byref(desc), ctypes.byref(prm), _ptr(q_raw),
                                      _ptr(k_raw), _ptr(v_raw), _ptr(g_raw), _ptr(beta_logit),
                                      _ptr(init_state), _ptr(cu_seqlens), _ptr(out),
                                      _ptr(final_state), _ptr(workspace), ws_bytes,
                                      _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_fwd_chunked_prologue")
    return out, final_state


def fwd_checkpoint_count(seqlens, num_heads: int, ckpt_every: int,
                         dtype: torch.dtype = torch.bfloat16) -> int:
    """Number of states fwd_chunked_checkpoints writes: sum of L_n // ckpt_every (ckpt_every a
    positive multiple of 64)."""
    lib = load_library()
    desc = make_desc(seqlens, num_heads, dtype)
    n = int(lib.kda_fwd_checkpoint_count(ctypes.byref(desc), int(ckpt_every)))
    if n < 0:
        raise KdaError(-1, "kda_fwd_checkpoint_count")
    return n


def fwd_chunked_checkpoints(q, k, v, log_alpha, beta, cu_seqlens, seqlens, ckpt_every: int,
                            init_state=None, out=None, final_state=None, checkpoints=None,
                            workspace=None, stream=None):
    """fwd_chunked that also returns the fp32 state after every ``ckpt_every`` tokens of each
    sequence (positions ckpt_every, 2 ckpt_every, ... <= L_n), as ``checkpoints`` of shape
    [count, H, 128, 128]: sequence by sequence, positions in increasing order.  Outputs and
    final states are bit-identical to fwd_chunked.  Returns (out, final_state, checkpoints)."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("fwd_chunked_checkpoints needs CUDA tensors")
    T, H, d = q.shape
    N = len(seqlens)
    dt = q.dtype
    for name, t, shp in (("k", k, (T, H, d)), ("v", v, (T, H, d)),
                         ("log_alpha", log_alpha, (T, H, d)), ("beta", beta, (T, H))):
        _check_io(name, t, shp, dt, dev)
    _check_io("cu_seqlens", cu_seqlens, (N + 1,), torch.int32, dev)
    if init_state is not None:
        _check_io("init_state", init_state, (N, H, d, d), torch.float32, dev)
    if out is None:
        out = torch.empty((T, H, d), dtype=dt, device=dev)
    _check_io("out", out, (T, H, d), dt, dev)
    if final_state is None:
        final_state = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    _check_io("final_state", final_state, (N, H, d, d), torch.float32, dev)
    count = fwd_checkpoint_count(seqlens, H, ckpt_every, dt)
    if checkpoints is None:
        checkpoints = torch.empty((count, H, d, d), dtype=torch.float32, device=dev)
    _check_io("checkpoints", checkpoints, (count, H, d, d), torch.float32, dev)
    desc = make_desc(seqlens, H, dt, d)
    need = int(lib.kda_fwd_workspace_bytes(ctypes.byref(desc)))
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.kda_fwd_chunked_ckpt(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                  _ptr(beta), _ptr(init_state), _ptr(cu_seqlens), _ptr(out),
                                  _ptr(final_state), int(ckpt_every),
                                  _ptr(checkpoints) if count else None, _ptr(workspace), ws_bytes,
                                  _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_fwd_chunked_ckpt")
    return out, final_state, checkpoints


def fwd_chunked_noalloc(q, k, v, log_alpha, beta, cu_seqlens, seqlens, init_state=None,
                        out=None, final_state=None, stream=None):
    """Chunked prefill through kda_fwd_chunked_noalloc: for callers that cannot allocate
    device scratch, the library's built-in 48 MiB array serves as the segment workspace (a
    call needing more raises KdaError(KDA_ERR_WORKSPACE)).  ``out`` must be given, as this path
    allocates nothing; ``final_state`` may be None to skip the final states.  Calls share the
    array, so overlapping calls on different streams must not be issued."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("fwd_chunked_noalloc needs CUDA tensors")
    T, H, d = q.shape
    N = len(seqlens)
    dt = q.dtype
    for name, t, shp in (("k", k, (T, H, d)), ("v", v, (T, H, d)),
                         ("log_alpha", log_alpha, (T, H, d)), ("beta", beta, (T, H)),
                         ("out", out, (T, H, d))):
        if t is None:
            raise ValueError(f"{name} must be given")
        _check_io(name, t, shp, dt, dev)
    _check_io("cu_seqlens", cu_seqlens, (N + 1,), torch.int32, dev)
    if init_state is not None:
        _check_io("init_state", init_state, (N, H, d, d), torch.float32, dev)
    if final_state is not None:
        _check_io("final_state", final_state, (N, H, d, d), torch.float32, dev)
    desc = make_desc(seqlens, H, dt, d)
    st = lib.kda_fwd_chunked_noalloc(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(log_alpha), _ptr(beta), _ptr(init_state),
                                     _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                     _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_fwd_chunked_noalloc")
    return out, final_state


def fwd_host_workspace_bytes(seqlens, num_heads: int, dtype: torch.dtype = torch.bfloat16,
                             parts: int = 0) -> int:
    lib = load_library()
    return int(lib.kda_fwd_host_workspace_bytes(ctypes.byref(make_desc(seqlens, num_heads, dtype)),
                                                int(parts)))


def fwd_chunked_host(q, k, v, log_alpha, beta, seqlens, init_state=None, out=None,
                     final_state=None, parts: int = 0, workspace=None, device=None):
    """Chunked prefill on HOST tensors (pinned memory for overlap): ``kda_fwd_chunked_host``.

    Same arguments and results as ``fwd_chunked`` except that every tensor lives on the host
    (cu_seqlens is derived from ``seqlens``).  The library cuts the tokens into ``parts``
    token-range parts (0: its default) and overlaps the upload of one part, the kernels of the
    previous one and the download of the one before; a sequence cut by a part boundary resumes
    from its fp32 state, so it agrees with ``fwd_chunked`` within rounding (bit for bit when it
    lies inside the first part).  ``workspace`` (optional): a uint8 device tensor of at least
    ``fwd_host_workspace_bytes(seqlens, H, dtype, parts)`` bytes.  The call returns when ``out``
    and ``final_state`` hold the results."""
    lib = load_library()
    dev = torch.device(device if device is not None else "cuda")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    T, H, d = q.shape
    N = len(seqlens)
    dt = q.dtype
    cpu = torch.device("cpu")
    for name, t, shp in (("q", q, (T, H, d)), ("k", k, (T, H, d)), ("v", v, (T, H, d)),
                         ("log_alpha", log_alpha, (T, H, d)), ("beta", beta, (T, H))):
        _check_io(name, t, shp, dt, cpu)
    if init_state is not None:
        _check_io("init_state", init_state, (N, H, d, d), torch.float32, cpu)
    if out is None:
        out = torch.empty((T, H, d), dtype=dt).pin_memory()
    _check_io("out", out, (T, H, d), dt, cpu)
    if final_state is None:
        final_state = torch.empty((N, H, d, d), dtype=torch.float32).pin_memory()
    _check_io("final_state", final_state, (N, H, d, d), torch.float32, cpu)
    desc = make_desc(seqlens, H, dt)
    need = int(lib.kda_fwd_host_workspace_bytes(ctypes.byref(desc), int(parts)))
    if need == 0:
        raise KdaError(-1, "kda_fwd_host_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    st = lib.kda_fwd_chunked_host(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                                  _ptr(beta), _ptr(init_state), _ptr(out), _ptr(final_state),
                                  int(parts), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(),
                                  _stream_handle(None, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_fwd_chunked_host")
    return out, final_state


def decode_step(q, k, v, log_alpha, beta, state, out=None, stream=None):
    """One decode token per (sequence, head); ``state`` [N, H, 128, 128] fp32 is updated in
    place.  q, k, log_alpha, v: [N, H, 128]; beta: [N, H].  Returns out [N, H, 128]."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("decode_step needs CUDA tensors")
    N, H, d = q.shape
    dt = q.dtype
    for name, t, shp in (("k", k, (N, H, d)), ("v", v, (N, H, d)),
                         ("log_alpha", log_alpha, (N, H, d)), ("beta", beta, (N, H))):
        _check_io(name, t, shp, dt, dev)
    _check_io("state", state, (N, H, d, d), torch.float32, dev)
    if out is None:
        out = torch.empty((N, H, d), dtype=dt, device=dev)
    _check_io("out", out, (N, H, d), dt, dev)
    desc = KdaDesc(N, H, N, d, d, _DTYPES.get(dt, 99), 0, None)
    st = lib.kda_decode_step(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                             _ptr(beta), _ptr(state), _ptr(out), _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_step")
    return out


def decode_window(q, k, v, log_alpha, beta, cu_seqlens, seqlens, state, commit=None, out=None,
                  want_out: bool = True, stream=None):
    """A run of decode tokens per sequence in one pass over the state (speculative decoding:
    replayed accepted tokens, the bonus token and the next draft window).  q, k, log_alpha, v:
    [T, H, 128]; beta: [T, H]; cu_seqlens: int32 [N+1] on the device, seqlens the same run
    lengths (0..64) on the host; state [N, H, 128, 128] fp32.  Every token's output is
    returned; the state after the first commit[n] tokens of run n is written back into
    ``state`` (commit: int32 [N] on the device, or None to commit every token)."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("decode_window needs CUDA tensors")
    T, H, d = q.shape
    N = len(seqlens)
    dt = q.dtype
    for name, t, shp in (("k", k, (T, H, d)), ("v", v, (T, H, d)),
                         ("log_alpha", log_alpha, (T, H, d)), ("beta", beta, (T, H))):
        _check_io(name, t, shp, dt, dev)
    _check_io("cu_seqlens", cu_seqlens, (N + 1,), torch.int32, dev)
    _check_io("state", state, (N, H, d, d), torch.float32, dev)
    if commit is not None:
        _check_io("commit", commit, (N,), torch.int32, dev)
    if out is None and want_out:
        out = torch.empty((T, H, d), dtype=dt, device=dev)
    if out is not None:
        _check_io("out", out, (T, H, d), dt, dev)
    desc = make_desc(seqlens, H, dt, d)
    st = lib.kda_decode_window(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                               _ptr(beta), _ptr(cu_seqlens), _ptr(state), _ptr(out), _ptr(commit),
                               _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_window")
    return out


def read_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the sticky device status code."""
    lib = load_library()
    s = None if stream is None else ctypes.c_void_p(stream.cuda_stream)
    if s is None and torch.cuda.is_available():
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return int(lib.kda_read_device_status(s))


def launch_count() -> int:
    return int(load_library().kda_launch_count())


def decode_step_prologue(q_raw, k_raw, v_raw, g_raw, beta_logit, state, A_log, dt_bias=None,
                         lower_bound: float = -5.0, q_scale: float = 128 ** -0.5, out=None,
                         stream=None):
    """``decode_step`` on raw projections, the input prologue fused into the kernel (arguments
    as ``decode_step`` and ``prologue``).  Returns out [N, H, 128]."""
    lib = load_library()
    dev = q_raw.device
    if dev.type != "cuda":
        raise ValueError("decode_step_prologue needs CUDA tensors")
    N, H, d = q_raw.shape
    dt = q_raw.dtype
    for name, t, shp in (("k_raw", k_raw, (N, H, d)), ("v_raw", v_raw, (N, H, d)),
                         ("g_raw", g_raw, (N, H, d)), ("beta_logit", beta_logit, (N, H))):
        _check_io(name, t, shp, dt, dev)
    _check_io("state", state, (N, H, d, d), torch.float32, dev)
    prm = _prologue_params(A_log, dt_bias, lower_bound, q_scale, H, d, dev)
    if out is None:
        out = torch.empty((N, H, d), dtype=dt, device=dev)
    _check_io("out", out, (N, H, d), dt, dev)
    desc = make_desc([1] * N, H, dt, d)
    st = lib.kda_decode_step_prologue(ctypes.byref(desc), ctypes.byref(prm), _ptr(q_raw),
                                      _ptr(k_raw), _ptr(v_raw), _ptr(g_raw), _ptr(beta_logit),
                                      _ptr(state), _ptr(out), _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_step_prologue")
    return out


def decode_window_prologue(q_raw, k_raw, v_raw, g_raw, beta_logit, cu_seqlens, seqlens, state,
                           A_log, dt_bias=None, lower_bound: float = -5.0,
                           q_scale: float = 128 ** -0.5, commit=None, out=None,
                           want_out: bool = True, stream=None):
    """``decode_window`` on raw projections, the input prologue fused into the kernel
    (arguments as ``decode_window`` and ``prologue``)."""
    lib = load_library()
    dev = q_raw.device
    if dev.type != "cuda":
        raise ValueError("decode_window_prologue needs CUDA tensors")
    T, H, d = q_raw.shape
    N = len(seqlens)
    dt = q_raw.dtype
    for name, t, shp in (("k_raw", k_raw, (T, H, d)), ("v_raw", v_raw, (T, H, d)),
                         ("g_raw", g_raw, (T, H, d)), ("beta_logit", beta_logit, (T, H))):
        _check_io(name, t, shp, dt, dev)
    _check_io("cu_seqlens", cu_seqlens, (N + 1,), torch.int32, dev)
    _check_io("state", state, (N, H, d, d), torch.float32, dev)
    if commit is not None:
        _check_io("commit", commit, (N,), torch.int32, dev)
    prm = _prologue_params(A_log, dt_bias, lower_bound, q_scale, H, d, dev)
    if out is None and want_out:
        out = torch.empty((T, H, d), dtype=dt, device=dev)
    if out is not None:
        _check_io("out", out, (T, H, d), dt, dev)
    desc = make_desc(seqlens, H, dt, d)
    st = lib.kda_decode_window_prologue(ctypes.byref(desc), ctypes.byref(prm), _ptr(q_raw),
                                        _ptr(k_raw), _ptr(v_raw), _ptr(g_raw), _ptr(beta_logit),
                                        _ptr(cu_seqlens), _ptr(state), _ptr(out), _ptr(commit),
                                        _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_window_prologue")
    return out


def prologue_conv(q_raw, k_raw, v_raw, g_raw, beta_logit, cu_seqlens, seqlens, A_log, w_q, w_k,
                  w_v, dt_bias=None, cache_in=None, cache_out=None, lower_bound: float = -5.0,
                  q_scale: float = 128 ** -0.5, stream=None):
    """The short convolution (kernel 4) of q_raw, k_raw, v_raw, then the input prologue.
    w_q, w_k, w_v: fp32 [H, 128, 4]; cache_in / cache_out: bf16 [N, 3, 3, H, 128] or None
    (cache_out may be cache_in).  Returns (q, k, v, log_alpha, beta), bf16."""
    lib = load_library()
    dev = q_raw.device
    if dev.type != "cuda":
        raise ValueError("prologue_conv needs CUDA tensors")
    T, H, d = q_raw.shape
    N = len(seqlens)
    dt = q_raw.dtype
    for name, t, shp in (("k_raw", k_raw, (T, H, d)), ("v_raw", v_raw, (T, H, d)),
                         ("g_raw", g_raw, (T, H, d)), ("beta_logit", beta_logit, (T, H))):
        _check_io(name, t, shp, dt, dev)
    _check_io("cu_seqlens", cu_seqlens, (N + 1,), torch.int32, dev)
    for name, w in (("w_q", w_q), ("w_k", w_k), ("w_v", w_v)):
        _check_io(name, w, (H, d, 4), torch.float32, dev)
    for name, c in (("cache_in", cache_in), ("cache_out", cache_out)):
        if c is not None:
            _check_io(name, c, (N, 3, 3, H, d), dt, dev)
    prm = _prologue_params(A_log, dt_bias, lower_bound, q_scale, H, d, dev)
    conv = KdaConvParams(w_q.data_ptr(), w_k.data_ptr(), w_v.data_ptr(),
                         None if cache_in is None else cache_in.data_ptr(),
                         None if cache_out is None else cache_out.data_ptr())
    outs = [torch.empty((T, H, d), dtype=dt, device=dev) for _ in range(4)]
    beta = torch.empty((T, H), dtype=dt, device=dev)
    desc = make_desc(seqlens, H, dt, d)
    st = lib.kda_prologue_conv(ctypes.byref(desc), ctypes.byref(prm), ctypes.byref(conv),
                               _ptr(cu_seqlens), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw),
                               _ptr(g_raw), _ptr(beta_logit), _ptr(outs[0]), _ptr(outs[1]),
                               _ptr(outs[2]), _ptr(outs[3]), _ptr(beta),
                               _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_prologue_conv")
    return outs[0], outs[1], outs[2], outs[3], beta


def selftest_wait_timeout(stream=None, device=None) -> int:
    """Launch the bounded-wait self-test (one CTA whose wait runs out after about 2 s) and
    return the device status it leaves (KDA_ERR_TIMEOUT, -5, when the bound works)."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    h = _stream_handle(stream, dev)
    st = lib.kda_selftest_wait_timeout(h)
    if st != KDA_OK:
        raise KdaError(st, "kda_selftest_wait_timeout")
    return int(lib.kda_read_device_status(h))


def bwd(q, k, v, log_alpha, beta, cu_seqlens, seqlens, d_out, init_state=None, d_state=None,
        workspace=None, stream=None):
    """Gradients of the recurrence: given d_out (fp32 [T, H, 128], the gradient of a loss with
    respect to the outputs) and optionally d_state (fp32 [N, H, 128, 128], with respect to the
    final states), returns (dq, dk, dv, dlog_alpha, dbeta, dinit_state), fp32."""
    lib = load_library()
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("bwd needs CUDA tensors")
    T, H, d = q.shape
    N = len(seqlens)
    dt = q.dtype
    for name, t, shp in (("k", k, (T, H, d)), ("v", v, (T, H, d)),
                         ("log_alpha", log_alpha, (T, H, d)), ("beta", beta, (T, H))):
        _check_io(name, t, shp, dt, dev)
    _check_io("cu_seqlens", cu_seqlens, (N + 1,), torch.int32, dev)
    _check_io("d_out", d_out, (T, H, d), torch.float32, dev)
    for name, t in (("init_state", init_state), ("d_state", d_state)):
        if t is not None:
            _check_io(name, t, (N, H, d, d), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dk, dv, dg = (torch.empty((T, H, d), **f32) for _ in range(4))
    dbeta = torch.empty((T, H), **f32)
    dinit = torch.empty((N, H, d, d), **f32)
    desc = make_desc(seqlens, H, dt, d)
    need = int(lib.kda_bwd_workspace_bytes(ctypes.byref(desc)))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = lib.kda_bwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                     _ptr(init_state), _ptr(cu_seqlens), _ptr(d_out), _ptr(d_state), _ptr(dq),
                     _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dinit), _ptr(workspace),
                     workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_bwd")
    return dq, dk, dv, dg, dbeta, dinit
