"""GB300-native Kimi Delta Attention (KDA) forward: chunked varlen prefill and decode.

The compute lives in a C-ABI shared library of hand-written sm_103a CUDA kernels
(``csrc/``, declared in ``include/kda.h``).  This package is the thin Python binding over it:
argument marshalling only, every step of the operator runs in the library's kernels.
The library is loaded lazily on first use and its absence is an error, never a fallback.
"""
from . import binding  # noqa: F401
from .binding import (  # noqa: F401
    KdaError,
    bwd,
    decode_step,
    decode_step_prologue,
    decode_window,
    decode_window_prologue,
    fwd_checkpoint_count,
    fwd_chunked,
    fwd_chunked_checkpoints,
    fwd_chunked_host,
    fwd_host_workspace_bytes,
    fwd_chunked_prologue,
    fwd_plan,
    fwd_workspace_bytes,
    launch_count,
    library_path,
    load_library,
    prologue,
    prologue_conv,
    read_device_status,
    selftest_wait_timeout,
)

__all__ = [
    "KdaError", "bwd", "decode_step", "decode_step_prologue", "decode_window", "decode_window_prologue", "fwd_checkpoint_count", "fwd_chunked", "fwd_chunked_checkpoints",
    "fwd_chunked_host", "fwd_host_workspace_bytes", "fwd_chunked_prologue", "fwd_workspace_bytes", "prologue", "prologue_conv",
    "launch_count",
    "library_path", "load_library", "read_device_status", "selftest_wait_timeout",
]
