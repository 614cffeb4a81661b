"""Shared comparison helpers for the GPU parity tests.

Tolerance (stated for bf16 inputs and an fp32 state): both tensors are divided by the
oracle's RMS over the whole tensor; the gate is relative L2 error <= 1e-2 and max absolute
error <= 5e-2 of that RMS.  Outputs and final states are assessed separately.

Outputs stored as bf16 (the operator returns o in its input dtype): each element's own storage
rounding, half a bf16 unit in the last place of the larger of |gpu| and |ref|, is not counted
against the max-abs term (the relative L2 term counts everything).  The gate bounds the
computation; bf16 storage alone moves an element by up to 2^-9 of its magnitude, which exceeds
5e-2 of the RMS wherever an output is more than 25.6 times the RMS, as happens under fast decay.
Both figures are logged."""
from __future__ import annotations

import os

import numpy as np

REL_L2_TOL = 1e-2
MAX_ABS_TOL = 5e-2


def oracle_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def errors(gpu, ref):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    rms = float(np.sqrt(np.mean(r * r)))
    if rms == 0.0:
        rms = 1.0
    denom = float(np.linalg.norm(r)) or 1.0
    return float(np.linalg.norm(g - r) / denom), float(np.abs(g - r).max() / rms)


def bf16_half_ulp(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits): 2^(floor(log2|x|) - 8)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def _as_array(x):
    """(float64 array, whether x is a bf16 tensor)."""
    try:
        import torch
        if torch.is_tensor(x):
            return x.detach().double().cpu().numpy(), x.dtype == torch.bfloat16
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64), False


def assert_close(name, gpu, ref, rel_tol=REL_L2_TOL, max_tol=MAX_ABS_TOL):
    """gpu: a numpy array or a torch tensor (a bf16 tensor gets the storage allowance)."""
    g, stored_bf16 = _as_array(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    rel, mx = errors(g, r)
    mx_gate = mx
    if stored_bf16:
        rms = float(np.sqrt(np.mean(r * r))) or 1.0
        excess = np.abs(g - r) - bf16_half_ulp(np.maximum(np.abs(g), np.abs(r)))
        mx_gate = float(max(excess.max(), 0.0) / rms)
    log = os.environ.get("KDA_PARITY_LOG")
    if log:
        import json
        test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
        with open(log, "a") as f:
            f.write(json.dumps({"test": test, "name": name, "rel_l2": rel, "max_over_rms": mx,
                                "max_over_rms_beyond_storage": mx_gate, "n": int(g.size)}) + "\n")
    assert rel <= rel_tol and mx_gate <= max_tol, \
        f"{name}: rel_l2={rel:.3e} max/rms={mx:.3e} (beyond bf16 storage {mx_gate:.3e})"
    return rel, mx
