"""Shared comparison helpers for the GPU parity tests.

Tolerance (stated for bf16 inputs and an fp32 state): both tensors are divided by the
oracle's RMS over the whole tensor; the gate is relative L2 error <= 1e-2 and max absolute
error <= 5e-2 of that RMS.  Outputs and final states are judged separately."""
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


def assert_close(name, gpu, ref, rel_tol=REL_L2_TOL, max_tol=MAX_ABS_TOL):
    g = np.asarray(gpu, dtype=np.float64)
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    rel, mx = errors(g, ref)
    log = os.environ.get("KDA_PARITY_LOG")
    if log:
        import json
        test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
        with open(log, "a") as f:
            f.write(json.dumps({"test": test, "name": name, "rel_l2": rel, "max_over_rms": mx,
                                "n": int(g.size)}) + "\n")
    assert rel <= rel_tol and mx <= max_tol, f"{name}: rel_l2={rel:.3e} max/rms={mx:.3e}"
    return rel, mx
