"""fp64 oracle of the KDA input prologue: raw per-token projections -> (q, k, v, g, beta).

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``): only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may use it.  Plain numpy in
float64, one formula per line, no blocking or reordering.

What it follows:
- the decay gate with a lower bound, g = lower_bound * sigmoid(exp(A_log[h]) * (g_raw + dt_bias)),
  which keeps every g inside (lower_bound, 0) ("How Kimi K3 Engineered Its Way to the Frontier",
  section "How KDA updates its state", the paragraph on K3's replacement of the softplus gate);
- queries and keys pass through Swish and are then L2-normalised over the 128 channels; values
  pass through Swish ("Kimi K3: a 2.8T open model that turns compute into intelligence 2.5x
  better", section "Kimi Delta Attention: constant-size memory over a million tokens").  The
  short convolution that precedes Swish there is the caller's: the raw inputs here are its
  outputs;
- beta arrives as logits and passes through a sigmoid (same page, section "FlashKDA: the
  equation, shipped as a kernel").

Readings where the pages are silent: the L2 norm divides by sqrt(sum of squares + eps) with
eps = 1e-6 (a zero row stays zero); q is multiplied by ``q_scale`` after normalisation (the
pages apply no scale; callers pass 1/sqrt(128) for the usual attention scaling).

Exported as ``oracle.prologue``.  Pinned by ``tests/test_oracle_prologue.py`` (closed forms, symmetries and invariants).
"""
from __future__ import annotations

import numpy as np

L2_EPS = 1e-6


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def sigmoid(x):
    """1 / (1 + e^{-x}), elementwise, fp64."""
    x = _f64(x)
    return 1.0 / (1.0 + np.exp(-x))


def swish(x):
    """x * sigmoid(x) (SiLU), elementwise, fp64."""
    x = _f64(x)
    return x * sigmoid(x)


def l2_normalize(x, eps: float = L2_EPS):
    """Each row (last axis) divided by sqrt(sum of its squares + eps)."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def lower_bound_gate(g_raw, A_log, dt_bias=None, lower_bound: float = -5.0):
    """g = lower_bound * sigmoid(exp(A_log[h]) * (g_raw + dt_bias[h, :])).

    g_raw: [T, H, d_k]; A_log: [H]; dt_bias: [H, d_k] or None.  Returns fp64 [T, H, d_k]."""
    g = _f64(g_raw)
    H = g.shape[-2]
    if dt_bias is not None:
        g = g + _f64(dt_bias).reshape(H, -1)
    a = np.exp(_f64(A_log).reshape(H, 1))
    return lower_bound * sigmoid(a * g)


def prologue(q_raw, k_raw, v_raw, g_raw, beta_logit, A_log, dt_bias=None,
             lower_bound: float = -5.0, q_scale: float = 1.0, eps: float = L2_EPS):
    """The inputs of the recurrence from raw projections, all fp64.

    q_raw, k_raw, g_raw: [T, H, d_k]; v_raw: [T, H, d_v]; beta_logit: [T, H]; A_log: [H];
    dt_bias: [H, d_k] or None.  Returns (q, k, v, g, beta)."""
    q = l2_normalize(swish(q_raw), eps) * q_scale
    k = l2_normalize(swish(k_raw), eps)
    v = swish(v_raw)
    g = lower_bound_gate(g_raw, A_log, dt_bias, lower_bound)
    beta = sigmoid(beta_logit)
    return q, k, v, g, beta
