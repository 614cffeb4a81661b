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

The short convolution itself (``short_conv``, ``prologue_conv``): a causal depthwise convolution
along each sequence's tokens with kernel size 4 and a cache of the 3 preceding raw inputs per
channel, three caches per layer (q, k, v) ("How Kimi K3 Engineered Its Way to the Frontier",
section "What the hybrid saves": three ShortConv caches with a kernel size of 4, 216 KiB per
layer in bf16).

Readings where the pages are silent: the L2 norm divides by sqrt(sum of squares + eps) with
eps = 1e-6 (a zero row stays zero); q is multiplied by ``q_scale`` after normalisation (the
pages apply no scale; callers pass 1/sqrt(128) for the usual attention scaling); the
convolution has no bias, tap 3 multiplies the current token, and inputs before a sequence's first
token come from its cache (zeros when none is given).

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


def short_conv(x, w, cu_seqlens, state=None):
    """Causal depthwise convolution of kernel 4 along each sequence's tokens.

    x: [T, H, d] (raw inputs); w: [H, d, 4], tap 3 on the current token; cu_seqlens: [N+1];
    state: [N, 3, H, d], the 3 inputs before each sequence's first token, oldest first (None:
    zeros).  y_t = sum_j w[:, :, j] x_{t-3+j}.  Returns (y [T, H, d], state_out [N, 3, H, d]:
    the last 3 inputs of each sequence, continuing from ``state`` when it is shorter)."""
    x = _f64(x)
    w = _f64(w)
    cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    T, H, d = x.shape
    N = len(cu) - 1
    y = np.zeros((T, H, d))
    state_out = np.zeros((N, 3, H, d))
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        prev = _f64(state[n]) if state is not None else np.zeros((3, H, d))
        ext = np.concatenate([prev, x[a:b]], axis=0)  # ext[t + 3] is x_{a + t}
        L = b - a
        for j in range(4):
            y[a:b] += w[:, :, j] * ext[j:j + L]
        state_out[n] = ext[-3:]
    return y, state_out


def prologue_conv(q_raw, k_raw, v_raw, g_raw, beta_logit, A_log, dt_bias, w_q, w_k, w_v,
                  cu_seqlens, conv_state=None, lower_bound: float = -5.0, q_scale: float = 1.0,
                  eps: float = L2_EPS):
    """The short convolution of q, k and v, then ``prologue``.  conv_state: [N, 3, 3, H, d]
    (tensor q/k/v, then the 3 cached inputs oldest first) or None.  Returns (q, k, v, g, beta,
    conv_state_out [N, 3, 3, H, d])."""
    st = [None if conv_state is None else _f64(conv_state)[:, i] for i in range(3)]
    qc, sq = short_conv(q_raw, w_q, cu_seqlens, st[0])
    kc, sk = short_conv(k_raw, w_k, cu_seqlens, st[1])
    vc, sv = short_conv(v_raw, w_v, cu_seqlens, st[2])
    q, k, v, g, beta = prologue(qc, kc, vc, g_raw, beta_logit, A_log, dt_bias, lower_bound,
                                q_scale, eps)
    return q, k, v, g, beta, np.stack([sq, sk, sv], axis=1)
