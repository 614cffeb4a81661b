"""fp64 oracle of the gradients of the KDA recurrence (the backward pass).

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``).

The forward is the token loop of "How Kimi K3 Engineered Its Way to the Frontier", section "How
KDA updates its state" (forget, erase-and-write, read), written once more in plain torch float64
so that reverse-mode automatic differentiation gives its exact gradients; no hand-derived formula
is involved.  For each (sequence, head) unit:

    S <- diag(exp(g_t)) S;   u <- beta_t (v_t - S^T k_t);   S <- S + k_t u^T;   o_t = S^T q_t

Given the gradients of a loss with respect to every o_t (d_out) and, optionally, the final state
(d_state), it returns the gradients with respect to q, k, v, g (the natural-log gate), beta and
the initial state.

Pinned by ``tests/test_oracle_backward.py``: central finite differences of the (separately
pinned) C forward oracle, and special cases with closed forms.
"""
from __future__ import annotations

import numpy as np
import torch


def _t64(x):
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    return x.detach().cpu().to(torch.float64)


def recurrence_backward(q, k, v, g, beta, cu_seqlens, d_out, state_in=None, d_state=None):
    """Gradients of the KDA forward.  q, k, g: [T, H, dk]; v, d_out: [T, H, dv]; beta: [T, H];
    state_in, d_state: [N, H, dk, dv] or None (zeros).  Returns (dq, dk, dv, dg, dbeta, dstate_in)
    as float64 numpy arrays of the same shapes."""
    q, k, v, g, beta, d_out = (_t64(x) for x in (q, k, v, g, beta, d_out))
    T, H, dk = q.shape
    dv = v.shape[-1]
    cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    N = len(cu) - 1
    s0 = _t64(state_in) if state_in is not None else torch.zeros(N, H, dk, dv, dtype=torch.float64)
    leaves = [x.clone().requires_grad_(True) for x in (q, k, v, g, beta, s0)]
    ql, kl, vl, gl, bl, sl = leaves
    loss = torch.zeros((), dtype=torch.float64)
    for n in range(N):
        for h in range(H):
            S = sl[n, h]
            for t in range(cu[n], cu[n + 1]):
                S = torch.exp(gl[t, h])[:, None] * S                    # forget
                u = bl[t, h] * (vl[t, h] - S.T @ kl[t, h])               # erase target
                S = S + torch.outer(kl[t, h], u)                         # write
                loss = loss + (S.T @ ql[t, h]) @ d_out[t, h]             # read, weighted by d_out
            if d_state is not None:
                loss = loss + (S * _t64(d_state)[n, h]).sum()
    grads = torch.autograd.grad(loss, leaves, allow_unused=True)
    out = []
    for gr, leaf in zip(grads, leaves):
        out.append(np.zeros(tuple(leaf.shape)) if gr is None else gr.numpy())
    return tuple(out)
