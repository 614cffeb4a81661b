"""Chunked form of KDA restated in fp64 numpy — test-only, not part of the oracle.

It spells out, step by step, the algebra the CUDA prefill path implements, so that the
algebra itself (decay factorisation about a mid-chunk reference, zero padding of the last
chunk, the unit-lower-triangular inverse, the state pass, and segment composition) is proven
equal to the token loop before any kernel runs.  Steps, per (sequence, head) unit, chunk of C
tokens, d_k x d_v state S (all fp64):

  G      = inclusive cumulative sum of g within the chunk          [C, d_k]
  r      = G_C / 2  (per key channel; the mid-chunk reference)
  Q_r    = q * exp(G - r);  K_p = k * exp(G - r);  K_m = k * exp(r - G)
  K_bar  = k * exp(G_C - G)
  A      = strict_lower(diag(beta) K_p K_m^T);   P = lower_incl(Q_r K_m^T)
  T      = (I + A)^{-1}   (16x16 diagonal blocks by the doubling product
                           (I-N)(I+N^2)(I+N^4)(I+N^8), off-diagonal blocks by block
                           forward substitution)
  W      = T diag(beta) K_p;   U_bar = T diag(beta) V
  S'     = diag(exp(r)) S
  U      = U_bar - W S';   O = Q_r S' + P U
  S      = diag(exp(G_C)) S + K_bar^T U

The pages fix the chunkwise idea ("How Kimi K3 Engineered Its Way to the Frontier", section
"FlashKDA steps the state once per 16 tokens": chunk-local dense matmuls, one state step per
chunk, result equal to the token loop; reciprocal cumulative decay; the 16x16 Neumann-series
inverse exact after three doubling rounds).  The segment composition S_out = M S_in + S~ is
the KCP decomposition ("k3_training_and_infra_notes", section 4.1).
"""
from __future__ import annotations

import numpy as np


def block_inverse_unit_lower(A: np.ndarray, block: int = 16) -> np.ndarray:
    """(I + A)^{-1} for strictly lower-triangular A, by 16x16 doubling + block substitution."""
    C = A.shape[0]
    assert C % block == 0
    nb = C // block
    T = np.zeros_like(A)
    eye = np.eye(block)
    for b in range(nb):
        s = slice(b * block, (b + 1) * block)
        N = A[s, s]
        N2 = N @ N
        N4 = N2 @ N2
        N8 = N4 @ N4
        T[s, s] = (eye - N) @ (eye + N2) @ (eye + N4) @ (eye + N8)
    for I in range(1, nb):
        si = slice(I * block, (I + 1) * block)
        for J in range(I):
            sj = slice(J * block, (J + 1) * block)
            acc = np.zeros((block, block))
            for K in range(J, I):
                sk = slice(K * block, (K + 1) * block)
                acc += A[si, sk] @ T[sk, sj]
            T[si, sj] = -T[si, si] @ acc
    return T


def block_inverse_nilpotent(A: np.ndarray, block: int = 16) -> np.ndarray:
    """(I + A)^{-1} in the form the prefill kernel evaluates it: the 16x16 diagonal blocks by
    forward substitution, then with D = blockdiag((I + A_II)^{-1}) and N = D A_off (strictly
    block-lower, so N^4 = 0 for four blocks): (I + A)^{-1} = (I - N + N^2 - N^3) D."""
    C = A.shape[0]
    nb = C // block
    D = np.zeros_like(A)
    for b in range(nb):
        s = slice(b * block, (b + 1) * block)
        Ab = A[s, s]
        X = np.zeros((block, block))
        for col in range(block):
            for i in range(block):
                X[i, col] = (1.0 if i == col else 0.0) - Ab[i, :i] @ X[:i, col]
        D[s, s] = X
    A_off = A.copy()
    for b in range(nb):
        s = slice(b * block, (b + 1) * block)
        A_off[s, s] = 0.0
    N = D @ A_off
    I = np.eye(C)
    return (I - N + N @ N - N @ N @ N) @ D


def chunk_step(S, q, k, v, g, beta):
    """One chunk (rows beyond the sequence already zero-padded).  Returns (O, S_new)."""
    C = q.shape[0]
    G = np.cumsum(g, axis=0)
    GC = G[-1]
    r = GC / 2.0
    Q_r = q * np.exp(G - r)
    K_p = k * np.exp(G - r)
    K_m = k * np.exp(r - G)
    K_bar = k * np.exp(GC - G)
    A = np.tril(beta[:, None] * (K_p @ K_m.T), -1)
    P = np.tril(Q_r @ K_m.T, 0)
    T = block_inverse_unit_lower(A)
    W = T @ (beta[:, None] * K_p)
    U_bar = T @ (beta[:, None] * v)
    S_r = np.exp(r)[:, None] * S
    U = U_bar - W @ S_r
    O = Q_r @ S_r + P @ U
    S_new = np.exp(GC)[:, None] * S + K_bar.T @ U
    return O, S_new


def _chunks(L, C):
    return [(c0, min(L, c0 + C)) for c0 in range(0, L, C)]


def _padded(x, c0, c1, C):
    out = np.zeros((C,) + x.shape[1:])
    out[: c1 - c0] = x[c0:c1]
    return out


def unit_forward(q, k, v, g, beta, S0, C=64):
    """Chunked forward of one unit: q,k,g [L,d_k], v [L,d_v], beta [L]."""
    L = q.shape[0]
    S = S0.copy()
    O = np.zeros((L, v.shape[1]))
    for c0, c1 in _chunks(L, C):
        Oc, S = chunk_step(S, *(_padded(x, c0, c1, C) for x in (q, k, v, g, beta)))
        O[c0:c1] = Oc[: c1 - c0]
    return O, S


def segment_transition(k, v, g, beta, C=64):
    """Pass A of segment parallelism: from a zero incoming state, carry the augmented state
    [S~ | M] (M starts at I, its 'values' are zero) through the segment.  Returns (M, S~)."""
    L, dk = k.shape
    dv = v.shape[1]
    X = np.concatenate([np.zeros((dk, dv)), np.eye(dk)], axis=1)
    for c0, c1 in _chunks(L, C):
        kk, vv, gg, bb = (_padded(x, c0, c1, C) for x in (k, v, g, beta))
        v_aug = np.concatenate([vv, np.zeros((C, dk))], axis=1)
        _, X = chunk_step(X, np.zeros_like(kk), kk, v_aug, gg, bb)
    return X[:, dv:], X[:, :dv]


def unit_forward_segmented(q, k, v, g, beta, S0, seg_len, C=64):
    """Pass A per segment, sequential combine S_in(s+1) = M_s S_in(s) + S~_s, then pass B."""
    L = q.shape[0]
    bounds = [(a, min(L, a + seg_len)) for a in range(0, L, seg_len)] or [(0, 0)]
    trans = [segment_transition(k[a:b], v[a:b], g[a:b], beta[a:b], C) for a, b in bounds]
    s_in = [S0]
    for M, St in trans[:-1]:
        s_in.append(M @ s_in[-1] + St)
    O = np.zeros((L, v.shape[1]))
    S = S0
    for (a, b), Si in zip(bounds, s_in):
        O[a:b], S = unit_forward(q[a:b], k[a:b], v[a:b], g[a:b], beta[a:b], Si, C)
    return O, S


def _unit_lower_inverse16(A):
    """(I + A)^{-1} for a strictly lower-triangular A by forward substitution, column by column."""
    C = A.shape[0]
    X = np.zeros((C, C))
    for col in range(C):
        for i in range(C):
            X[i, col] = (1.0 if i == col else 0.0) - A[i, :i] @ X[:i, col]
    return X


def backward_prep(k, v, q, g, beta, mm=np.matmul):
    """Chunk-local factors of the chunked backward (one chunk of C tokens, zero-padded).

    G = cumsum g; r = G_C / 2; a = exp(G_C)
    K_f = k exp(G), Q_f = q exp(G)                 (decay from the chunk start)
    K_p = k exp(G - r), K_m = k exp(r - G), Q_r = q exp(G - r)   (mid-chunk reference)
    K_bar = k exp(G_C - G)                         (decay to the chunk end)
    At = strict_lower(K_p K_m^T); A = diag(beta) At; P = lower_incl(Q_r K_m^T); T = (I + A)^-1
    W = T diag(beta) K_f; U_bar = T diag(beta) V; Q' = Q_f - P W
    """
    G = np.cumsum(g, axis=0)
    GC = G[-1]
    r = GC / 2.0
    f = dict(G=G, GC=GC, a=np.exp(GC), K_f=k * np.exp(G), Q_f=q * np.exp(G),
             K_p=k * np.exp(G - r), K_m=k * np.exp(r - G), Q_r=q * np.exp(G - r),
             K_bar=k * np.exp(GC - G))
    f["At"] = np.tril(mm(f["K_p"], f["K_m"].T), -1)
    f["P"] = np.tril(mm(f["Q_r"], f["K_m"].T), 0)
    f["T"] = _unit_lower_inverse16(beta[:, None] * f["At"])
    f["W"] = mm(f["T"], beta[:, None] * f["K_f"])
    f["U_bar"] = mm(f["T"], beta[:, None] * v)
    f["Qp"] = f["Q_f"] - mm(f["P"], f["W"])
    return f


def backward_chunk_grads(f, q, k, v, beta, dO, S, dE, U, mm=np.matmul):
    """Gradients of one chunk given its start state S, the gradient dE of its end state and
    its U = U_bar - W S.  Returns (dq, dk, dv, dG, dbeta) with dG the gradient with respect to
    the in-chunk cumulative decay G (the caller turns it into dg by a suffix sum)."""
    dU = mm(f["P"].T, dO) + mm(f["K_bar"], dE)
    dY = mm(f["T"].T, dU)
    R = v - mm(f["K_f"], S)
    dbeta = np.sum(dY * R, axis=1)
    dR = beta[:, None] * dY
    dA = -np.tril(mm(dY, U.T), -1)
    dbeta = dbeta + np.sum(dA * f["At"], axis=1)
    dAt = beta[:, None] * dA
    dP = np.tril(mm(dO, U.T), 0)
    dK_f = -mm(dR, S.T)
    dQ_f = mm(dO, S.T)
    dK_bar = mm(U, dE.T)
    dK_p = mm(dAt, f["K_m"])
    dK_m = mm(dAt.T, f["K_p"]) + mm(dP.T, f["Q_r"])
    dQ_r = mm(dP, f["K_m"])
    G, GC = f["G"], f["GC"]
    r = GC / 2.0
    dk = dK_f * np.exp(G) + dK_p * np.exp(G - r) + dK_m * np.exp(r - G) + dK_bar * np.exp(GC - G)
    dq = dQ_f * np.exp(G) + dQ_r * np.exp(G - r)
    dG = (dK_f * f["K_f"] + dK_p * f["K_p"] - dK_m * f["K_m"] - dK_bar * f["K_bar"]
          + dQ_f * f["Q_f"] + dQ_r * f["Q_r"])
    dG[-1] += np.sum(dK_bar * f["K_bar"], axis=0) + f["a"] * np.sum(dE * S, axis=1)
    return dq, dk, dR, dG, dbeta


def unit_backward(q, k, v, g, beta, S0, dO, dSN, C=16, operand=None):
    """Chunked backward of one unit in three steps: chunk-local factors; the forward chain
    S_{c+1} = diag(a) S_c + K_bar^T (U_bar - W S_c) and the reverse chain
    dE_{c-1} = diag(a) dE_c + Q'^T dO - W^T (K_bar dE_c); then per-chunk gradients.
    Returns (dq, dk, dv, dg, dbeta, dS0).  `operand`, if given, rounds both operands of every
    matrix product (fp64 accumulation), to model a tensor-core input format."""
    mm = np.matmul if operand is None else (lambda a, b: operand(a) @ operand(b))
    L = q.shape[0]
    chunks = _chunks(L, C)
    pads = [[_padded(x, c0, c1, C) for x in (q, k, v, g, beta, dO)] for c0, c1 in chunks]
    facs = [backward_prep(kk, vv, qq, gg, bb, mm) for qq, kk, vv, gg, bb, _ in pads]
    S, starts, Us = S0.copy(), [], []
    for f in facs:
        starts.append(S)
        U = f["U_bar"] - mm(f["W"], S)
        Us.append(U)
        S = f["a"][:, None] * S + mm(f["K_bar"].T, U)
    dE, ends = dSN.copy(), [None] * len(facs)
    for c in range(len(facs) - 1, -1, -1):
        f, dOc = facs[c], pads[c][5]
        ends[c] = dE
        dE = f["a"][:, None] * dE + mm(f["Qp"].T, dOc) - mm(f["W"].T, mm(f["K_bar"], dE))
    out = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(g), np.zeros(L)]
    for c, (c0, c1) in enumerate(chunks):
        qq, kk, vv, _, bb, dOc = pads[c]
        dq, dk, dv, dG, db = backward_chunk_grads(facs[c], qq, kk, vv, bb, dOc, starts[c],
                                                  ends[c], Us[c], mm)
        dg = np.cumsum(dG[::-1], axis=0)[::-1]
        n = c1 - c0
        for o, x in zip(out, (dq, dk, dv, dg, db)):
            o[c0:c1] = x[:n]
    return (*out, dE)
