"""Pins of the backward oracle (gradients of the KDA recurrence) to facts outside its own code:

- directional central differences of the separately pinned C forward oracle, for every input
  (q, k, v, g, beta, initial state), with and without a gradient on the final state;
- one token from a zero state, where o = beta (k . q) v gives closed-form gradients;
- beta = 0, where the values never enter the state and dv = 0.
Planted mistakes in copies of its source must each fail a pin.
"""
import os
import types

import numpy as np
import pytest

import oracle
from oracle import backward as B_REAL


def _loss(q, k, v, g, beta, cu, s0, d_out, d_state):
    o, s = oracle.recurrence(q, k, v, g, beta, cu, state_in=s0)
    val = float(np.sum(o * d_out))
    if d_state is not None:
        val += float(np.sum(s * d_state))
    return val


def _case(seed, lens=(3, 2), H=2, dk=4, dv=3):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k = rng.standard_normal((T, H, dk)), rng.standard_normal((T, H, dk)) * 0.5
    v = rng.standard_normal((T, H, dv))
    g = -np.abs(rng.standard_normal((T, H, dk))) * 0.3
    beta = rng.uniform(0.1, 0.9, (T, H))
    s0 = rng.standard_normal((len(lens), H, dk, dv)) * 0.2
    d_out = rng.standard_normal((T, H, dv))
    d_state = rng.standard_normal((len(lens), H, dk, dv))
    return q, k, v, g, beta, cu, s0, d_out, d_state


def pin_finite_differences(Bm):
    for use_ds in (False, True):
        q, k, v, g, beta, cu, s0, d_out, d_state = _case(11 + use_ds)
        ds = d_state if use_ds else None
        grads = Bm.recurrence_backward(q, k, v, g, beta, cu, d_out, state_in=s0, d_state=ds)
        inputs = [q, k, v, g, beta, s0]
        rng = np.random.default_rng(5)
        for i, (x, gr) in enumerate(zip(inputs, grads)):
            delta = rng.standard_normal(x.shape)
            eps = 1e-6
            plus = [a.copy() for a in inputs]
            minus = [a.copy() for a in inputs]
            plus[i] = x + eps * delta
            minus[i] = x - eps * delta
            fd = (_loss(*plus[:5], cu, plus[5], d_out, ds) -
                  _loss(*minus[:5], cu, minus[5], d_out, ds)) / (2 * eps)
            ad = float(np.sum(gr * delta))
            assert abs(fd - ad) <= 1e-6 * max(1.0, abs(fd)), (i, use_ds, fd, ad)


def pin_single_token(Bm):
    rng = np.random.default_rng(3)
    dk = dv = 5
    q, k = rng.standard_normal((1, 1, dk)), rng.standard_normal((1, 1, dk))
    v, do = rng.standard_normal((1, 1, dv)), rng.standard_normal((1, 1, dv))
    g = -np.abs(rng.standard_normal((1, 1, dk)))
    b = np.array([[0.7]])
    dq, dkk, dvv, dg, db, ds0 = Bm.recurrence_backward(q, k, v, g, b, [0, 1], do)
    kq, vdo = float(k.ravel() @ q.ravel()), float(v.ravel() @ do.ravel())
    assert np.allclose(dq.ravel(), 0.7 * vdo * k.ravel(), rtol=0, atol=1e-12)
    assert np.allclose(dkk.ravel(), 0.7 * vdo * q.ravel(), rtol=0, atol=1e-12)
    assert np.allclose(dvv.ravel(), 0.7 * kq * do.ravel(), rtol=0, atol=1e-12)
    assert abs(db.item() - kq * vdo) <= 1e-12 and np.all(dg == 0)
    # d o / d S0: o = S1^T q with S1 = D S0 + k u^T and u = beta (v - (D S0)^T k)
    a = np.exp(g.ravel())
    want = a[:, None] * (np.outer(q.ravel(), do.ravel()) - 0.7 * kq * np.outer(k.ravel(), do.ravel()))
    assert np.allclose(ds0[0, 0], want, rtol=0, atol=1e-12)


def pin_beta_zero(Bm):
    q, k, v, g, beta, cu, s0, d_out, d_state = _case(21)
    grads = Bm.recurrence_backward(q, k, v, g, np.zeros_like(beta), cu, d_out, state_in=s0,
                                   d_state=d_state)
    assert np.all(grads[2] == 0)               # values never reach the state
    assert np.any(grads[4] != 0)               # but beta still matters


PINS = [pin_finite_differences, pin_single_token, pin_beta_zero]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_backward_oracle_pins(pin):
    pin(B_REAL)


MISTAKES = [
    ("                S = torch.exp(gl[t, h])[:, None] * S", "                S = torch.exp(gl[t, h])[None, :] * S"),
    ("                u = bl[t, h] * (vl[t, h] - S.T @ kl[t, h])", "                u = bl[t, h] * (vl[t, h] - S @ kl[t, h])"),
    ("                S = S + torch.outer(kl[t, h], u)", "                S = S + torch.outer(u, kl[t, h])"),
    ("                loss = loss + (S.T @ ql[t, h]) @ d_out[t, h]", "                loss = loss + (S @ ql[t, h]) @ d_out[t, h]"),
    ("                loss = loss + (S * _t64(d_state)[n, h]).sum()", "                loss = loss + (S.T * _t64(d_state)[n, h]).sum()"),
]


@pytest.mark.parametrize("old,new", MISTAKES)
def test_planted_backward_mistakes_are_caught(old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "backward.py")).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("backward_mutant")
    exec(compile(src.replace(old, new), "backward_mutant", "exec"), mod.__dict__)
    failed = 0
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, RuntimeError, IndexError, ValueError):
            failed += 1
    assert failed > 0, f"no pin caught: {new}"
