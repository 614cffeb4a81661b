"""Pins of the prologue oracle (raw projections -> q, k, v, g, beta) to closed forms,
symmetries and invariants that hold independently of its code.

- sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, sigmoid(x) + sigmoid(-x) = 1.
- Swish: swish(0) = 0, swish(x) - swish(-x) = x, swish(ln 3) = (3/4) ln 3.
- L2 norm: |y|^2 = s / (s + eps) for a row with sum of squares s; (3, 4) -> (0.6, 0.8).
- Gate: an argument of 0 gives lower_bound / 2, an argument of ln 3 gives (3/4) lower_bound,
  g(u) + g(-u) = lower_bound, values stay in [lower_bound, 0] and fall as g_raw grows; A_log is
  per head and dt_bias per (head, channel), checked at asymmetric positions.
- Order: Swish before the norm, which a hand-worked row distinguishes from the reverse.
The last test plants mistakes in copies of the oracle source and checks that a pin fails.
"""
import math
import os
import types

import numpy as np
import pytest

import oracle
from oracle import input_prologue as P_REAL

LN3 = math.log(3.0)


def pin_sigmoid(P):
    assert P.sigmoid(0.0) == 0.5
    assert abs(P.sigmoid(LN3) - 0.75) < 1e-15
    x = np.linspace(-30, 30, 121)
    assert np.max(np.abs(P.sigmoid(x) + P.sigmoid(-x) - 1.0)) < 1e-15


def pin_swish(P):
    assert P.swish(0.0) == 0.0
    assert abs(P.swish(LN3) - 0.75 * LN3) < 1e-15
    x = np.linspace(-12, 12, 97)
    assert np.max(np.abs(P.swish(x) - P.swish(-x) - x)) < 1e-14
    assert abs(P.swish(40.0) - 40.0) < 1e-12


def pin_l2(P):
    y = P.l2_normalize(np.array([[3.0, 4.0, 0.0]]), eps=0.0)
    assert np.allclose(y, [[0.6, 0.8, 0.0]], rtol=0, atol=1e-15)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((4, 3, 128)) * 0.01
    s = np.sum(x * x, axis=-1)
    y = P.l2_normalize(x, eps=1e-6)
    assert np.allclose(np.sum(y * y, axis=-1), s / (s + 1e-6), rtol=1e-13, atol=0)
    assert np.all(P.l2_normalize(np.zeros((2, 128))) == 0.0)


def pin_gate(P):
    lb = -5.0
    T, H, d = 3, 2, 128
    g_raw = np.zeros((T, H, d))
    A_log = np.array([0.0, math.log(2.0)])
    dt = np.zeros((H, d))
    # argument 0 -> lb / 2 everywhere
    assert np.all(P.lower_bound_gate(g_raw, A_log, dt, lb) == lb / 2)
    # argument ln 3 at (t=2, h=1, c=5): exp(A_log[1]) = 2, g_raw + dt = ln3 / 2, via dt only
    dt2 = np.zeros((H, d))
    dt2[1, 5] = LN3 / 2
    g = P.lower_bound_gate(g_raw, A_log, dt2, lb)
    assert abs(g[2, 1, 5] - 0.75 * lb) < 1e-14
    assert g[2, 0, 5] == lb / 2 and g[2, 1, 4] == lb / 2  # other head, other channel untouched
    # argument ln 3 through g_raw at head 0 (exp(A_log[0]) = 1), no dt_bias
    g_raw2 = np.zeros((T, H, d))
    g_raw2[1, 0, 100] = LN3
    g = P.lower_bound_gate(g_raw2, A_log, None, lb)
    assert abs(g[1, 0, 100] - 0.75 * lb) < 1e-14 and g[1, 1, 100] == lb / 2
    # symmetry, range and monotonicity
    rng = np.random.default_rng(6)
    u = rng.standard_normal((8, H, d)) * 3
    A = rng.standard_normal(H) * 0.5
    gp = P.lower_bound_gate(u, A, None, lb)
    gm = P.lower_bound_gate(-u, A, None, lb)
    assert np.max(np.abs(gp + gm - lb)) < 1e-13
    assert np.all(gp <= 0.0) and np.all(gp >= lb)
    s = np.sort(rng.standard_normal(50) * 4)
    gs = P.lower_bound_gate(s.reshape(50, 1, 1) * np.ones((1, 1, 1)), np.zeros(1), None, lb)
    assert np.all(np.diff(gs.ravel()) < 0)


def pin_prologue(P):
    T, H, d = 2, 2, 128
    z = np.zeros((T, H, d))
    q_raw = z.copy()
    q_raw[1, 0, 0], q_raw[1, 0, 1] = LN3, -LN3  # Swish -> (3/4 ln3, -1/4 ln3), then unit length
    k_raw = z.copy()
    k_raw[0, 1, 7] = LN3                        # one nonzero channel -> unit vector
    v_raw = z.copy()
    v_raw[0, 0, 3] = LN3
    beta_logit = np.zeros((T, H))
    beta_logit[1, 1] = LN3
    q, k, v, g, beta = P.prologue(q_raw, k_raw, v_raw, z, beta_logit, np.zeros(H), None,
                                  lower_bound=-5.0, q_scale=0.5, eps=1e-30)
    r = math.sqrt(0.75 ** 2 + 0.25 ** 2)
    assert abs(q[1, 0, 0] - 0.5 * 0.75 / r) < 1e-14 and abs(q[1, 0, 1] + 0.5 * 0.25 / r) < 1e-14
    assert np.all(q[1, 0, 2:] == 0) and np.all(q[0] == 0) and np.all(q[1, 1] == 0)
    assert abs(k[0, 1, 7] - 1.0) < 1e-14 and np.count_nonzero(k) == 1
    assert abs(v[0, 0, 3] - 0.75 * LN3) < 1e-15 and np.count_nonzero(v) == 1
    assert np.all(g == -2.5)
    assert abs(beta[1, 1] - 0.75) < 1e-15 and beta[0, 0] == 0.5
    # random rows: |k| = 1 and |q| = q_scale up to eps, shapes kept
    rng = np.random.default_rng(7)
    xr = [rng.standard_normal((5, 3, d)) for _ in range(4)]
    q, k, v, g, beta = P.prologue(xr[0], xr[1], xr[2], xr[3], rng.standard_normal((5, 3)),
                                  rng.standard_normal(3), rng.standard_normal((3, d)),
                                  q_scale=0.25)
    assert np.allclose(np.linalg.norm(k, axis=-1), 1.0, atol=1e-5)
    assert np.allclose(np.linalg.norm(q, axis=-1), 0.25, atol=1e-5)
    assert q.shape == (5, 3, d) and beta.shape == (5, 3)


PINS = [pin_sigmoid, pin_swish, pin_l2, pin_gate, pin_prologue]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_prologue_oracle_pins(pin):
    pin(P_REAL)


def test_prologue_is_exported():
    assert oracle.prologue is P_REAL.prologue


MISTAKES = [
    ("return 1.0 / (1.0 + np.exp(-x))", "return 1.0 / (1.0 + np.exp(x))"),
    ("return x * sigmoid(x)", "return x * sigmoid(-x)"),
    ("np.sum(x * x, axis=-1, keepdims=True) + eps", "np.sum(x * x, axis=0, keepdims=True) + eps"),
    ("g = g + _f64(dt_bias).reshape(H, -1)", "g = g + _f64(dt_bias).reshape(-1, H).T"),
    ("return lower_bound * sigmoid(a * g)", "return lower_bound * sigmoid(a + g)"),
    ("a = np.exp(_f64(A_log).reshape(H, 1))", "a = _f64(A_log).reshape(H, 1)"),
    ("q = l2_normalize(swish(q_raw), eps) * q_scale", "q = swish(l2_normalize(q_raw, eps)) * q_scale"),
    ("q = l2_normalize(swish(q_raw), eps) * q_scale", "q = l2_normalize(swish(q_raw), eps)"),
    ("k = l2_normalize(swish(k_raw), eps)", "k = swish(k_raw)"),
    ("v = swish(v_raw)", "v = _f64(v_raw)"),
    ("beta = sigmoid(beta_logit)", "beta = _f64(beta_logit)"),
]


@pytest.mark.parametrize("old,new", MISTAKES)
def test_planted_prologue_mistakes_are_caught(old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "input_prologue.py")).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("prologue_mutant")
    exec(compile(src.replace(old, new), "prologue_mutant", "exec"), mod.__dict__)
    failed = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed > 0, f"no pin caught: {new}"


# ------------------------------ the short convolution ----------------------------------------
def pin_conv(P):
    rng = np.random.default_rng(8)
    T, H, d = 11, 2, 128
    x = rng.standard_normal((T, H, d))
    cu = [0, 7, 7, 11]                        # three sequences, the middle one empty
    ident = np.zeros((H, d, 4)); ident[..., 3] = 1.0
    y, st = P.short_conv(x, ident, cu)
    assert np.array_equal(y, x)               # tap 3 alone is the identity
    assert np.array_equal(st[0], x[4:7]) and np.array_equal(st[2], x[8:11])
    assert np.all(st[1] == 0)                 # an empty sequence passes its (zero) cache through
    delay = np.zeros((H, d, 4)); delay[..., 0] = 1.0
    y, _ = P.short_conv(x, delay, cu)
    assert np.array_equal(y[3:7], x[0:4]) and np.all(y[0:3] == 0)   # a 3-token delay
    assert np.all(y[7:10] == 0) and np.array_equal(y[10], x[7])     # reset at each sequence start
    # hand-worked taps at one asymmetric (head, channel): x_t = t + 1, w = (1, 2, 3, 4)
    w = np.zeros((H, d, 4)); w[1, 5] = [1.0, 2.0, 3.0, 4.0]
    xs = np.zeros((T, H, d)); xs[:, 1, 5] = np.arange(1, T + 1)
    y, _ = P.short_conv(xs, w, [0, T])
    assert y[5, 1, 5] == 1 * 3 + 2 * 4 + 3 * 5 + 4 * 6 and y[1, 1, 5] == 3 * 1 + 4 * 2
    assert np.count_nonzero(y[:, 0]) == 0 and np.count_nonzero(y[:, 1, 4]) == 0
    # two calls with the cache equal one call
    wr = rng.standard_normal((H, d, 4))
    y1, s1 = P.short_conv(x, wr, [0, T])
    ya, sa = P.short_conv(x[:5], wr, [0, 5])
    yb, sb = P.short_conv(x[5:], wr, [0, T - 5], state=sa)
    assert np.allclose(np.concatenate([ya, yb]), y1, rtol=0, atol=1e-13) and np.array_equal(sb, s1)
    # with a cache, the first outputs see the cached inputs: y_0 = w0 c0 + w1 c1 + w2 c2 + w3 x0
    c = rng.standard_normal((1, 3, H, d))
    y, _ = P.short_conv(x[:2], wr, [0, 2], state=c)
    want = wr[..., 0] * c[0, 0] + wr[..., 1] * c[0, 1] + wr[..., 2] * c[0, 2] + wr[..., 3] * x[0]
    assert np.allclose(y[0], want, rtol=0, atol=1e-13)


def pin_conv_cache_size(P):
    # three caches of the 3 inputs before the next token, 96 heads x 128 channels, bf16: the
    # pages' 216 KiB per layer
    x = np.zeros((4, 96, 128))
    _, st = P.short_conv(x, np.zeros((96, 128, 4)), [0, 4])
    assert 3 * st[0].size * 2 == 216 * 1024


def test_conv_pins():
    pin_conv(P_REAL)
    pin_conv_cache_size(P_REAL)


def test_prologue_conv_composes_conv_and_prologue():
    rng = np.random.default_rng(9)
    T, H, d = 9, 2, 128
    raw = [rng.standard_normal((T, H, d)) for _ in range(4)] + [rng.standard_normal((T, H))]
    A, dt = rng.standard_normal(H), rng.standard_normal((H, d))
    ws = [rng.standard_normal((H, d, 4)) for _ in range(3)]
    cs = rng.standard_normal((2, 3, 3, H, d))
    cu = [0, 4, 9]
    out = oracle.input_prologue.prologue_conv(*raw, A, dt, *ws, cu, cs, q_scale=0.5)
    conv = [P_REAL.short_conv(raw[i], ws[i], cu, cs[:, i]) for i in range(3)]
    ref = P_REAL.prologue(conv[0][0], conv[1][0], conv[2][0], raw[3], raw[4], A, dt, q_scale=0.5)
    for a, b in zip(out[:5], ref):
        assert np.array_equal(a, b)
    assert np.array_equal(out[5][:, 1], conv[1][1])


CONV_MISTAKES = [
    ("            y[a:b] += w[:, :, j] * ext[j:j + L]", "            y[a:b] += w[:, :, 3 - j] * ext[j:j + L]"),
    ("            y[a:b] += w[:, :, j] * ext[j:j + L]", "            y[a:b] += w[:, :, j] * ext[j + 1:j + 1 + L]"),
    ("        state_out[n] = ext[-3:]", "        state_out[n] = ext[:3]"),
    ("        prev = _f64(state[n]) if state is not None else np.zeros((3, H, d))",
     "        prev = _f64(state[n]) if state is not None else (ext[-3:] if n else np.zeros((3, H, d)))"),
]


@pytest.mark.parametrize("old,new", CONV_MISTAKES)
def test_planted_conv_mistakes_are_caught(old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "input_prologue.py")).read()
    assert src.count(old) == 1, old
    mod = types.ModuleType("prologue_mutant")
    exec(compile(src.replace(old, new), "prologue_mutant", "exec"), mod.__dict__)
    with pytest.raises((AssertionError, ValueError, IndexError, NameError, UnboundLocalError)):
        with np.errstate(all="ignore"):
            pin_conv(mod)
            pin_conv_cache_size(mod)
