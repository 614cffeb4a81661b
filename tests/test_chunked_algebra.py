"""The chunked algebra the CUDA path implements equals the oracle's token loop (fp64).

Proven on the CPU before any kernel: padding of a ragged last chunk, the inverse, the
mid-chunk decay reference and segment composition.  Tolerance 1e-10 relative to the largest
magnitude (the forms are exact; only the rounding order differs)."""
import numpy as np
import pytest

import oracle
from tests.chunked_restatement import (block_inverse_nilpotent, block_inverse_unit_lower,
                                       unit_forward, unit_forward_segmented)


def _inputs(L, d, seed, gate=0.1, dv=None):
    rng = np.random.default_rng(seed)
    dv = dv or d
    q = rng.standard_normal((L, d)); q /= np.linalg.norm(q, axis=1, keepdims=True) * np.sqrt(d)
    k = rng.standard_normal((L, d)); k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((L, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    g = -np.log1p(np.exp(rng.standard_normal((L, d)))) * gate
    S0 = rng.standard_normal((d, dv)) * 0.01
    return q, k, v, g, beta, S0


def _oracle_unit(q, k, v, g, beta, S0):
    L = q.shape[0]
    o, s = oracle.recurrence(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None],
                             [0, L], state_in=S0[None, None])
    return o[:, 0], s[0, 0]


def _close(a, b, tol=1e-10):
    scale = max(1.0, float(np.abs(b).max()))
    assert np.abs(a - b).max() <= tol * scale, np.abs(a - b).max()


def test_neumann_doubling_exact_for_16x16_strictly_lower():
    """The 16x16 strictly-lower inverse is exact after three doubling rounds."""
    rng = np.random.default_rng(0)
    for _ in range(5):
        A = np.tril(rng.standard_normal((64, 64)) * 0.3, -1)
        T = block_inverse_unit_lower(A)
        _close(T, np.linalg.inv(np.eye(64) + A), 1e-11)


def test_block_nilpotent_inverse_form():
    """The kernel's form: diagonal blocks by substitution, then (I - N + N^2 - N^3) D."""
    rng = np.random.default_rng(1)
    for scale in (0.05, 0.3, 0.5):
        A = np.tril(rng.standard_normal((64, 64)) * scale, -1)
        _close(block_inverse_nilpotent(A), np.linalg.inv(np.eye(64) + A), 1e-10)


@pytest.mark.parametrize("L", [1, 15, 16, 17, 63, 64, 65, 200])
def test_chunked_equals_token_loop(L):
    x = _inputs(L, 32, seed=L)
    o_c, s_c = unit_forward(*x, C=64)
    o_r, s_r = _oracle_unit(*x)
    _close(o_c, o_r)
    _close(s_c, s_r)


def test_chunked_equals_token_loop_d128_strong_decay():
    x = _inputs(300, 128, seed=7, gate=1.0)   # cumulative log-decay per chunk about -50
    o_c, s_c = unit_forward(*x, C=64)
    o_r, s_r = _oracle_unit(*x)
    _close(o_c, o_r)
    _close(s_c, s_r)


@pytest.mark.parametrize("L,seg", [(256, 64), (300, 128), (129, 64), (64, 64)])
def test_segment_composition_equals_token_loop(L, seg):
    x = _inputs(L, 32, seed=100 + L)
    o_s, s_s = unit_forward_segmented(*x, seg_len=seg, C=64)
    o_r, s_r = _oracle_unit(*x)
    _close(o_s, o_r)
    _close(s_s, s_r)


def test_rectangular_value_dim():
    x = _inputs(90, 16, seed=3, dv=24)
    o_c, s_c = unit_forward(*x, C=32)
    o_r, s_r = _oracle_unit(*x)
    _close(o_c, o_r)
    _close(s_c, s_r)


def _oracle_unit_backward(q, k, v, g, beta, S0, dO, dSN):
    L = q.shape[0]
    got = oracle.recurrence_backward(q[:, None], k[:, None], v[:, None], g[:, None],
                                     beta[:, None], [0, L], dO[:, None],
                                     state_in=S0[None, None], d_state=dSN[None, None])
    return [x[:, 0] for x in got[:5]] + [got[5][0, 0]]


@pytest.mark.parametrize("L,gate", [(1, 0.1), (15, 0.1), (16, 0.1), (17, 0.1), (50, 0.1),
                                    (64, 2.0), (37, 6.0)])
def test_chunked_backward_equals_autograd_of_the_token_loop(L, gate):
    """The 16-token chunked backward (factors about the chunk's mid reference, forward and
    reverse state chains, per-chunk gradients, suffix sum of dG) equals reverse-mode autograd
    of the oracle's token loop: ragged last chunks, and gates down to a mean of -6 per token."""
    from tests.chunked_restatement import unit_backward
    q, k, v, g, beta, S0 = _inputs(L, 32, seed=100 + L, gate=gate, dv=24)
    rng = np.random.default_rng(200 + L)
    dO = rng.standard_normal((L, 24))
    dSN = rng.standard_normal((32, 24)) * 0.1
    got = unit_backward(q, k, v, g, beta, S0, dO, dSN, C=16)
    ref = _oracle_unit_backward(q, k, v, g, beta, S0, dO, dSN)
    for a, b in zip(got, ref):
        _close(a, b, 1e-9)
