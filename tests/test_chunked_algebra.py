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


def _round_tf32(x):
    """Round to tf32 (10 explicit mantissa bits), to nearest with ties away from zero, as the
    tensor-core input conversion of fp32 operands does."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    b = a.view(np.uint32).astype(np.uint64)
    b = ((b + 0x1000) & 0xFFFFE000).astype(np.uint32)
    return b.view(np.float32).astype(np.float64)


def _round_bf16(x):
    """Round to bf16 (7 explicit mantissa bits), to nearest even."""
    import torch
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def test_backward_operand_precision_choice():
    """Why the backward's products take tf32 operands: on the GPU test's bounded-gate input
    (log alpha = -5 sigmoid(2z), 300 tokens), the chunked backward with every product's operands
    rounded to tf32 meets the parity gate against the token-loop oracle, while bf16 operands miss
    its max-abs term on dg.  Accumulation stays fp64 here (fp32 in the kernels)."""
    import torch
    from kimi_delta_attention_03_gb300 import synth
    from tests.chunked_restatement import unit_backward
    from tests.parity import errors, MAX_ABS_TOL, REL_L2_TOL
    x = synth.make_inputs([300], 1, torch.bfloat16, seed=77, bounded_gate=-5.0)
    gen = torch.Generator().manual_seed(78)
    d_out = torch.randn(300, 1, 128, generator=gen)
    d_state = torch.randn(1, 1, 128, 128, generator=gen) * 0.1
    ref = oracle.recurrence_backward(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                     x["cu_seqlens"], d_out, state_in=x["init_state"],
                                     d_state=d_state)
    f64 = lambda t: t[:, 0].double().numpy()
    args = [f64(x[key]) for key in ("q", "k", "v", "log_alpha", "beta")]
    args += [x["init_state"][0, 0].double().numpy(), f64(d_out), d_state[0, 0].double().numpy()]
    worst = {}
    for name, rnd in (("tf32", _round_tf32), ("bf16", _round_bf16)):
        got = unit_backward(*args, C=16, operand=rnd)
        errs = [errors(g, r[:, 0] if r.ndim == 3 else (r[:, 0] if r.ndim == 2 else r[0, 0]))
                for g, r in zip(got, ref)]
        worst[name] = (max(e[0] for e in errs), max(e[1] for e in errs))
    assert worst["tf32"][0] <= REL_L2_TOL and worst["tf32"][1] <= MAX_ABS_TOL, worst
    assert worst["bf16"][1] > MAX_ABS_TOL, worst
