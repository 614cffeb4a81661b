"""GPU parity of the input prologue (raw projections -> q, k, v, log alpha, beta):

- the standalone prologue kernel against the fp64 oracle, element by element, within one bf16
  rounding of each output (plus, for the Swish outputs, the SFU tanh's error against the row);
- the prologue fused into the prefill against the unfused pipeline (standalone prologue, then
  the plain prefill), bit for bit, including an empty sequence, ragged tails, a segmented
  sequence and no dt_bias;
- the fused prefill against the fp64 oracle (oracle prologue, then the token loop).
"""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_03_gb300 import synth
from tests.parity import assert_close, oracle_threads

pytestmark = pytest.mark.gpu
DEV = "cuda"
QS = 128 ** -0.5
LB = -5.0


def kda():
    import kimi_delta_attention_03_gb300 as m
    return m


def _raw(lens, H, seed, dt_bias=True):
    # N(0, 1) raw gates, with or without an N(0, 1) bias: log alpha spans the bounded gate's
    # whole range (lower_bound, 0) and averages about lower_bound / 2 = -2.5 per token
    x = synth.make_raw_inputs(lens, H, seed=seed, device=DEV)
    if not dt_bias:
        x["dt_bias"] = None
    return x


def _raw_args(x):
    return (x["q_raw"], x["k_raw"], x["v_raw"], x["g_raw"], x["beta_logit"])


def _oracle_inputs(x):
    return oracle.prologue(*_raw_args(x), x["A_log"], x["dt_bias"], lower_bound=LB, q_scale=QS)


@pytest.mark.parametrize("dt_bias", [True, False])
def test_prologue_kernel_matches_oracle(dt_bias):
    x = _raw([300, 64, 1], 4, seed=41, dt_bias=dt_bias)
    outs = kda().prologue(*_raw_args(x), x["A_log"], x["dt_bias"], lower_bound=LB, q_scale=QS)
    torch.cuda.synchronize()
    ref = _oracle_inputs(x)
    for name, got, want in zip(("q", "k", "v", "log_alpha", "beta"), outs, ref):
        assert got.dtype == torch.bfloat16
        g = got.float().cpu().numpy().astype(np.float64)
        # one bf16 rounding (at most 2^-8 relative) of a value computed in fp32: to ~1e-6 for
        # log alpha and beta (exp2 / reciprocal sigmoid); Swish uses the SFU tanh, whose error
        # (about |x| 2.5e-4 before the norm) is bounded against the RMS of the row
        tol = 2.0 ** -8 * np.abs(want) * (1 + 1e-4) + 1e-7
        if name in ("q", "k", "v"):
            tol = tol + 3e-3 * np.sqrt(np.mean(want * want, axis=-1, keepdims=True))
        bad = np.abs(g - want) > tol
        assert not bad.any(), f"{name}: {int(bad.sum())} elements off, first at " \
                              f"{np.argwhere(bad)[0]}: {g[bad][0]} vs {want[bad][0]}"
    assert np.all(outs[3].float().cpu().numpy() <= 0) and np.all(outs[3].float().cpu().numpy() >= LB)


@pytest.mark.parametrize("lens,H,dt_bias", [
    ([300, 64, 0, 129, 1, 1000], 3, True),
    ([300, 64, 0, 129, 1, 1000], 3, False),
    ([70000, 40], 1, True),               # the first sequence is split into segments
])
def test_fused_prologue_equals_prologue_then_prefill(lens, H, dt_bias):
    x = _raw(lens, H, seed=42, dt_bias=dt_bias)
    q, k, v, g, b = kda().prologue(*_raw_args(x), x["A_log"], x["dt_bias"], lower_bound=LB,
                                   q_scale=QS)
    o1, s1 = kda().fwd_chunked(q, k, v, g, b, x["cu_seqlens"], x["seqlens"],
                               init_state=x["init_state"])
    o2, s2 = kda().fwd_chunked_prologue(*_raw_args(x), x["cu_seqlens"], x["seqlens"], x["A_log"],
                                        x["dt_bias"], lower_bound=LB, q_scale=QS,
                                        init_state=x["init_state"])
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    assert torch.equal(o1, o2)
    assert torch.equal(s1, s2)


@pytest.mark.parametrize("dt_bias", [True, False])
def test_fused_prologue_matches_oracle(dt_bias):
    lens = [300, 64, 0, 129, 1000]
    H = 3
    x = _raw(lens, H, seed=43, dt_bias=dt_bias)
    out, fin = kda().fwd_chunked_prologue(*_raw_args(x), x["cu_seqlens"], x["seqlens"],
                                          x["A_log"], x["dt_bias"], lower_bound=LB, q_scale=QS,
                                          init_state=x["init_state"])
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    q, k, v, g, b = _oracle_inputs(x)
    cu, s0 = x["cu_seqlens"].cpu(), x["init_state"].cpu()
    # the kernel's contract rounds each prologue output to bf16 where an unfused pipeline stores
    # it; the oracle applies the same rounding to its own fp64 prologue values
    to_bf16 = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    o_ref, s_ref = oracle.recurrence(*map(to_bf16, (q, k, v, g, b)), cu, state_in=s0,
                                     threads=oracle_threads())
    assert_close("out", out.cpu(), o_ref)
    assert_close("state", fin.cpu().numpy(), s_ref)
    # against the unrounded fp64 prologue, the bf16 storage of the inputs costs well under the
    # 1e-2 relative L2 error bound (its element-wise tail is the inputs' rounding, not the kernel's)
    o64, s64 = oracle.recurrence(q, k, v, g, b, cu, state_in=s0, threads=oracle_threads())
    assert_close("out vs fp64 prologue", out.cpu(), o64, max_tol=np.inf)
    assert_close("state vs fp64 prologue", fin.cpu().numpy(), s64, max_tol=np.inf)


@pytest.mark.parametrize("dt_bias", [True, False])
def test_fused_prologue_full_size_equals_unfused_and_sampled_oracle(dt_bias):
    """The 4 x 8192-token, 32-head workload in the benchmark's launch configuration, on raw gates
    with and without a bias (log alpha across the whole bounded range): the fused call equals
    the unfused pipeline bit for bit, and three (sequence, head) units checked one by one against
    the oracle (oracle prologue, rounded as the contract states, then the token loop)."""
    w = synth.workloads()["prefill_4x8k"]
    x = synth.make_raw_inputs(list(w.lengths), w.heads, seed=w.seed, s0_std=w.s0_std, device=DEV)
    if not dt_bias:
        x["dt_bias"] = None
    out, fin = kda().fwd_chunked_prologue(*_raw_args(x), x["cu_seqlens"], x["seqlens"],
                                          x["A_log"], x["dt_bias"], lower_bound=LB, q_scale=QS,
                                          init_state=x["init_state"])
    q, k, v, g, b = kda().prologue(*_raw_args(x), x["A_log"], x["dt_bias"], lower_bound=LB,
                                   q_scale=QS)
    o2, s2 = kda().fwd_chunked(q, k, v, g, b, x["cu_seqlens"], x["seqlens"],
                               init_state=x["init_state"])
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    assert torch.equal(out, o2) and torch.equal(fin, s2)
    del q, k, v, g, b, o2, s2
    L = w.lengths[0]
    to_bf16 = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    for n, h in ((0, 0), (2, 17), (3, 31)):
        rows = slice(n * L, (n + 1) * L)
        pick = lambda t: t[rows, h:h + 1].cpu()
        dtb = x["dt_bias"][h:h + 1].cpu() if dt_bias else None
        ref_in = oracle.prologue(*(pick(t) for t in _raw_args(x)), x["A_log"][h:h + 1].cpu(),
                                 dtb, lower_bound=LB, q_scale=QS)
        o_ref, s_ref = oracle.recurrence(*map(to_bf16, ref_in), [0, L],
                                         state_in=x["init_state"][n:n + 1, h:h + 1].cpu())
        assert_close(f"out[{n},{h}]", out[rows, h:h + 1].cpu(), o_ref)
        assert_close(f"state[{n},{h}]", fin[n:n + 1, h:h + 1].cpu().numpy(), s_ref)


def test_fused_prologue_at_the_gate_bound_matches_oracle():
    """Raw gates far above zero put every log alpha at the lower bound (-5): a 64-token block
    decays by 320 in log space and runs as 16-token windows.  The result equals the unfused
    pipeline bit for bit and the oracle within the stated bound."""
    x = _raw([256, 70], 2, seed=44, dt_bias=False)
    x["g_raw"] = torch.full_like(x["g_raw"], 10.0)
    out, fin = kda().fwd_chunked_prologue(*_raw_args(x), x["cu_seqlens"], x["seqlens"],
                                          x["A_log"], None, lower_bound=LB, q_scale=QS,
                                          init_state=x["init_state"])
    q, k, v, g, b = kda().prologue(*_raw_args(x), x["A_log"], None, lower_bound=LB, q_scale=QS)
    o2, s2 = kda().fwd_chunked(q, k, v, g, b, x["cu_seqlens"], x["seqlens"],
                               init_state=x["init_state"])
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    assert torch.equal(out, o2) and torch.equal(fin, s2)
    assert LB <= g.float().min().item() <= LB + 0.05
    to_bf16 = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    ref_in = oracle.prologue(*_raw_args(x), x["A_log"], None, lower_bound=LB, q_scale=QS)
    o_ref, s_ref = oracle.recurrence(*map(to_bf16, ref_in), x["cu_seqlens"].cpu(),
                                     state_in=x["init_state"].cpu(), threads=oracle_threads())
    assert_close("out", out.cpu(), o_ref)
    assert_close("state", fin.cpu().numpy(), s_ref)


def test_fused_prologue_reports_a_gate_beyond_the_supported_range():
    """A lower bound of -30 lets a four-token group decay by up to 120 in one channel, beyond
    what the windows cover; the call reports KDA_ERR_DECAY_RANGE in the device status word
    instead of returning silently wrong results."""
    x = _raw([256, 70], 2, seed=44, dt_bias=False)
    x["g_raw"] = torch.full_like(x["g_raw"], 10.0)
    assert kda().read_device_status() == 0
    kda().fwd_chunked_prologue(*_raw_args(x), x["cu_seqlens"], x["seqlens"], x["A_log"], None,
                               lower_bound=-30.0, q_scale=QS, init_state=x["init_state"])
    assert kda().read_device_status() == -6
    assert kda().read_device_status() == 0  # read and cleared


# ------------------------------ decode on raw projections ------------------------------------
def test_decode_step_prologue_equals_prologue_then_step_and_oracle():
    N, H = 300, 4
    x = _raw([1] * N, H, seed=45)
    state0 = (torch.randn(N, H, 128, 128, generator=torch.Generator(device=DEV).manual_seed(45),
                          device=DEV) * 0.02)
    s1, s2 = state0.clone(), state0.clone()
    o1 = kda().decode_step_prologue(*_raw_args(x), s1, x["A_log"], x["dt_bias"], lower_bound=LB,
                                    q_scale=QS)
    q, k, v, g, b = kda().prologue(*_raw_args(x), x["A_log"], x["dt_bias"], lower_bound=LB,
                                   q_scale=QS)
    o2 = kda().decode_step(q, k, v, g, b, s2)
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    # oracle: the prologue (rounded as the contract states), then the decode step, on a sample
    to_bf16 = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    idx = [0, 7, 150, 299]
    ref_in = _oracle_inputs(x)
    sel = lambda a: to_bf16(a[idx])
    o_ref, s_ref = oracle.decode_step(*map(sel, ref_in), state0[idx].cpu())
    assert_close("out", o1[idx].cpu(), o_ref)
    assert_close("state", s1[idx].cpu().numpy(), s_ref)


def test_decode_window_prologue_equals_prologue_then_window():
    rng = np.random.default_rng(46)
    N, H = 200, 4  # more units than the window kernel's persistent grid has CTAs
    lens = rng.integers(0, 17, N).tolist()
    lens[0], lens[1] = 64, 0
    commit = torch.tensor([int(rng.integers(0, L + 1)) for L in lens], dtype=torch.int32,
                          device=DEV)
    x = _raw(lens, H, seed=46)
    state0 = x["init_state"] * 2.0
    s1, s2 = state0.clone(), state0.clone()
    o1 = kda().decode_window_prologue(*_raw_args(x), x["cu_seqlens"], lens, s1, x["A_log"],
                                      x["dt_bias"], lower_bound=LB, q_scale=QS, commit=commit)
    q, k, v, g, b = kda().prologue(*_raw_args(x), x["A_log"], x["dt_bias"], lower_bound=LB,
                                   q_scale=QS)
    o2 = kda().decode_window(q, k, v, g, b, x["cu_seqlens"], lens, s2, commit=commit)
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


# ------------------------------ the short convolution ----------------------------------------
def _conv_weights(H, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    return [torch.randn(H, 128, 4, generator=gen, device=DEV) * 0.5 for _ in range(3)]


def test_prologue_conv_matches_oracle():
    lens = [300, 2, 0, 65, 1]
    H = 3
    x = _raw(lens, H, seed=47)
    w = _conv_weights(H, 47)
    N = len(lens)
    cache_in = (torch.randn(N, 3, 3, H, 128, generator=torch.Generator(device=DEV).manual_seed(7),
                            device=DEV)).to(torch.bfloat16)
    cache_out = torch.empty_like(cache_in)
    outs = kda().prologue_conv(*_raw_args(x), x["cu_seqlens"], lens, x["A_log"], *w,
                               dt_bias=x["dt_bias"], cache_in=cache_in, cache_out=cache_out,
                               lower_bound=LB, q_scale=QS)
    torch.cuda.synchronize()
    ref = oracle.input_prologue.prologue_conv(
        *_raw_args(x), x["A_log"], x["dt_bias"], *(t.cpu() for t in w), x["cu_seqlens"].cpu(),
        cache_in.cpu(), lower_bound=LB, q_scale=QS)
    for name, got, want in zip(("q", "k", "v", "log_alpha", "beta"), outs, ref[:5]):
        g = got.float().cpu().numpy().astype(np.float64)
        tol = 2.0 ** -8 * np.abs(want) * (1 + 1e-4) + 1e-7
        if name in ("q", "k", "v"):  # plus the SFU tanh of Swish (and fp32 convolution sums)
            tol = tol + 3e-3 * np.sqrt(np.mean(want * want, axis=-1, keepdims=True))
        bad = np.abs(g - want) > tol
        assert not bad.any(), f"{name}: {int(bad.sum())} elements off"
    assert np.array_equal(cache_out.float().cpu().numpy(), ref[5])


def test_prologue_conv_split_calls_equal_one_call():
    """Each sequence's tokens in two calls, the cache carried in place between them, give the
    bits of one call."""
    lens = [130, 5, 64, 2]
    H = 2
    x = _raw(lens, H, seed=48)
    w = _conv_weights(H, 48)
    N = len(lens)
    one = kda().prologue_conv(*_raw_args(x), x["cu_seqlens"], lens, x["A_log"], *w,
                              dt_bias=x["dt_bias"], lower_bound=LB, q_scale=QS)
    cu = x["cu_seqlens"].cpu().tolist()
    first = [L // 2 for L in lens]
    parts = ([(cu[n], cu[n] + first[n]) for n in range(N)],
             [(cu[n] + first[n], cu[n + 1]) for n in range(N)])
    cache = torch.zeros(N, 3, 3, H, 128, dtype=torch.bfloat16, device=DEV)
    pieces = []
    for rng_ in parts:
        rows = torch.cat([torch.arange(a, b) for a, b in rng_]).to(DEV)
        sub_lens = [b - a for a, b in rng_]
        sub_cu = torch.tensor([0] + np.cumsum(sub_lens).tolist(), dtype=torch.int32, device=DEV)
        raw = [t[rows].contiguous() for t in _raw_args(x)]
        out = kda().prologue_conv(*raw, sub_cu, sub_lens, x["A_log"], *w, dt_bias=x["dt_bias"],
                                  cache_in=cache, cache_out=cache, lower_bound=LB, q_scale=QS)
        pieces.append((rows, out))
    torch.cuda.synchronize()
    for i in range(5):
        merged = torch.empty_like(one[i])
        for rows, out in pieces:
            merged[rows] = out[i]
        assert torch.equal(merged, one[i])
