"""GPU parity of the backward pass (gradients of the recurrence) against the fp64 oracle, which
differentiates the token loop with reverse-mode autograd and is pinned by finite differences of
the forward oracle.  Sequences cross several 16-token chunks, one is empty, and the initial
state and the gradient on the final state are each present or absent; gates span the bounded
gate's whole range, and a chunk that decays beyond the factors' exponent range is reported."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_03_gb300 import synth
from tests.parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAMES = ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dinit_state")


def kda():
    import kimi_delta_attention_03_gb300 as m
    return m


@pytest.mark.parametrize("dtype,with_init,with_dstate", [
    (torch.bfloat16, True, True), (torch.bfloat16, False, False), (torch.float32, True, False)])
def test_backward_matches_oracle(dtype, with_init, with_dstate):
    lens = [5, 0, 20, 33]
    H = 2
    x = synth.make_inputs(lens, H, dtype, seed=71, device=DEV)
    gen = torch.Generator(device=DEV).manual_seed(72)
    T, N = sum(lens), len(lens)
    d_out = torch.randn(T, H, 128, generator=gen, device=DEV)
    d_state = torch.randn(N, H, 128, 128, generator=gen, device=DEV) * 0.1 if with_dstate else None
    init = x["init_state"] if with_init else None
    got = kda().bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                    x["seqlens"], d_out, init_state=init, d_state=d_state)
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    ref = oracle.recurrence_backward(
        x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["log_alpha"].cpu(), x["beta"].cpu(),
        x["cu_seqlens"].cpu(), d_out.cpu(), state_in=None if init is None else init.cpu(),
        d_state=None if d_state is None else d_state.cpu())
    for name, g, r in zip(NAMES, got, ref):
        assert_close(name, g.cpu().numpy(), r)
    # the empty sequence passes the final-state gradient straight through
    want = d_state[1] if d_state is not None else torch.zeros_like(got[5][1])
    assert torch.equal(got[5][1], want)


def test_backward_long_sequence():
    """2048 tokens cross 128 chunks of 16 tokens (the state at every chunk start kept); a second
    sequence of 17 tokens ends on a one-token chunk."""
    lens, H = [2048, 17], 1
    x = synth.make_inputs(lens, H, torch.bfloat16, seed=73, device=DEV)
    gen = torch.Generator(device=DEV).manual_seed(74)
    d_out = torch.randn(sum(lens), H, 128, generator=gen, device=DEV)
    d_state = torch.randn(len(lens), H, 128, 128, generator=gen, device=DEV) * 0.1
    got = kda().bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                    x["seqlens"], d_out, init_state=x["init_state"], d_state=d_state)
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    ref = oracle.recurrence_backward(
        x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["log_alpha"].cpu(), x["beta"].cpu(),
        x["cu_seqlens"].cpu(), d_out.cpu(), state_in=x["init_state"].cpu(), d_state=d_state.cpu())
    for name, g, r in zip(NAMES, got, ref):
        assert_close(name, g.cpu().numpy(), r)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_backward_bounded_gate_range(dtype):
    """log alpha = -5 sigmoid(2z): the lower-bound gate of "How KDA updates its state" over its
    whole range (down to -5 per token), ragged lengths, with an initial state and a final-state
    gradient; bf16 and fp32 inputs."""
    lens, H = [300, 7, 129], 2
    x = synth.make_inputs(lens, H, dtype, seed=77, device=DEV, bounded_gate=-5.0)
    gen = torch.Generator(device=DEV).manual_seed(78)
    d_out = torch.randn(sum(lens), H, 128, generator=gen, device=DEV)
    d_state = torch.randn(len(lens), H, 128, 128, generator=gen, device=DEV) * 0.1
    got = kda().bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                    x["seqlens"], d_out, init_state=x["init_state"], d_state=d_state)
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    ref = oracle.recurrence_backward(
        x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["log_alpha"].cpu(), x["beta"].cpu(),
        x["cu_seqlens"].cpu(), d_out.cpu(), state_in=x["init_state"].cpu(), d_state=d_state.cpu())
    for name, g, r in zip(NAMES, got, ref):
        assert_close(name, g.cpu().numpy(), r)


def test_backward_decay_near_the_chunk_range_limit():
    """log alpha = -9.5 in a few channels: each 16-token chunk decays by 152 there, just inside
    the factors' limit of 160 (mean -10 per token), so the mid-chunk reference puts factors near
    e^(+-76) in fp32; compared with the oracle."""
    lens, H = [200, 45], 1
    x = synth.make_inputs(lens, H, torch.bfloat16, seed=91, device=DEV)
    la = x["log_alpha"].clone()
    la[:, :, 3] = -9.5
    la[:, :, 77] = -9.5
    la[:, :, 100] = -9.5
    gen = torch.Generator(device=DEV).manual_seed(92)
    d_out = torch.randn(sum(lens), H, 128, generator=gen, device=DEV)
    d_state = torch.randn(len(lens), H, 128, 128, generator=gen, device=DEV) * 0.1
    got = kda().bwd(x["q"], x["k"], x["v"], la, x["beta"], x["cu_seqlens"], x["seqlens"], d_out,
                    init_state=x["init_state"], d_state=d_state)
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    ref = oracle.recurrence_backward(
        x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), la.cpu(), x["beta"].cpu(),
        x["cu_seqlens"].cpu(), d_out.cpu(), state_in=x["init_state"].cpu(), d_state=d_state.cpu())
    for name, g, r in zip(NAMES, got, ref):
        assert_close(name, g.cpu().numpy(), r)


def test_backward_decay_beyond_the_chunk_range_is_reported():
    """A 16-token chunk whose decay passes 160 in a channel (here -12 per token) leaves the
    factors' exponent range: KDA_ERR_DECAY_RANGE, and the next call is still correct."""
    lens, H = [40], 1
    x = synth.make_inputs(lens, H, torch.bfloat16, seed=79, device=DEV)
    la = x["log_alpha"].clone()
    la[:, :, 5] = -12.0
    d_out = torch.ones(40, 1, 128, device=DEV)
    assert kda().read_device_status() == 0
    kda().bwd(x["q"], x["k"], x["v"], la, x["beta"], x["cu_seqlens"], x["seqlens"], d_out,
              init_state=x["init_state"])
    torch.cuda.synchronize()
    assert kda().read_device_status() == -6
    got = kda().bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                    x["seqlens"], d_out, init_state=x["init_state"])
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    ref = oracle.recurrence_backward(
        x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["log_alpha"].cpu(), x["beta"].cpu(),
        x["cu_seqlens"].cpu(), d_out.cpu(), state_in=x["init_state"].cpu())
    for name, g, r in zip(NAMES, got, ref):
        assert_close(name, g.cpu().numpy(), r)


def test_backward_device_lengths_beyond_the_workspace_are_reported():
    """The workspace is sized from the host lengths (one record per 16-token chunk); a device
    cu_seqlens with other lengths and a different chunk total (same token total) would index
    past it, so the first launch compares the totals, reports KDA_ERR_INVALID_ARG and the later
    launches compute nothing."""
    host, device = [16, 16], [0, 2, 32]
    x = synth.make_inputs(host, 1, torch.bfloat16, seed=75, device=DEV)
    d_out = torch.ones(32, 1, 128, device=DEV)
    bad_cu = torch.tensor(device, dtype=torch.int32, device=DEV)
    assert kda().read_device_status() == 0
    kda().bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], bad_cu, x["seqlens"], d_out,
              init_state=x["init_state"])
    torch.cuda.synchronize()
    assert kda().read_device_status() == -1


def test_backward_full_size_first_and_last_unit():
    """The benchmark's 4 x 8192-token, 32-head backward (a 4.4 GB workspace, so the last unit's
    offsets pass 2^32 bytes), in the launch the benchmark times; the first and the last
    (sequence, head) unit compared with the oracle run on those units alone."""
    w = synth.workloads()["prefill_4x8k"]
    x = synth.make_workload(w, device=DEV)
    T, H, N, L = x["q"].shape[0], w.heads, len(w.lengths), w.lengths[0]
    gen = torch.Generator(device=DEV).manual_seed(76)
    d_out = torch.randn(T, H, 128, generator=gen, device=DEV)
    d_state = torch.randn(N, H, 128, 128, generator=gen, device=DEV) * 0.1
    got = kda().bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                    x["seqlens"], d_out, init_state=x["init_state"], d_state=d_state)
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    for n, h in ((0, 0), (N - 1, H - 1)):
        rows = slice(n * L, (n + 1) * L)
        pick = lambda t: t[rows, h:h + 1].cpu()
        ref = oracle.recurrence_backward(
            *(pick(x[key]) for key in ("q", "k", "v", "log_alpha", "beta")), [0, L],
            pick(d_out), state_in=x["init_state"][n:n + 1, h:h + 1].cpu(),
            d_state=d_state[n:n + 1, h:h + 1].cpu())
        mine = [t[rows, h:h + 1] for t in got[:5]] + [got[5][n:n + 1, h:h + 1]]
        for name, g, r in zip(NAMES, mine, ref):
            assert_close(f"{name}[{n},{h}]", g.cpu().numpy(), r)


def test_backward_packing_is_bit_exact():
    """A sequence's gradients do not depend on what is packed beside it: the chunk offsets come
    from its own length, and no launch mixes two sequences' data."""
    lens, H = [37, 300, 5], 2
    x = synth.make_inputs(lens, H, torch.bfloat16, seed=81, device=DEV)
    gen = torch.Generator(device=DEV).manual_seed(82)
    d_out = torch.randn(sum(lens), H, 128, generator=gen, device=DEV)
    d_state = torch.randn(len(lens), H, 128, 128, generator=gen, device=DEV) * 0.1
    got = kda().bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                    x["seqlens"], d_out, init_state=x["init_state"], d_state=d_state)
    a, b = lens[0], lens[0] + lens[1]
    pick = lambda t: t[a:b].contiguous()
    alone = kda().bwd(*(pick(x[key]) for key in ("q", "k", "v", "log_alpha", "beta")),
                      torch.tensor([0, lens[1]], dtype=torch.int32, device=DEV), [lens[1]],
                      pick(d_out), init_state=x["init_state"][1:2].contiguous(),
                      d_state=d_state[1:2].contiguous())
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    for g_all, g_one in zip(got[:5], alone[:5]):
        assert torch.equal(g_all[a:b], g_one)
    assert torch.equal(got[5][1:2], alone[5])


def test_backward_many_short_sequences():
    """More than 1,024 sequences (the chunk-offset scan runs over several tiles), lengths 0 to 3,
    so most chunks are ragged; compared with the oracle."""
    rng = np.random.default_rng(83)
    lens = [int(n) for n in rng.integers(0, 4, size=1300)]
    H = 1
    x = synth.make_inputs(lens, H, torch.bfloat16, seed=84, device=DEV)
    gen = torch.Generator(device=DEV).manual_seed(85)
    d_out = torch.randn(sum(lens), H, 128, generator=gen, device=DEV)
    got = kda().bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                    x["seqlens"], d_out, init_state=x["init_state"])
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    ref = oracle.recurrence_backward(
        x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["log_alpha"].cpu(), x["beta"].cpu(),
        x["cu_seqlens"].cpu(), d_out.cpu(), state_in=x["init_state"].cpu())
    for name, g, r in zip(NAMES, got, ref):
        assert_close(name, g.cpu().numpy(), r)


def test_backward_all_sequences_empty():
    """No tokens at all: the initial-state gradient is the final-state gradient, bit for bit."""
    lens, H = [0, 0, 0], 2
    x = synth.make_inputs(lens, H, torch.bfloat16, seed=86, device=DEV)
    d_state = torch.randn(3, H, 128, 128, device=DEV)
    d_out = torch.zeros(0, H, 128, device=DEV)
    got = kda().bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                    x["seqlens"], d_out, init_state=x["init_state"], d_state=d_state)
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    assert torch.equal(got[5], d_state)
