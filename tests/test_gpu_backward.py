"""GPU parity of the backward pass (gradients of the recurrence) against the fp64 oracle, which
differentiates the token loop with reverse-mode autograd and is pinned by finite differences of
the forward oracle.  Sequences cross several 16-token recompute blocks, one is empty, and the
initial state and the gradient on the final state are each present or absent."""
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
    """2048 tokens cross 128 recompute blocks (the state at every 16th token kept, the rest
    replayed); a second sequence of 17 tokens ends on a one-token block."""
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
