"""GPU parity of the decode step (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_03_gb300 import synth
from tests.parity import assert_close, oracle_threads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def kda():
    import kimi_delta_attention_03_gb300 as m
    return m


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_small(dtype):
    d = synth.make_decode_inputs(5, 3, dtype, seed=21, device=DEV)
    before = d["state"].cpu()
    o = kda().decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["state"])
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.decode_step(d["q"].cpu(), d["k"].cpu(), d["v"].cpu(),
                                      d["log_alpha"].cpu(), d["beta"].cpu(), before)
    assert o.dtype == dtype
    assert_close("out", o.float().cpu().numpy(), o_ref)
    assert_close("state", d["state"].cpu().numpy(), s_ref)


def test_decode_three_steps_equal_three_token_recurrence():
    N, H, steps = 6, 2, 3
    x = synth.make_inputs([steps] * N, H, torch.bfloat16, seed=22, device=DEV)
    state = x["init_state"].clone()
    outs = []
    for t in range(steps):
        idx = torch.arange(N, device=DEV) * steps + t
        sel = {key: x[key][idx].contiguous() for key in ("q", "k", "v", "log_alpha", "beta")}
        outs.append(kda().decode_step(sel["q"], sel["k"], sel["v"], sel["log_alpha"],
                                      sel["beta"], state))
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.recurrence(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(),
                                     x["log_alpha"].cpu(), x["beta"].cpu(),
                                     x["cu_seqlens"].cpu(), state_in=x["init_state"].cpu())
    o = torch.stack(outs, 1).reshape(N * steps, H, 128)
    assert_close("out", o.float().cpu().numpy(), o_ref)
    assert_close("state", state.cpu().numpy(), s_ref)


def test_decode_512x96_full_size_sampled():
    """The full decode workload in the benchmark's launch configuration; the oracle checks a
    seeded sample of 768 (sequence, head) units one by one."""
    w = synth.workloads()["decode_512x96"]
    d = synth.make_decode_inputs(512, 96, torch.bfloat16, seed=w.seed, state_std=w.s0_std,
                                 device=DEV)
    gen = torch.Generator().manual_seed(99)
    units = torch.randperm(512 * 96, generator=gen)[:768].sort().values
    n_idx, h_idx = units // 96, units % 96
    before = d["state"][n_idx.to(DEV), h_idx.to(DEV)].cpu()
    o = kda().decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["state"])
    torch.cuda.synchronize()
    pick = lambda t: t[n_idx.to(DEV), h_idx.to(DEV)].cpu()[:, None]
    o_ref, s_ref = oracle.recurrence(pick(d["q"]), pick(d["k"]), pick(d["v"]),
                                     pick(d["log_alpha"]), pick(d["beta"]),
                                     np.arange(769, dtype=np.int32), state_in=before[:, None],
                                     threads=oracle_threads())
    assert_close("out", pick(o).float().numpy(), o_ref)
    after = d["state"][n_idx.to(DEV), h_idx.to(DEV)].cpu()[:, None]
    assert_close("state", after.numpy(), s_ref)
    assert kda().read_device_status() == 0
