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
    assert_close("out", o.cpu(), o_ref)
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
    assert_close("out", o.cpu(), o_ref)
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
    assert_close("out", pick(o), o_ref)
    after = d["state"][n_idx.to(DEV), h_idx.to(DEV)].cpu()[:, None]
    assert_close("state", after.numpy(), s_ref)
    assert kda().read_device_status() == 0


# ------------------------------ decode windows (speculative decoding) -------------------------
def _window_inputs(lens, H, seed):
    x = synth.make_inputs(lens, H, torch.bfloat16, seed=seed, device=DEV)
    x["init_state"] = x["init_state"] * 2.0  # N(0, 0.02^2), as the decode workload
    return x


def test_decode_window_outputs_and_committed_states_match_oracle():
    """Every token's output equals the token loop's; the state written back is the token loop's
    state after the first commit[n] tokens of each run, and is left untouched for commit 0."""
    lens = [5, 1, 0, 8, 64, 3, 17]
    commit = [5, 0, 0, 3, 64, 2, 40]  # 40 is clamped to the run length 17
    H = 3
    x = _window_inputs(lens, H, seed=31)
    state = x["init_state"].clone()
    out = kda().decode_window(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                              x["seqlens"], state,
                              commit=torch.tensor(commit, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    o_ref, _ = oracle.recurrence(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["log_alpha"].cpu(),
                                 x["beta"].cpu(), x["cu_seqlens"].cpu(),
                                 state_in=x["init_state"].cpu(), want_state=False,
                                 threads=oracle_threads())
    assert_close("out", out.cpu(), o_ref)
    # committed states: the oracle's final states of the committed prefixes
    cu = x["cu_seqlens"].cpu().tolist()
    c = [min(cm, L) for cm, L in zip(commit, lens)]
    rows = [torch.arange(cu[n], cu[n] + c[n]) for n in range(len(lens))]
    pick = lambda t: torch.cat([t.cpu()[r] for r in rows])
    cu2 = np.concatenate([[0], np.cumsum(c)]).astype(np.int32)
    _, s_ref = oracle.recurrence(pick(x["q"]), pick(x["k"]), pick(x["v"]), pick(x["log_alpha"]),
                                 pick(x["beta"]), cu2, state_in=x["init_state"].cpu(),
                                 want_out=False, threads=oracle_threads())
    assert_close("state", state.cpu().numpy(), s_ref)
    for n in range(len(lens)):
        if c[n] == 0:
            assert torch.equal(state[n], x["init_state"][n])


def test_decode_window_of_single_tokens_equals_decode_step():
    N, H = 9, 4
    d = synth.make_decode_inputs(N, H, torch.bfloat16, seed=32, device=DEV)
    s1 = d["state"].clone()
    s2 = d["state"].clone()
    o1 = kda().decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], s1)
    cu = torch.arange(N + 1, dtype=torch.int32, device=DEV)
    o2 = kda().decode_window(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], cu, [1] * N, s2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_decode_window_verify_then_commit():
    """Verify a draft window without touching the state, then replay the accepted prefix and
    commit it: the outputs do not depend on the commit counts, and the committed state is the
    one a full run would have left after those tokens."""
    lens = [6, 6, 6, 6]
    accepted = [0, 2, 5, 6]
    H = 2
    x = _window_inputs(lens, H, seed=33)
    state = x["init_state"].clone()
    zeros = torch.zeros(len(lens), dtype=torch.int32, device=DEV)
    o_verify = kda().decode_window(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                   x["cu_seqlens"], x["seqlens"], state, commit=zeros)
    torch.cuda.synchronize()
    assert torch.equal(state, x["init_state"])
    o_commit = kda().decode_window(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                   x["cu_seqlens"], x["seqlens"], state,
                                   commit=torch.tensor(accepted, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(o_verify, o_commit)
    # a full commit of the same runs passes through the accepted states on the way
    for n, a in enumerate(accepted):
        if a == 0:
            assert torch.equal(state[n], x["init_state"][n])
    ref = x["init_state"].clone()
    kda().decode_window(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                        x["seqlens"], ref, commit=torch.tensor([6] * 4, dtype=torch.int32,
                                                               device=DEV), want_out=False)
    torch.cuda.synchronize()
    assert torch.equal(state[3], ref[3])  # accepted the whole window


def test_decode_window_many_units_equals_token_steps():
    """More (sequence, head) units than the window kernel's persistent grid has CTAs, so each
    CTA takes several units and prefetches the next one's state and token rows while it works.
    Outputs and committed states are bit for bit those of single-token steps taken token by
    token (the window repeats the step's arithmetic in the same order; the step itself is
    checked against the oracle above)."""
    rng = np.random.default_rng(34)
    N, H = 300, 4
    lens = rng.integers(0, 65, N).tolist()
    lens[0], lens[1], lens[2] = 64, 0, 1
    commit = [int(rng.integers(0, L + 1)) for L in lens]
    x = _window_inputs(lens, H, seed=34)
    state = x["init_state"].clone()
    out = kda().decode_window(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                              lens, state,
                              commit=torch.tensor(commit, dtype=torch.int32, device=DEV))
    cu = x["cu_seqlens"].cpu().tolist()
    work = x["init_state"].clone()
    committed = x["init_state"].clone()
    ref_out = torch.zeros_like(out)
    for j in range(max(lens)):
        act = [n for n in range(N) if lens[n] > j]
        rows = torch.tensor([cu[n] + j for n in act], device=DEV)
        ia = torch.tensor(act, device=DEV)
        s = work[ia].contiguous()
        sel = {key: x[key][rows].contiguous() for key in ("q", "k", "v", "log_alpha", "beta")}
        ref_out[rows] = kda().decode_step(sel["q"], sel["k"], sel["v"], sel["log_alpha"],
                                          sel["beta"], s)
        work[ia] = s
        done = [n for n in act if commit[n] == j + 1]
        if done:
            idx = torch.tensor(done, device=DEV)
            committed[idx] = work[idx]
    torch.cuda.synchronize()
    assert kda().read_device_status() == 0
    assert torch.equal(out, ref_out)
    assert torch.equal(state, committed)


def test_decode_window_fp32_inputs_match_oracle():
    """The window kernel's fp32-input instantiation: ragged runs, partial commits."""
    lens = [3, 0, 9, 1, 20]
    commit = [2, 0, 9, 0, 11]
    H = 2
    x = synth.make_inputs(lens, H, torch.float32, seed=35, device=DEV)
    x["init_state"] = x["init_state"] * 2.0
    state = x["init_state"].clone()
    out = kda().decode_window(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                              lens, state,
                              commit=torch.tensor(commit, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert out.dtype == torch.float32
    o_ref, _ = oracle.recurrence(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["log_alpha"].cpu(),
                                 x["beta"].cpu(), x["cu_seqlens"].cpu(),
                                 state_in=x["init_state"].cpu(), want_state=False)
    assert_close("out", out.cpu().numpy(), o_ref)
    cu = x["cu_seqlens"].cpu().tolist()
    rows = [torch.arange(cu[n], cu[n] + commit[n]) for n in range(len(lens))]
    pick = lambda t: torch.cat([t.cpu()[r] for r in rows])
    cu2 = np.concatenate([[0], np.cumsum(commit)]).astype(np.int32)
    _, s_ref = oracle.recurrence(pick(x["q"]), pick(x["k"]), pick(x["v"]), pick(x["log_alpha"]),
                                 pick(x["beta"]), cu2, state_in=x["init_state"].cpu(),
                                 want_out=False)
    assert_close("state", state.cpu().numpy(), s_ref)
