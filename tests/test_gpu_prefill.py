"""GPU parity of the chunked prefill (through the C ABI) against the fp64 oracle.

Small cases span several chunks and a ragged tail; the full-size workloads run in the same
launch configuration the benchmark times, compared on output windows the oracle records
plus every final state.  Packing is checked bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_03_gb300 import synth
from tests.parity import assert_close, errors, oracle_threads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def kda():
    import kimi_delta_attention_03_gb300 as m
    return m


def run_gpu(x, init=True, expect_status=0, **kw):
    out, fin = kda().fwd_chunked(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                 x["cu_seqlens"], x["seqlens"],
                                 init_state=x["init_state"] if init else None, **kw)
    torch.cuda.synchronize()
    if expect_status is not None:
        st = kda().read_device_status()
        assert st == expect_status, f"device status {st} (expected {expect_status})"
    return out, fin


def run_oracle(x, init=True, windows=None, want_out=True):
    s0 = x["init_state"].cpu() if (init and x["init_state"] is not None) else None
    return oracle.recurrence(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), x["log_alpha"].cpu(),
                             x["beta"].cpu(), x["cu_seqlens"].cpu(), state_in=s0,
                             windows=windows, want_out=want_out, threads=oracle_threads())


def rows_of(t, windows):
    return torch.cat([t[lo:hi] for lo, hi in windows]) if windows else t


def check_status():
    assert kda().read_device_status() == 0


def test_tiny_fp32_workload():
    w = synth.workloads()["tiny_fp32"]
    x = synth.make_workload(w, device=DEV)
    out, fin = run_gpu(x)
    o_ref, s_ref = run_oracle(x)
    assert out.dtype == torch.float32
    assert_close("out", out.cpu().numpy(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)
    check_status()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ragged_lengths(dtype):
    lens = [1, 15, 16, 17, 63, 64, 65, 130, 0, 200, 127, 128, 129]
    x = synth.make_inputs(lens, 3, dtype, seed=5, device=DEV)
    out, fin = run_gpu(x)
    o_ref, s_ref = run_oracle(x)
    assert_close("out", out.cpu(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)
    # the zero-length sequence's final state is its initial state, bit for bit
    assert torch.equal(fin[8], x["init_state"][8])
    check_status()


def test_more_sequences_than_the_ranked_dispatch_covers():
    """Beyond 2,048 sequences the CTAs run in packing order instead of longest first; the
    results match the oracle, and the first sequences keep their bits from a small batch that
    is dispatched longest first."""
    rng = np.random.default_rng(11)
    lens = [int(x) for x in rng.integers(0, 141, size=2100)]
    x = synth.make_inputs(lens, 1, torch.bfloat16, seed=12, device=DEV)
    out, fin = run_gpu(x)
    o_ref, s_ref = run_oracle(x)
    assert_close("out", out.cpu(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)
    k = 40
    cu = x["cu_seqlens"].cpu().tolist()
    xs = {key: x[key][:cu[k]].contiguous() for key in ("q", "k", "v", "log_alpha", "beta")}
    xs["init_state"] = x["init_state"][:k].contiguous()
    xs["cu_seqlens"] = x["cu_seqlens"][:k + 1].contiguous()
    xs["seqlens"] = lens[:k]
    o1, f1 = run_gpu(xs)
    assert torch.equal(o1, out[:cu[k]]) and torch.equal(f1, fin[:k])


def _checkpoint_reference(x, lens, every):
    """Oracle states after every `every` tokens: the final states of the packed prefixes."""
    cu = x["cu_seqlens"].cpu().tolist()
    cuts = [(n, m * every) for n, L in enumerate(lens) for m in range(1, L // every + 1)]
    rows = [torch.arange(cu[n], cu[n] + p_) for n, p_ in cuts]
    pick = lambda t: torch.cat([t.cpu()[r] for r in rows])
    cu2 = np.concatenate([[0], np.cumsum([p_ for _, p_ in cuts])]).astype(np.int32)
    s0 = x["init_state"].cpu()[[n for n, _ in cuts]]
    _, s_ref = oracle.recurrence(pick(x["q"]), pick(x["k"]), pick(x["v"]), pick(x["log_alpha"]),
                                 pick(x["beta"]), cu2, state_in=s0, want_out=False,
                                 threads=oracle_threads())
    return s_ref


@pytest.mark.parametrize("every", [64, 256])
def test_checkpoints_match_oracle_prefix_states(every):
    """The state after every `every` tokens of each sequence equals the token loop's state on
    that prefix; outputs and final states stay those of the plain call, bit for bit."""
    lens = [1100, 64, 513, 0, 2085, 255]
    x = synth.make_inputs(lens, 2, torch.bfloat16, seed=21, device=DEV)
    out, fin, ck = kda().fwd_chunked_checkpoints(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                                 x["cu_seqlens"], x["seqlens"], every,
                                                 init_state=x["init_state"])
    torch.cuda.synchronize()
    check_status()
    o0, f0 = run_gpu(x)
    assert torch.equal(out, o0) and torch.equal(fin, f0)
    s_ref = _checkpoint_reference(x, lens, every)
    assert ck.shape[0] == s_ref.shape[0] == sum(L // every for L in lens)
    assert_close("checkpoints", ck.cpu().numpy(), s_ref)


def test_checkpoints_of_a_segmented_sequence():
    """A sequence above 64K tokens runs as segments; checkpoints that fall inside segments and
    on their boundaries come out of the second pass with the right positions."""
    lens = [70000, 300]
    # 16 chunks: checkpoints inside the 65-chunk segments, and the 65th on the boundary of
    # segments 15 and 16 (chunk 1040)
    every = 1024
    assert kda().binding.fwd_plan(lens, 1)["segment_chunks"] == 65
    x = synth.make_inputs(lens, 1, torch.bfloat16, seed=22, device=DEV)
    out, fin, ck = kda().fwd_chunked_checkpoints(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                                 x["cu_seqlens"], x["seqlens"], every,
                                                 init_state=x["init_state"])
    torch.cuda.synchronize()
    check_status()
    s_ref = _checkpoint_reference(x, lens, every)
    assert ck.shape[0] == 70000 // every
    assert_close("checkpoints", ck.cpu().numpy(), s_ref)


def test_no_initial_state():
    x = synth.make_inputs([100, 33], 2, torch.bfloat16, seed=6, device=DEV)
    out, fin = run_gpu(x, init=False)
    o_ref, s_ref = run_oracle(x, init=False)
    assert_close("out", out.cpu(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)


def test_packing_is_bit_exact_and_does_not_leak():
    lens = [70, 0, 129, 64, 1, 200]
    x = synth.make_inputs(lens, 4, torch.bfloat16, seed=8, device=DEV)
    out, fin = run_gpu(x)
    cu = x["cu_seqlens"].cpu().tolist()
    for n, L in enumerate(lens):
        lo, hi = cu[n], cu[n + 1]
        xs = {key: x[key][lo:hi].contiguous() for key in ("q", "k", "v", "log_alpha", "beta")}
        xs["init_state"] = x["init_state"][n:n + 1].contiguous()
        xs["cu_seqlens"] = torch.tensor([0, L], dtype=torch.int32, device=DEV)
        xs["seqlens"] = [L]
        o1, f1 = run_gpu(xs)
        assert torch.equal(o1, out[lo:hi]), f"sequence {n}: packed output differs"
        assert torch.equal(f1[0], fin[n]), f"sequence {n}: packed final state differs"
    # perturb sequence 2; sequences 3.. keep their bits
    y = {key: (val.clone() if torch.is_tensor(val) else val) for key, val in x.items()}
    y["v"][cu[2]:cu[3]] += 1.0
    y["log_alpha"][cu[2]:cu[3]] *= 2
    out2, fin2 = run_gpu(y)
    assert torch.equal(out2[cu[3]:], out[cu[3]:])
    assert torch.equal(fin2[3:], fin[3:])
    assert torch.equal(out2[:cu[2]], out[:cu[2]])
    assert not torch.equal(fin2[2], fin[2])


def test_canaries_outside_outputs_untouched():
    lens = [77, 5]
    x = synth.make_inputs(lens, 2, torch.bfloat16, seed=9, device=DEV)
    T, H = sum(lens), 2
    pad = 4096
    out_buf = torch.full((pad + T * H * 128 + pad,), -12345.0, dtype=torch.bfloat16, device=DEV)
    fin_buf = torch.full((pad + 2 * H * 128 * 128 + pad,), 777.0, dtype=torch.float32,
                         device=DEV)
    out = out_buf[pad:pad + T * H * 128].view(T, H, 128)
    fin = fin_buf[pad:pad + 2 * H * 128 * 128].view(2, H, 128, 128)
    run_gpu(x, out=out, final_state=fin)
    assert (out_buf[:pad] == -12345.0).all() and (out_buf[-pad:] == -12345.0).all()
    assert (fin_buf[:pad] == 777.0).all() and (fin_buf[-pad:] == 777.0).all()
    o_ref, s_ref = run_oracle(x)
    assert_close("out", out.cpu(), o_ref)


def test_init_state_may_alias_final_state():
    x = synth.make_inputs([150, 64, 3], 2, torch.bfloat16, seed=10, device=DEV)
    ref_out, ref_fin = run_gpu(x)
    state = x["init_state"].clone()
    out, fin = kda().fwd_chunked(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                 x["cu_seqlens"], x["seqlens"], init_state=state,
                                 final_state=state)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(state, ref_fin)


def test_resume_from_saved_state_and_decode_continuation():
    T, T1, H = 300, 130, 2
    x = synth.make_inputs([T + 1], H, torch.bfloat16, seed=11, device=DEV)
    part = lambda a, b: {**{key: x[key][a:b].contiguous() for key in
                            ("q", "k", "v", "log_alpha", "beta")},
                         "cu_seqlens": torch.tensor([0, b - a], dtype=torch.int32, device=DEV),
                         "seqlens": [b - a], "init_state": x["init_state"]}
    full_out, full_fin = run_gpu(part(0, T + 1))
    a_out, a_fin = run_gpu(part(0, T1))
    pb = part(T1, T)
    pb["init_state"] = a_fin
    b_out, b_fin = run_gpu(pb)
    o_ref, s_ref = run_oracle(part(0, T))
    assert_close("resumed out", torch.cat([a_out, b_out]).cpu(), o_ref)
    assert_close("resumed state", b_fin.cpu().numpy(), s_ref)
    # one more token through the decode path equals the prefill's last token
    state = b_fin.clone()
    xt = {key: x[key][T:T + 1].contiguous() for key in ("q", "k", "v", "log_alpha", "beta")}
    o_dec = kda().decode_step(xt["q"], xt["k"], xt["v"], xt["log_alpha"], xt["beta"], state)
    torch.cuda.synchronize()
    o_ref1, s_ref1 = run_oracle(part(0, T + 1), windows=[(T, T + 1)])
    assert_close("decode after prefill out", o_dec.cpu(), o_ref1)
    assert_close("decode after prefill state", state.cpu().numpy(), s_ref1)
    assert_close("prefill(T+1) last", full_out[T:].cpu(), o_ref1)


def _host_copies(x, init):
    host = {nm: x[nm].cpu().pin_memory() for nm in ("q", "k", "v", "log_alpha", "beta")}
    s0 = x["init_state"].cpu().pin_memory() if init else None
    return host, s0


@pytest.mark.parametrize("parts", [1, 2, 3, 8])
@pytest.mark.parametrize("init", [True, False])
def test_host_buffer_call_matches_oracle(parts, init):
    """kda_fwd_chunked_host (pinned host buffers; uploads, kernels and downloads overlapped by
    token-range part) against the oracle.  With one part it is one kernel call over every
    sequence and gives the bits of the device call; with more, a sequence cut by a part boundary
    resumes from its fp32 state, and a sequence of at most one chunk (always inside the first
    part) still gets the device call's bits."""
    lens = [1000, 64, 3, 2048, 0, 517, 130]
    x = synth.make_inputs(lens, 4, torch.bfloat16, seed=21, device=DEV)
    out_d, fin_d = run_gpu(x, init=init)
    host, s0 = _host_copies(x, init)
    out_h, fin_h = kda().fwd_chunked_host(host["q"], host["k"], host["v"], host["log_alpha"],
                                          host["beta"], x["seqlens"], init_state=s0, parts=parts)
    assert out_h.device.type == "cpu" and fin_h.device.type == "cpu"
    check_status()
    o_ref, s_ref = run_oracle(x, init=init)
    assert_close("out", out_h, o_ref)
    assert_close("final_state", fin_h.numpy(), s_ref)
    if parts == 1:
        assert torch.equal(out_h, out_d.cpu()) and torch.equal(fin_h, fin_d.cpu())
    starts = np.concatenate([[0], np.cumsum(lens)])
    for n, length in enumerate(lens):
        if length <= 64:
            rows = slice(int(starts[n]), int(starts[n + 1]))
            assert torch.equal(out_h[rows], out_d.cpu()[rows])
            assert torch.equal(fin_h[n], fin_d.cpu()[n])


def test_host_buffer_call_long_sequence_and_fp32():
    """A sequence longer than 65,536 tokens is cut into parts of at most that span even with
    parts = 1 (so no part needs the segment workspace); fp32 inputs take the same pipeline."""
    x = synth.make_inputs([70000, 100, 0], 1, torch.bfloat16, seed=22, device=DEV)
    host, s0 = _host_copies(x, True)
    out_h, fin_h = kda().fwd_chunked_host(host["q"], host["k"], host["v"], host["log_alpha"],
                                          host["beta"], x["seqlens"], init_state=s0, parts=1)
    check_status()
    o_ref, s_ref = run_oracle(x)
    assert_close("out", out_h, o_ref)
    assert_close("final_state", fin_h.numpy(), s_ref)
    assert torch.equal(fin_h[2], x["init_state"][2].cpu())  # empty: the initial state
    x32 = synth.make_inputs([300, 0, 129], 2, torch.float32, seed=23, device=DEV)
    host, s0 = _host_copies(x32, True)
    out_h, fin_h = kda().fwd_chunked_host(host["q"], host["k"], host["v"], host["log_alpha"],
                                          host["beta"], x32["seqlens"], init_state=s0, parts=3)
    check_status()
    o_ref, s_ref = run_oracle(x32)
    assert_close("out fp32", out_h.numpy(), o_ref)
    assert_close("final_state fp32", fin_h.numpy(), s_ref)


def test_host_buffer_call_equal_lengths():
    """Equal lengths: each part's rows of all sequences move in one strided copy per tensor."""
    x = synth.make_inputs([300] * 5, 2, torch.bfloat16, seed=24, device=DEV)
    host, s0 = _host_copies(x, True)
    out_h, fin_h = kda().fwd_chunked_host(host["q"], host["k"], host["v"], host["log_alpha"],
                                          host["beta"], x["seqlens"], init_state=s0, parts=4)
    check_status()
    o_ref, s_ref = run_oracle(x)
    assert_close("out", out_h, o_ref)
    assert_close("final_state", fin_h.numpy(), s_ref)


def test_host_buffer_call_bounded_gate():
    """Gates over K3's whole bounded range (decay windows shorter than a chunk) through the
    host-buffer call: sequences resumed from their fp32 state at part boundaries, against the
    oracle."""
    lens = [1000, 3000, 17, 0, 640]
    x = synth.make_inputs(lens, 2, torch.bfloat16, seed=25, device=DEV, bounded_gate=-5.0)
    host, s0 = _host_copies(x, True)
    out_h, fin_h = kda().fwd_chunked_host(host["q"], host["k"], host["v"], host["log_alpha"],
                                          host["beta"], x["seqlens"], init_state=s0, parts=5)
    check_status()
    o_ref, s_ref = run_oracle(x)
    assert_close("out", out_h, o_ref)
    assert_close("final_state", fin_h.numpy(), s_ref)


def test_host_buffer_call_pageable_memory():
    """Pageable (not pinned) host inputs and outputs: the copies no longer overlap, but the call
    gives the same results as with pinned buffers."""
    lens = [700, 64, 1500]
    x = synth.make_inputs(lens, 2, torch.bfloat16, seed=26, device=DEV)
    pinned, s0p = _host_copies(x, True)
    out_p, fin_p = kda().fwd_chunked_host(pinned["q"], pinned["k"], pinned["v"],
                                          pinned["log_alpha"], pinned["beta"], x["seqlens"],
                                          init_state=s0p, parts=4)
    pageable = {nm: x[nm].cpu() for nm in ("q", "k", "v", "log_alpha", "beta")}
    assert not pageable["q"].is_pinned()
    out_h = torch.empty_like(pageable["q"])
    fin_h = torch.empty((len(lens), 2, 128, 128), dtype=torch.float32)
    kda().fwd_chunked_host(pageable["q"], pageable["k"], pageable["v"], pageable["log_alpha"],
                           pageable["beta"], x["seqlens"], init_state=x["init_state"].cpu(),
                           out=out_h, final_state=fin_h, parts=4)
    check_status()
    assert torch.equal(out_h, out_p) and torch.equal(fin_h, fin_p)


def test_host_buffer_call_full_size():
    """The benchmark's end-to-end call: 4 x 8192 tokens, 32 heads, 8 parts (each copy one
    strided run over the four sequences).  Every output and state against the device call through the parity gate, and
    the first and last (sequence, head) units against the oracle run on those units alone."""
    w = synth.workloads()["prefill_4x8k"]
    x = synth.make_workload(w, device=DEV)
    out_d, fin_d = run_gpu(x)
    host, s0 = _host_copies(x, True)
    out_h, fin_h = kda().fwd_chunked_host(host["q"], host["k"], host["v"], host["log_alpha"],
                                          host["beta"], x["seqlens"], init_state=s0, parts=8)
    check_status()
    assert_close("out vs device call", out_h, out_d.cpu().float().numpy())
    assert_close("final_state vs device call", fin_h.numpy(), fin_d.cpu().numpy())
    L, N, H = w.lengths[0], len(w.lengths), w.heads
    for n, h in ((0, 0), (N - 1, H - 1)):
        rows = slice(n * L, (n + 1) * L)
        o_ref, s_ref = oracle.recurrence(
            *(x[key][rows, h:h + 1].cpu() for key in ("q", "k", "v", "log_alpha", "beta")),
            torch.tensor([0, L], dtype=torch.int32),
            state_in=x["init_state"][n:n + 1, h:h + 1].cpu(), threads=oracle_threads())
        assert_close(f"out[{n},{h}]", out_h[rows, h:h + 1], o_ref)
        assert_close(f"final_state[{n},{h}]", fin_h[n:n + 1, h:h + 1].numpy(), s_ref)


def test_deterministic():
    x = synth.make_inputs([513, 77], 3, torch.bfloat16, seed=12, device=DEV)
    o1, f1 = run_gpu(x)
    o2, f2 = run_gpu(x)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


# ------------------------- the bounded gate's whole range ------------------------------
# K3's gate is lower_bound * sigmoid(...) with lower_bound = -5 ("How Kimi K3 Engineered Its Way
# to the Frontier", section "How KDA updates its state"), so every log alpha in [-5, 0] is a
# legitimate input.  A 64-token chunk of such gates decays by up to 320 in one channel; the
# prefill then runs the block as shorter decay windows and must still match the token loop.
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_bounded_gate_whole_range_matches_oracle(dtype):
    lens = [1, 15, 16, 17, 63, 64, 65, 130, 0, 200, 127, 513]
    x = synth.make_inputs(lens, 3, dtype, seed=14, device=DEV, bounded_gate=-5.0)
    la = x["log_alpha"].float()
    assert la.min().item() >= -5.0 and la.max().item() <= 0.0
    out, fin = run_gpu(x)
    o_ref, s_ref = run_oracle(x)
    assert_close("out", out.cpu(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)


@pytest.mark.parametrize("lg", [-5.0, -4.9, -2.6, -20.0])
def test_constant_fast_decay_matches_oracle(lg):
    """Every token at one decay: -5 and -4.9 (16-token windows), -2.6 (a 64-token chunk decays by
    166: 28-token windows), -20 (the steepest gate the four-token groups cover: 4-token windows).
    Half the channels decay slowly, so the state still carries information across windows."""
    lens = [300, 64, 77]
    x = synth.make_inputs(lens, 2, torch.bfloat16, seed=15, device=DEV)
    x["log_alpha"][..., :64] = lg
    out, fin = run_gpu(x)
    o_ref, s_ref = run_oracle(x)
    assert_close("out", out.cpu(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)


def test_fast_decay_packing_is_bit_exact():
    """Windows depend on a sequence's own gates only: packed equals separate, bit for bit."""
    lens = [70, 200, 1, 129]
    x = synth.make_inputs(lens, 2, torch.bfloat16, seed=16, device=DEV, bounded_gate=-5.0)
    out, fin = run_gpu(x)
    cu = x["cu_seqlens"].cpu().tolist()
    for n, L in enumerate(lens):
        lo, hi = cu[n], cu[n + 1]
        xs = {key: x[key][lo:hi].contiguous() for key in ("q", "k", "v", "log_alpha", "beta")}
        xs["init_state"] = x["init_state"][n:n + 1].contiguous()
        xs["cu_seqlens"] = torch.tensor([0, L], dtype=torch.int32, device=DEV)
        xs["seqlens"] = [L]
        o1, f1 = run_gpu(xs)
        assert torch.equal(o1, out[lo:hi]) and torch.equal(f1[0], fin[n]), f"sequence {n}"


@pytest.mark.parametrize("every", [64, 256])
def test_fast_decay_checkpoints(every):
    """Windows never cross a 64-token block, so checkpoints land on window ends; they match the
    oracle's prefix states and leave outputs and final states bit-identical to the plain call."""
    lens = [1100, 64, 513, 2085]
    x = synth.make_inputs(lens, 2, torch.bfloat16, seed=17, device=DEV, bounded_gate=-5.0)
    out, fin, ck = kda().fwd_chunked_checkpoints(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                                 x["cu_seqlens"], x["seqlens"], every,
                                                 init_state=x["init_state"])
    torch.cuda.synchronize()
    check_status()
    o0, f0 = run_gpu(x)
    assert torch.equal(out, o0) and torch.equal(fin, f0)
    assert_close("checkpoints", ck.cpu().numpy(), _checkpoint_reference(x, lens, every))


def test_fast_decay_segmented_sequence():
    """A split sequence (segments, their transitions, the combine and the second pass) with
    the bounded gate's whole range; channel 0 decays slowly so the state crosses segments."""
    lens = [70000, 300]
    x = synth.make_inputs(lens, 1, torch.bfloat16, seed=18, device=DEV, bounded_gate=-5.0)
    x["log_alpha"][..., 0] = -0.001
    out, fin = run_gpu(x)
    o_ref, s_ref = run_oracle(x)
    assert_close("out", out.cpu(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)


def test_decay_range_is_reported():
    """Beyond the supported domain of the chunked (bf16) path: a four-token group decaying by
    more than 80 (log alpha below -20), or a positive log alpha, sets KDA_ERR_DECAY_RANGE."""
    x = synth.make_inputs([64], 1, torch.bfloat16, seed=13, device=DEV)
    x["log_alpha"] = torch.full_like(x["log_alpha"], -25.0)  # four tokens: -100
    assert kda().read_device_status() == 0
    run_gpu(x, expect_status=-6)
    assert kda().read_device_status() == 0  # cleared by the read
    x["log_alpha"] = torch.full_like(x["log_alpha"], -0.01)
    x["log_alpha"][5, 0, 3] = 0.5
    run_gpu(x, expect_status=-6)


@pytest.mark.parametrize("host,device", [
    ([70000, 100], [0, 100, 70100]),  # same total: the split moves to the other sequence
    ([100, 28], [0, 28, 128]),         # same total, no split
])
def test_device_cu_seqlens_disagreeing_with_host_lengths_is_reported(host, device):
    """Every CTA checks its device-derived length (and every derived offset) against the host
    plan before it touches memory: a disagreement sets KDA_ERR_INVALID_ARG and nothing is
    written.  The buffers are sized from the host lengths, and the device lengths keep the same
    total, so no access could leave them even if a check were missing.  The next call with
    agreeing arrays still matches the oracle."""
    x = synth.make_inputs(host, 2, torch.bfloat16, seed=19, device=DEV)
    bad_cu = torch.tensor(device, dtype=torch.int32, device=DEV)
    assert kda().read_device_status() == 0
    out = torch.full_like(x["q"], 7.0)
    kda().fwd_chunked(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], bad_cu, x["seqlens"],
                      init_state=x["init_state"], out=out)
    torch.cuda.synchronize()
    assert kda().read_device_status() == -1  # KDA_ERR_INVALID_ARG
    assert (out == 7.0).all()  # no CTA wrote
    got, fin = run_gpu(x)
    o_ref, s_ref = run_oracle(x)
    assert_close("out", got.cpu(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)


def test_fp32_inputs_compute_any_gate_exactly():
    """fp32 inputs run the token loop in fp32, which has no exponent range to leave: a gate of
    -25 matches the oracle to fp32 accuracy."""
    xf = synth.make_inputs([100, 3], 2, torch.float32, seed=13, device=DEV)
    xf["log_alpha"][..., :64] = -25.0
    out, fin = run_gpu(xf)
    o_ref, s_ref = run_oracle(xf)
    assert_close("out", out.cpu(), o_ref, rel_tol=1e-5, max_tol=1e-4)
    assert_close("final_state", fin.cpu().numpy(), s_ref, rel_tol=1e-5, max_tol=1e-4)


# ------------------------------- full-size workloads -----------------------------------
def _windows_per_sequence(seqlens, head=128, tail=128):
    wins, t0 = [], 0
    for L in seqlens:
        if L:
            wins.append((t0, t0 + min(L, head)))
            if L > head:
                wins.append((max(t0 + head, t0 + L - tail), t0 + L))
        t0 += L
    return wins


def test_prefill_4x8k_full_size():
    w = synth.workloads()["prefill_4x8k"]
    x = synth.make_workload(w, device=DEV)
    out, fin = run_gpu(x)
    wins = _windows_per_sequence(x["seqlens"], 512, 512)
    o_ref, s_ref = run_oracle(x, windows=wins)
    assert_close("out", rows_of(out, wins).cpu(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)
    check_status()


def test_long_256k_full_size_error_does_not_grow():
    w = synth.workloads()["long_256k"]
    x = synth.make_workload(w, device=DEV)
    out, fin = run_gpu(x)
    T = x["q"].shape[0]
    W = 16384
    wins = [(0, W), (T - W, T)]
    o_ref, s_ref = run_oracle(x, windows=wins)
    o = rows_of(out, wins).cpu()
    first = errors(o[:W].float().numpy(), o_ref[:W])
    last = errors(o[W:].float().numpy(), o_ref[W:])
    assert_close("out first 16K", o[:W], o_ref[:W])
    assert_close("out last 16K", o[W:], o_ref[W:])
    assert_close("final_state", fin.cpu().numpy(), s_ref)
    assert tuple(fin.shape) == (1, 16, 128, 128)
    assert last[0] <= 2.0 * first[0], (first, last)
    check_status()


def test_prefill_4x8k_full_size_fast_decay_half_the_channels():
    """The benchmark's 4 x 8192-token, 32-head launch with log alpha = -4.9 (near K3's bound) in
    half the key channels: every 64-token block runs as four 16-token windows."""
    w = synth.workloads()["prefill_4x8k"]
    x = synth.make_workload(w, device=DEV)
    x["log_alpha"][..., :64] = -4.9
    out, fin = run_gpu(x)
    wins = _windows_per_sequence(x["seqlens"], 512, 512)
    o_ref, s_ref = run_oracle(x, windows=wins)
    assert_close("out", rows_of(out, wins).cpu(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)


def test_varlen_64_full_size():
    w = synth.workloads()["varlen_64"]
    x = synth.make_workload(w, device=DEV)
    out, fin = run_gpu(x)
    wins = _windows_per_sequence(x["seqlens"])
    o_ref, s_ref = run_oracle(x, windows=wins)
    assert_close("out", rows_of(out, wins).cpu(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)
    check_status()


# ------------------------------ segment parallelism ------------------------------------
def test_segmented_sequences_match_oracle():
    """Sequences above 1024 chunks run as segments (transition + state-from-zero per segment,
    composed, then rerun); the result equals the token loop."""
    # 1094, 2, 1032, 1024 chunks: split (17 segments of 65), whole, split (16 of 65), whole
    lens = [70000, 100, 66000, 65536]
    x = synth.make_inputs(lens, 2, torch.bfloat16, seed=31, device=DEV)
    info = kda().binding.fwd_plan(lens, 2)
    assert info["split_sequences"] == 2 and info["work_items"] == 17 + 1 + 16 + 1
    out, fin = run_gpu(x)
    o_ref, s_ref = run_oracle(x)
    assert_close("out", out.cpu(), o_ref)
    assert_close("final_state", fin.cpu().numpy(), s_ref)


def test_segmented_packing_is_bit_exact_and_aliasing_safe():
    lens = [70, 70000, 0, 33]
    x = synth.make_inputs(lens, 2, torch.bfloat16, seed=32, device=DEV)
    out, fin = run_gpu(x)
    cu = x["cu_seqlens"].cpu().tolist()
    for n, L in enumerate(lens):
        lo, hi = cu[n], cu[n + 1]
        xs = {key: x[key][lo:hi].contiguous() for key in ("q", "k", "v", "log_alpha", "beta")}
        xs["init_state"] = x["init_state"][n:n + 1].contiguous()
        xs["cu_seqlens"] = torch.tensor([0, L], dtype=torch.int32, device=DEV)
        xs["seqlens"] = [L]
        o1, f1 = run_gpu(xs)
        assert torch.equal(o1, out[lo:hi]) and torch.equal(f1[0], fin[n]), f"sequence {n}"
    state = x["init_state"].clone()
    out2, _ = kda().fwd_chunked(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                x["cu_seqlens"], x["seqlens"], init_state=state,
                                final_state=state)
    torch.cuda.synchronize()
    assert torch.equal(out2, out) and torch.equal(state, fin)
