"""The compute calls under CUDA graph capture: a captured prefill (plain and with the fused input
prologue), decode step and decode window replay to the same bits as eager calls on the same
buffers (serving loops are replayed from graphs, so the calls must launch nothing that capture
forbids)."""
import pytest
import torch

from kimi_delta_attention_03_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def kda():
    import kimi_delta_attention_03_gb300 as m
    return m


def test_prefill_replays_from_a_graph():
    lens = [700, 64, 1300, 5]
    x = synth.make_inputs(lens, 4, torch.bfloat16, seed=51, device=DEV)
    out_e, fin_e = kda().fwd_chunked(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                     x["cu_seqlens"], x["seqlens"], init_state=x["init_state"])
    out = torch.empty_like(out_e)
    fin = torch.empty_like(fin_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture
        kda().fwd_chunked(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                          x["seqlens"], init_state=x["init_state"], out=out, final_state=fin)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    fin.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        kda().fwd_chunked(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                          x["seqlens"], init_state=x["init_state"], out=out, final_state=fin)
    for _ in range(2):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, out_e) and torch.equal(fin, fin_e)
    assert kda().read_device_status() == 0


def test_prologue_prefill_replays_from_a_graph():
    lens = [700, 64, 1300, 5]
    x = synth.make_raw_inputs(lens, 4, seed=53, device=DEV)
    raw = (x["q_raw"], x["k_raw"], x["v_raw"], x["g_raw"], x["beta_logit"])
    out_e, fin_e = kda().fwd_chunked_prologue(*raw, x["cu_seqlens"], x["seqlens"], x["A_log"],
                                              x["dt_bias"], init_state=x["init_state"])
    out = torch.empty_like(out_e)
    fin = torch.empty_like(fin_e)
    call = lambda: kda().fwd_chunked_prologue(*raw, x["cu_seqlens"], x["seqlens"], x["A_log"],
                                              x["dt_bias"], init_state=x["init_state"], out=out,
                                              final_state=fin)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(2):
        out.zero_()
        fin.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, out_e) and torch.equal(fin, fin_e)
    assert kda().read_device_status() == 0


def test_decode_steps_replay_from_a_graph():
    N, H, steps = 16, 8, 3
    d = synth.make_decode_inputs(N, H, torch.bfloat16, seed=52, device=DEV)
    ref_state = d["state"].clone()
    ref_out = [kda().decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], ref_state)
               for _ in range(steps)]
    state = d["state"].clone()
    out = torch.empty_like(d["q"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        warm = state.clone()
        kda().decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], warm, out=out)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        kda().decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], state, out=out)
    for t in range(steps):  # each replay advances the state in place, as the eager loop did
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out[t])
    assert torch.equal(state, ref_state)


def test_decode_window_replays_from_a_graph():
    lens = [4, 4, 2, 0, 4]
    x = synth.make_inputs(lens, 3, torch.bfloat16, seed=53, device=DEV)
    commit = torch.tensor([2, 4, 0, 0, 1], dtype=torch.int32, device=DEV)
    ref_state = x["init_state"].clone()
    ref_out = kda().decode_window(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                  x["cu_seqlens"], x["seqlens"], ref_state, commit=commit)
    state = x["init_state"].clone()
    out = torch.empty_like(ref_out)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        warm = state.clone()
        kda().decode_window(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                            x["seqlens"], warm, commit=commit, out=out)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        kda().decode_window(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                            x["seqlens"], state, commit=commit, out=out)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(state, ref_state)
