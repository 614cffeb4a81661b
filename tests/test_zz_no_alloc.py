"""The entry point for callers that cannot allocate device memory.

kda_fwd_chunked_noalloc serves callers that may not call cudaMalloc where they run (allocator
callbacks, hosts that forbid device allocation, latency-critical paths): it uses the library's
built-in scratch array as the segment workspace.  Checked through the C ABI against
kda_fwd_chunked on two calls in a row.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from kimi_delta_attention_03_gb300 import synth
from tests.parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_noalloc_matches_the_allocating_entry_point_twice():
    """Two calls in a row on different inputs (different lengths and seeds, both splitting
    sequences into segments, the second with fast decay), each equal bit for bit to
    kda_fwd_chunked on the same inputs: the shared scratch array keeps the first call's
    contents, so the second call would expose any slot read before it is written."""
    import kimi_delta_attention_03_gb300 as kda
    from kimi_delta_attention_03_gb300 import binding
    cases = [([70000, 100, 66000], 41, None), ([66000, 3, 71000, 5], 42, -5.0)]
    for call, (lens, seed, gate) in enumerate(cases):
        x = synth.make_inputs(lens, 2, torch.bfloat16, seed=seed, device=DEV, bounded_gate=gate)
        need = binding.fwd_workspace_bytes(lens, 2)
        assert 0 < need <= (48 << 20)
        ref_out, ref_fin = kda.fwd_chunked(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                           x["cu_seqlens"], x["seqlens"],
                                           init_state=x["init_state"])
        out = torch.full_like(x["q"], float("nan"))
        fin = torch.full((len(lens), 2, 128, 128), float("nan"), dtype=torch.float32, device=DEV)
        binding.fwd_chunked_noalloc(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                    x["cu_seqlens"], x["seqlens"], init_state=x["init_state"],
                                    out=out, final_state=fin)
        torch.cuda.synchronize()
        assert binding.read_device_status() == 0
        assert torch.equal(out, ref_out), f"call {call}: outputs differ"
        assert torch.equal(fin, ref_fin), f"call {call}: final states differ"
        assert_close(f"out (call {call})", out.cpu(), ref_out.float().cpu().numpy())
        assert_close(f"final_state (call {call})", fin.cpu().numpy(), ref_fin.cpu().numpy())


def test_noalloc_rejects_requests_beyond_the_scratch_limit():
    from kimi_delta_attention_03_gb300 import binding
    lib = binding.load_library()
    lens = [262144]            # 19 segments at 16 heads
    H = 16                     # 3 * 19 * 16 * 64 KiB = 57 MiB of workspace needed
    assert binding.fwd_workspace_bytes(lens, H) > (48 << 20)
    desc = binding.make_desc(lens, H, torch.bfloat16)
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: the call is refused first
    st = lib.kda_fwd_chunked_noalloc(ctypes.byref(desc), fake, fake, fake, fake, fake, None,
                                     fake, ctypes.c_void_p(2 << 20), None, None)
    assert st == -3  # KDA_ERR_WORKSPACE
