"""Failure detection, tested without a GPU fault: every wait in the kernels is bounded, so a
barrier phase that never completes ends as a status code, not a hang.  The self-test launches one
CTA that waits, through the kernels' own bounded-wait code, on a phase nothing completes (no TMEM,
copies or MMAs in flight); the sticky status word must then read KDA_ERR_TIMEOUT, clear on read,
and the context must still run the next call correctly."""
import pytest
import torch

import oracle
from kimi_delta_attention_03_gb300 import synth
from tests.parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
KDA_ERR_TIMEOUT = -5


def test_bounded_wait_reports_timeout_and_the_context_survives():
    from kimi_delta_attention_03_gb300 import binding
    import kimi_delta_attention_03_gb300 as kda
    kda.read_device_status()  # start from a clear status word
    assert binding.selftest_wait_timeout() == KDA_ERR_TIMEOUT
    assert kda.read_device_status() == 0  # read and cleared
    d = synth.make_decode_inputs(3, 2, torch.bfloat16, seed=61, device=DEV)
    before = d["state"].cpu()
    o = kda.decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["state"])
    torch.cuda.synchronize()
    assert kda.read_device_status() == 0
    o_ref, s_ref = oracle.decode_step(d["q"].cpu(), d["k"].cpu(), d["v"].cpu(),
                                      d["log_alpha"].cpu(), d["beta"].cpu(), before)
    assert_close("out", o.cpu(), o_ref)
    assert_close("state", d["state"].cpu().numpy(), s_ref)
