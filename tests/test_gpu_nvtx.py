"""With KDA_NVTX=1 every entry point wraps its launches in an NVTX range named after it, so a
profiler's timeline shows which library call launched which kernels.  The results must not
change: a prefill and a decode step run in two fresh processes, with and without the ranges,
give the same bits."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCRIPT = """
import sys, torch
sys.path.insert(0, {root!r})
import kimi_delta_attention_03_gb300 as kda
from kimi_delta_attention_03_gb300 import synth
x = synth.make_inputs([100, 33], 2, torch.bfloat16, seed=6, device="cuda")
out, fin = kda.fwd_chunked(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                           x["seqlens"], init_state=x["init_state"])
d = synth.make_decode_inputs(4, 3, torch.bfloat16, seed=7, device="cuda")
o = kda.decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["state"])
torch.cuda.synchronize()
assert kda.read_device_status() == 0
torch.save({{"out": out.cpu(), "fin": fin.cpu(), "o": o.cpu(), "s": d["state"].cpu()}}, sys.argv[1])
"""


def test_nvtx_ranges_leave_results_unchanged(tmp_path):
    res = {}
    for flag in ("0", "1"):
        path = tmp_path / f"nvtx{flag}.pt"
        subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT), str(path)],
                       env=dict(os.environ, KDA_NVTX=flag), check=True, timeout=600)
        res[flag] = torch.load(path)
    for key in ("out", "fin", "o", "s"):
        assert torch.equal(res["0"][key], res["1"][key]), key
