"""Benchmark of the KDA forward hot path on GB300.

One step = one chunked prefill call over the prefill_4x8k workload (4 sequences x 8192
tokens, 32 heads, d = 128, bf16 inputs, fp32 state) with every input resident in HBM.  The
decode step on the decode_512x96 workload (512 sequences x 96 heads, fp32 state updated in
place) is timed in the same run and reported under "decode".

Prints ONE JSON line (rank 0).  With --impl reference the fp64 CPU oracle is timed instead,
on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill Mtokens/s (% bf16 TC roofline); decode state-update GB/s on 1 GB300"
D = 128
CHUNK = 64
BYTES_PER_TOKEN_HEAD = 4 * D * 2 + 2 + D * 2        # q, k, v, log_alpha in; beta; o out
FLOPS_PER_TOKEN_HEAD = 8 * CHUNK * D + 6 * D * D + 2 * CHUNK * D   # dense chunk tiles
STATE_BYTES = D * D * 4
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        p = json.load(open(path))
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# The traffic records cover the prefill and decode kernels: the hash that dates them is taken
# over those kernels' translation units and every shared header they include.
_RECORDED_SOURCES = ("kda_prefill_tc.cu", "kda_decode.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kimi_delta_attention_03_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f in _RECORDED_SOURCES or f.endswith(".cuh"):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(name: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path)).get(name)
    except Exception:
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.result = None
        if self.proc is None:
            return False
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 9:
                continue
            try:
                sm.append(float(row[1]))
                mx.append(float(row[2]))
            except ValueError:
                continue
            for nm, val in zip(names, row[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(nm)
        if sm:
            self.result = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                           "reasons": sorted(reasons), "samples": len(sm)}
        return False


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(x, tokens: int, threads: int):
    """Time the fp64 oracle on the first ``tokens`` tokens of every sequence of ``x``, all
    heads (the whole workload when ``tokens`` covers the longest sequence)."""
    import oracle
    cu = x["cu_seqlens"].cpu().tolist()
    take = [min(tokens, cu[n + 1] - cu[n]) for n in range(len(cu) - 1)]
    rows = torch.cat([torch.arange(cu[n], cu[n] + take[n]) for n in range(len(take))])
    sl = lambda t: t.cpu()[rows].contiguous()
    cu2 = [0]
    for n in take:
        cu2.append(cu2[-1] + n)
    s0 = x["init_state"].cpu() if x["init_state"] is not None else None
    args = [sl(x[key]) for key in ("q", "k", "v", "log_alpha", "beta")]
    t0 = time.perf_counter()
    oracle.recurrence(*args, cu2, state_in=s0, threads=threads)
    return time.perf_counter() - t0, cu2[-1]


def sample_text(x, tokens: int, heads: int) -> str:
    cu = x["cu_seqlens"].cpu().tolist()
    lens = [cu[n + 1] - cu[n] for n in range(len(cu) - 1)]
    if tokens >= max(lens):
        return (f"the whole workload ({len(lens)} sequences x {max(lens)} tokens, {heads} "
                f"heads), fp64 token loop")
    return (f"first {tokens} tokens of each of the {len(lens)} sequences, {heads} heads, "
            f"fp64 token loop")


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: bounded samples of the same workload."""
    if rank != 0:
        return
    from kimi_delta_attention_03_gb300 import synth
    w = synth.workloads()["prefill_4x8k"]
    x = synth.make_workload(w, device="cpu")
    threads = cpu_cores()
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle_sample(x, min(256, args.ref_tokens), threads)
    runs = [oracle_sample(x, args.ref_tokens, threads) for _ in range(args.steps)]
    sec = sum(t for t, _ in runs) / len(runs)
    value = runs[0][1] / sec / 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Mtokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample_tokens": runs[0][1], "heads": w.heads,
                   "d": D},
        "cpu_baseline": {"value": value, "unit": "Mtokens/s", "cores": threads,
                         "kind": "oracle", "sample": sample_text(x, args.ref_tokens, w.heads)},
        "e2e": {"value": value, "unit": "Mtokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_device(fn, steps, stream):
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    stop.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(stop) / steps  # ms per step


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=8192,
                    help="oracle sample: first N tokens of every sequence (8192 = all)")
    ap.add_argument("--cpu-baseline-tokens", type=int, default=8192,
                    help="oracle sample of the cpu_baseline leg, as --ref-tokens")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--case", default="full", choices=["full", "small", "small_prologue"],
                    help="small: a reduced prefill (4 x 4096 tokens, 8 heads) and decode "
                         "(64 x 96) for ncu section captures; small_prologue: the same prefill "
                         "plus the fused and unfused input prologue; not benchmark figures")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip timing the long-context and varlen prefill workloads")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
        barrier(world)
        return

    import kimi_delta_attention_03_gb300 as kda
    from kimi_delta_attention_03_gb300 import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    hbm_peak, tc_peak, peak_kind = peaks()

    small = args.case in ("small", "small_prologue")
    if small:
        args.no_extra = args.no_e2e = args.no_cpu_baseline = True

    # ---------------- prefill (headline) ----------------
    w = synth.workloads()["prefill_4x8k"]
    if small:
        from dataclasses import replace
        w = replace(w, name="prefill_small (B=4, T=4096, H=8, bf16; profiling case)",
                    lengths=(4096,) * 4, heads=8)
    x = synth.make_workload(w, device=dev)
    T, H = x["q"].shape[0], w.heads
    out = torch.empty_like(x["q"])
    fin = torch.empty((len(w.lengths), H, D, D), dtype=torch.float32, device=dev)

    def step():
        kda.fwd_chunked(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                        x["seqlens"], init_state=x["init_state"], out=out, final_state=fin)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    launches0 = kda.launch_count()
    with ClockSampler(local) as clk:
        ms = time_device(step, args.steps, stream)
    launches = kda.launch_count() - launches0
    barrier(world)
    ms_max = max_over_ranks(ms, world)
    tokens_all = T * world
    value = tokens_all / (ms_max * 1e-3) / 1e6
    units = len(w.lengths) * H
    alg_bytes = T * H * BYTES_PER_TOKEN_HEAD + units * 2 * STATE_BYTES
    alg_flops = T * H * FLOPS_PER_TOKEN_HEAD
    achieved_gbs = alg_bytes / (ms * 1e-3) / 1e9
    achieved_tf = alg_flops / (ms * 1e-3) / 1e12
    t_hbm = alg_bytes / (hbm_peak * 1e9)
    t_tc = alg_flops / (tc_peak * 1e12)
    roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved_gbs / hbm_peak, "peak_kind": peak_kind,
                "traffic": recorded_traffic("kda_prefill") if args.case == "full" else None,
                "algorithmic_bytes_per_launch": alg_bytes,
                "tensor_achieved_tflops": achieved_tf, "tensor_peak_tflops": tc_peak,
                "tensor_frac": achieved_tf / tc_peak,
                "frac_of_roofline_time": max(t_hbm, t_tc) / (ms * 1e-3)}

    # ---------------- decode ----------------
    decode = None
    if not args.no_decode:
        wd = synth.workloads()["decode_512x96"]
        n_dec = 64 if small else 512
        dd = synth.make_decode_inputs(n_dec, 96, torch.bfloat16, seed=wd.seed,
                                      state_std=wd.s0_std, device=dev)
        dout = torch.empty_like(dd["q"])

        def dstep():
            kda.decode_step(dd["q"], dd["k"], dd["v"], dd["log_alpha"], dd["beta"],
                            dd["state"], out=dout)

        for _ in range(args.warmup):
            dstep()
        barrier(world)
        dms = time_device(dstep, args.steps, stream)
        dms = max_over_ranks(dms, world)
        dunits = n_dec * 96
        dbytes = dunits * (2 * STATE_BYTES + BYTES_PER_TOKEN_HEAD)
        dgbs = dbytes / (dms * 1e-3) / 1e9
        decode = {"metric": "decode state-update GB/s", "value": dgbs * world, "unit": "GB/s",
                  "ms_per_step": dms, "workload": wd.name,
                  "roofline": {"bound": "hbm", "achieved": dgbs, "peak": hbm_peak,
                               "unit": "GB/s", "frac": dgbs / hbm_peak,
                               "peak_kind": peak_kind,
                               "traffic": (recorded_traffic("kda_decode")
                                           if args.case == "full" else None),
                               "algorithmic_bytes_per_launch": dbytes}}
        # speculative-decoding window: runs of 4 tokens per sequence (accepted replay, bonus,
        # draft), 2 of them committed; the state crosses HBM once each way
        run, keep = 4, 2
        xw = synth.make_inputs([run] * n_dec, 96, torch.bfloat16, seed=wd.seed, s0_std=wd.s0_std,
                               device=dev)
        wstate = xw["init_state"]
        wout = torch.empty_like(xw["q"])
        wcommit = torch.full((n_dec,), keep, dtype=torch.int32, device=dev)

        def wstep():
            kda.decode_window(xw["q"], xw["k"], xw["v"], xw["log_alpha"], xw["beta"],
                              xw["cu_seqlens"], xw["seqlens"], wstate, commit=wcommit, out=wout)

        for _ in range(args.warmup):
            wstep()
        barrier(world)
        wms = max_over_ranks(time_device(wstep, args.steps, stream), world)
        wbytes = dunits * (2 * STATE_BYTES + run * BYTES_PER_TOKEN_HEAD)
        decode["window"] = {"workload": f"{n_dec} sequences x 96 heads, runs of {run} tokens, "
                                        f"{keep} committed", "ms_per_step": wms,
                            "tokens_per_s": n_dec * run * world / (wms * 1e-3),
                            "hbm_gbs": wbytes / (wms * 1e-3) / 1e9,
                            "hbm_frac": wbytes / (wms * 1e-3) / 1e9 / hbm_peak}
        # the same step and window on raw projections, the input prologue fused into the kernels
        xp = synth.make_raw_inputs([1] * n_dec, 96, seed=wd.seed, s0_std=None, device=dev)
        xpw = synth.make_raw_inputs([run] * n_dec, 96, seed=wd.seed, s0_std=None, device=dev)
        praw = lambda z: (z["q_raw"], z["k_raw"], z["v_raw"], z["g_raw"], z["beta_logit"])

        def pstep():
            kda.decode_step_prologue(*praw(xp), dd["state"], xp["A_log"], xp["dt_bias"], out=dout)

        def pwstep():
            kda.decode_window_prologue(*praw(xpw), xpw["cu_seqlens"], xpw["seqlens"], wstate,
                                       xpw["A_log"], xpw["dt_bias"], commit=wcommit, out=wout)

        def ustep():  # unfused: the prologue pass, then the plain step
            q_, k_, v_, g_, b_ = kda.prologue(*praw(xp), xp["A_log"], xp["dt_bias"])
            kda.decode_step(q_, k_, v_, g_, b_, dd["state"], out=dout)

        def uwstep():
            q_, k_, v_, g_, b_ = kda.prologue(*praw(xpw), xpw["A_log"], xpw["dt_bias"])
            kda.decode_window(q_, k_, v_, g_, b_, xpw["cu_seqlens"], xpw["seqlens"], wstate,
                              commit=wcommit, out=wout)

        ptimes = {}
        for name, fn in (("step", pstep), ("window", pwstep), ("step_unfused", ustep),
                         ("window_unfused", uwstep)):
            for _ in range(args.warmup):
                fn()
            barrier(world)
            ptimes[name] = max_over_ranks(time_device(fn, args.steps, stream), world)
        decode["prologue"] = {
            "workload": "the same step and window on raw projections (prologue fused)",
            "step_ms": ptimes["step"], "step_hbm_gbs": dbytes / (ptimes["step"] * 1e-3) / 1e9,
            "window_ms": ptimes["window"],
            "window_hbm_gbs": wbytes / (ptimes["window"] * 1e-3) / 1e9,
            "unfused_step_ms": ptimes["step_unfused"],
            "unfused_window_ms": ptimes["window_unfused"]}
        del xw, wstate, wout, wcommit, xp, xpw, dd, dout

    # ---------------- the other prefill workloads (reported, not the headline) ------------
    extra = None
    if not args.no_extra:
        extra = {}
        for key in ("long_256k", "varlen_64"):
            we = synth.workloads()[key]
            xe = synth.make_workload(we, device=dev)
            oute = torch.empty_like(xe["q"])
            fine = torch.empty((len(we.lengths), we.heads, D, D), dtype=torch.float32, device=dev)
            wse = torch.empty(max(1, kda.fwd_workspace_bytes(xe["seqlens"], we.heads)),
                              dtype=torch.uint8, device=dev)

            def estep_x():
                kda.fwd_chunked(xe["q"], xe["k"], xe["v"], xe["log_alpha"], xe["beta"],
                                xe["cu_seqlens"], xe["seqlens"], init_state=xe["init_state"],
                                out=oute, final_state=fine, workspace=wse)

            for _ in range(2):
                estep_x()
            k_x = max(2, min(args.steps, 5))
            ms_x = max_over_ranks(time_device(estep_x, k_x, stream), world)
            Tx = xe["q"].shape[0]
            bytes_x = Tx * we.heads * BYTES_PER_TOKEN_HEAD + len(we.lengths) * we.heads * 2 * STATE_BYTES
            extra[key] = {"workload": we.name, "tokens": Tx, "ms_per_step": ms_x, "steps": k_x,
                          "value": Tx * world / (ms_x * 1e-3) / 1e6, "unit": "Mtokens/s",
                          "hbm_frac_of_roofline": bytes_x / (ms_x * 1e-3) / 1e9 / hbm_peak,
                          "plan": kda.fwd_plan(xe["seqlens"], we.heads)}
            del xe, oute, fine, wse
        # the headline prefill with a state checkpoint every 512 tokens (prefix-cache use)
        every = 512
        ckpts = torch.empty((kda.fwd_checkpoint_count(x["seqlens"], H, every), H, D, D),
                            dtype=torch.float32, device=dev)

        def estep_ck():
            kda.fwd_chunked_checkpoints(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                        x["cu_seqlens"], x["seqlens"], every,
                                        init_state=x["init_state"], out=out, final_state=fin,
                                        checkpoints=ckpts)

        for _ in range(2):
            estep_ck()
        k_c = max(2, min(args.steps, 10))
        ms_c = max_over_ranks(time_device(estep_ck, k_c, stream), world)
        extra["prefill_4x8k_ckpt512"] = {
            "workload": w.name + " + state checkpoint every 512 tokens", "tokens": T,
            "checkpoints": int(ckpts.shape[0]) * H, "ms_per_step": ms_c, "steps": k_c,
            "value": T * world / (ms_c * 1e-3) / 1e6, "unit": "Mtokens/s",
            "overhead_vs_plain": ms_c / ms_max - 1.0}
        del ckpts
        # the headline shape with the bounded gate's whole range (log alpha = -5 sigmoid(2 z),
        # mean -2.5): blocks run as shorter decay windows
        xb = synth.make_inputs(w.lengths, H, w.dtype, w.seed, s0_std=w.s0_std, device=dev,
                               bounded_gate=-5.0)

        def estep_bg():
            kda.fwd_chunked(xb["q"], xb["k"], xb["v"], xb["log_alpha"], xb["beta"],
                            xb["cu_seqlens"], xb["seqlens"], init_state=xb["init_state"], out=out,
                            final_state=fin)

        for _ in range(2):
            estep_bg()
        k_b = max(2, min(args.steps, 10))
        ms_bg = max_over_ranks(time_device(estep_bg, k_b, stream), world)
        extra["prefill_4x8k_bounded_gate"] = {
            "workload": w.name + " with log alpha = -5 sigmoid(2 z) (the bounded gate's range)",
            "tokens": T, "ms_per_step": ms_bg, "steps": k_b,
            "value": T * world / (ms_bg * 1e-3) / 1e6, "unit": "Mtokens/s",
            "slowdown_vs_plain": ms_bg / ms_max}
        del xb

    if not args.no_extra or args.case == "small_prologue":
        extra = {} if extra is None else extra
        # the headline prefill on raw projections: the input prologue fused into the kernel,
        # against the unfused pipeline (the standalone prologue pass, then the plain prefill).
        # The gate's bias is centred at -6, which keeps log alpha near zero (a few hundredths per
        # token, the decay range of the plain workload), so that the figure is the prologue's own
        # cost; the unbiased recipe (log alpha across the whole range) is timed after it.
        xr = synth.make_raw_inputs(x["seqlens"], H, seed=w.seed, s0_std=w.s0_std, device=dev,
                                   dt_center=-6.0)
        raw = (xr["q_raw"], xr["k_raw"], xr["v_raw"], xr["g_raw"], xr["beta_logit"])

        def estep_pf():
            kda.fwd_chunked_prologue(*raw, xr["cu_seqlens"], xr["seqlens"], xr["A_log"],
                                     xr["dt_bias"], init_state=xr["init_state"], out=out,
                                     final_state=fin)

        def estep_pp():
            return kda.prologue(*raw, xr["A_log"], xr["dt_bias"])

        def estep_pu():
            q_, k_, v_, g_, b_ = estep_pp()
            kda.fwd_chunked(q_, k_, v_, g_, b_, xr["cu_seqlens"], xr["seqlens"],
                            init_state=xr["init_state"], out=out, final_state=fin)

        gen_w = torch.Generator(device=dev).manual_seed(w.seed)
        conv_w = [torch.randn(H, D, 4, generator=gen_w, device=dev) * 0.5 for _ in range(3)]
        conv_cache = torch.zeros(len(w.lengths), 3, 3, H, D, dtype=torch.bfloat16, device=dev)

        def estep_pc():  # the short convolution and the prologue, cache updated in place
            return kda.prologue_conv(*raw, xr["cu_seqlens"], xr["seqlens"], xr["A_log"], *conv_w,
                                     dt_bias=xr["dt_bias"], cache_in=conv_cache,
                                     cache_out=conv_cache)

        k_p = max(2, min(args.steps, 10))
        times = {}
        for name, fn in (("fused", estep_pf), ("unfused", estep_pu), ("prologue", estep_pp),
                         ("prologue_conv", estep_pc)):
            for _ in range(2):
                fn()
            times[name] = max_over_ranks(time_device(fn, k_p, stream), world)
        pro_bytes = T * H * 2 * (4 * D * 2 + 2)  # raw in, transformed out (bf16)
        extra["prefill_4x8k_prologue"] = {
            "workload": w.name + " on raw projections (Swish, L2 norm, bounded gate, sigmoid)",
            "tokens": T, "ms_per_step": times["fused"], "steps": k_p,
            "value": T * world / (times["fused"] * 1e-3) / 1e6, "unit": "Mtokens/s",
            "unfused_ms_per_step": times["unfused"],
            "fused_saving_vs_unfused": 1.0 - times["fused"] / times["unfused"],
            "overhead_vs_plain": times["fused"] / ms_max - 1.0,
            "prologue_kernel_ms": times["prologue"],
            "prologue_kernel_hbm_frac": pro_bytes / (times["prologue"] * 1e-3) / 1e9 / hbm_peak,
            "prologue_conv_ms": times["prologue_conv"],
            "prologue_conv_hbm_frac": pro_bytes / (times["prologue_conv"] * 1e-3) / 1e9 / hbm_peak}
        xu = synth.make_raw_inputs(x["seqlens"], H, seed=w.seed, s0_std=w.s0_std, device=dev)
        raw_u = (xu["q_raw"], xu["k_raw"], xu["v_raw"], xu["g_raw"], xu["beta_logit"])

        def estep_pfu():
            kda.fwd_chunked_prologue(*raw_u, xu["cu_seqlens"], xu["seqlens"], xu["A_log"],
                                     xu["dt_bias"], init_state=xu["init_state"], out=out,
                                     final_state=fin)

        for _ in range(2):
            estep_pfu()
        ms_pfu = max_over_ranks(time_device(estep_pfu, k_p, stream), world)
        extra["prefill_4x8k_prologue"]["unbiased_gate_ms_per_step"] = ms_pfu
        extra["prefill_4x8k_prologue"]["unbiased_gate_value"] = T * world / (ms_pfu * 1e-3) / 1e6
        del xr, raw, conv_w, conv_cache, xu, raw_u

    # ---------------- backward (gradients) on the headline workload ----------------
    if not args.no_extra or args.case == "small":
        extra = {} if extra is None else extra
        gen_b = torch.Generator(device=dev).manual_seed(w.seed)
        d_out = torch.randn(T, H, D, generator=gen_b, device=dev)
        bws = torch.empty(max(16, kda.binding.load_library().kda_bwd_workspace_bytes(
            ctypes.byref(kda.binding.make_desc(x["seqlens"], H, x["q"].dtype)))),
            dtype=torch.uint8, device=dev)

        def bstep():
            return kda.bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["cu_seqlens"],
                           x["seqlens"], d_out, init_state=x["init_state"], workspace=bws)

        bstep()
        ms_b = max_over_ranks(time_device(bstep, 5, stream), world)
        # dense tf32 products per 16-token chunk and head, in multiply-adds: prep 2 x 16*16*128;
        # forward chain 2 x 16*128*128 + 16*16*128; reverse 6 x 16*128*128 + 10 x 16*16*128
        chunks = sum((n + 15) // 16 for n in x["seqlens"])
        flops_b = 2.0 * chunks * H * (8 * 16 * 128 * 128 + 13 * 16 * 16 * 128)
        extra["backward_4x8k" if not small else "backward_small"] = {
            "workload": w.name + ": gradients of q, k, v, log alpha, beta and the initial state",
            "tokens": T, "ms_per_step": ms_b, "steps": 5,
            "value": T * world / (ms_b * 1e-3) / 1e6, "unit": "Mtokens/s",
            "algorithmic_tflop_per_step": flops_b / 1e12,
            "tensor_tflops": flops_b / (ms_b * 1e-3) / 1e12,
            "kernels": "index, prep (chunk-parallel), forward chain, reverse chain (one CTA per unit)",
            "workspace_bytes": int(bws.numel())}
        del d_out, bws

    # ---------------- end to end (host buffers, copies inside the timed region) ------------
    e2e = None
    if not args.no_e2e:
        names = ("q", "k", "v", "log_alpha", "beta")
        host = {nm: x[nm].cpu().pin_memory() for nm in names}
        host["init_state"] = x["init_state"].cpu().pin_memory()
        host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        host_fin = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = host_out.numel() * host_out.element_size() + host_fin.numel() * 4

        parts = 8
        # every part's cumulative lengths (N + 1 int32; every sequence spans every part here)
        h2d += 4 * parts * (len(x["seqlens"]) + 1)
        e_ws = torch.empty(kda.fwd_host_workspace_bytes(x["seqlens"], H, x["q"].dtype, parts),
                           dtype=torch.uint8, device=dev)

        def estep():
            # the C-ABI host-buffer call: uploads, kernels and downloads overlapped by part
            kda.fwd_chunked_host(host["q"], host["k"], host["v"], host["log_alpha"], host["beta"],
                                 x["seqlens"], init_state=host["init_state"], out=host_out,
                                 final_state=host_fin, parts=parts, workspace=e_ws)

        for _ in range(2):
            estep()
        barrier(world)
        esteps = max(3, min(args.steps, 5))
        ems = max_over_ranks(time_device(estep, esteps, stream), world)
        e2e = {"value": tokens_all / (ems * 1e-3) / 1e6, "unit": "Mtokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ems,
               "steps": esteps, "api": "kda_fwd_chunked_host", "parts": parts,
               "workspace_bytes": int(e_ws.numel())}
        del e_ws

    # ---------------- CPU baseline (oracle, rank 0 only, N = 1 only) ----------------
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = cpu_cores()
        xs = synth.make_workload(w, device="cpu")
        # passes over the sample until about 10 s of CPU work (at most 20 passes)
        runs = []
        while sum(t for t, _ in runs) < 10.0 and len(runs) < 20:
            runs.append(oracle_sample(xs, args.cpu_baseline_tokens, threads))
        sec = sum(t for t, _ in runs)
        cpu_base = {"value": sum(n for _, n in runs) / sec / 1e6, "unit": "Mtokens/s",
                    "cores": threads, "kind": "oracle", "seconds": sec, "passes": len(runs),
                    "sample": sample_text(xs, args.cpu_baseline_tokens, H)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "Mtokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "global_batch": len(w.lengths) * world,
                       "seq_len": w.lengths[0], "heads": H, "d_k": D, "d_v": D,
                       "chunk": CHUNK, "state": "fp32",
                       "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (%.2f GB read per step)" % (alg_bytes / 1e9)},
            "roofline": roofline, "cpu_baseline": cpu_base, "e2e": e2e,
            "clocks": getattr(clk, "result", None), "gpu_launches": launches,
            "decode": decode, "other_prefill_workloads": extra,
        }
        print(json.dumps(line), flush=True)
    barrier(world)


if __name__ == "__main__":
    main()
