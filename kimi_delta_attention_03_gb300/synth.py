"""Seeded synthetic inputs for the KDA forward workloads.

This module holds the input recipes only — random draws, the per-(token, head) L2
normalisation of q and k that the KDA layer applies before the operator, and the gate and
write-strength squashing that produce log-alpha and beta.  It contains none of the
recurrence's arithmetic.  Both the CUDA path (tests, bench) and the fp64 oracle receive the
exact tensors it returns, so the two sides never draw their own inputs.

Recipe (same for every workload, "Kimi K3" on ai.thesatyajit.com, section "Kimi Delta
Attention": q and k are L2-normalised per head; alpha in (0,1)^{d_k}; beta in (0,1)):
  draw order q, k, v, beta-logit, gate-noise, S0 from one torch.Generator(seed);
  q, k ~ N(0,1), L2-normalised over the d_k channels of each (token, head); q *= 1/sqrt(d_k)
  v ~ N(0,1);  beta = sigmoid(N(0,1));  log_alpha = -softplus(N(0,1)) * gate_scale
  S0 ~ N(0, s0_std^2) per entry (zeros when s0_std is None).
With ``bounded_gate=lb`` the gate instead spans K3's whole bounded range: log_alpha =
lb * sigmoid(2 N(0,1)) lies in (lb, 0) with mean lb / 2 ("How Kimi K3 Engineered Its Way to the
Frontier", section "How KDA updates its state": the gate is a lower bound times a sigmoid).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch
import torch.nn.functional as F

D_K = 128
D_V = 128


@dataclass(frozen=True)
class Workload:
    """One named workload.  ``lengths`` are the packed sequence lengths."""
    name: str
    lengths: tuple
    heads: int
    dtype: torch.dtype
    seed: int
    gate_scale: float = 0.1
    s0_std: float | None = 0.01
    decode: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))


def loguniform_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    """Sequence lengths floor(exp(U(ln lo, ln hi))), drawn on the CPU from ``seed``."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    u = torch.rand(n, generator=gen, dtype=torch.float64)
    lens = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    return tuple(int(x) for x in lens.clamp(lo, hi).tolist())


def workloads() -> dict:
    """The five workloads of this project, by name."""
    return {
        "tiny_fp32": Workload("tiny_fp32 (B=1, H=2, T=256, fp32)", (256,), 2, torch.float32,
                              seed=0, s0_std=None),
        "prefill_4x8k": Workload("prefill_4x8k (B=4, T=8192, H=32, bf16)", (8192,) * 4, 32,
                                 torch.bfloat16, seed=1),
        "long_256k": Workload("long_256k (B=1, T=262144, H=16, bf16, slow decay)", (262144,),
                              16, torch.bfloat16, seed=2, gate_scale=0.02),
        "decode_512x96": Workload("decode_512x96 (N=512, H=96, 1 token, fp32 state)",
                                  (1,) * 512, 96, torch.bfloat16, seed=3, s0_std=0.02,
                                  decode=True),
        "varlen_64": Workload("varlen_64 (64 seqs log-uniform [512, 65536], H=8, bf16)",
                              loguniform_lengths(64, 512, 65536, seed=4), 8, torch.bfloat16,
                              seed=4),
    }


def make_inputs(lengths, heads: int, dtype: torch.dtype, seed: int, gate_scale: float = 0.1,
                s0_std: float | None = 0.01, device="cpu", d_k: int = D_K, d_v: int = D_V,
                zero_length_ok: bool = True, bounded_gate: float | None = None) -> dict:
    """Packed-varlen inputs with layout [T_tot, H, d] (batch folded into tokens).

    Returns a dict with q, k, v, log_alpha ([T,H,d], ``dtype``), beta ([T,H], ``dtype``),
    init_state ([N,H,d_k,d_v] fp32 or None), cu_seqlens (int32 on ``device``) and
    seqlens (python list, the host copy)."""
    lengths = [int(x) for x in lengths]
    if any(x < 0 for x in lengths) or (not zero_length_ok and any(x == 0 for x in lengths)):
        raise ValueError("bad lengths")
    n = len(lengths)
    T = sum(lengths)
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(seed)
    f32 = torch.float32
    q = torch.randn(T, heads, d_k, generator=gen, device=dev, dtype=f32)
    k = torch.randn(T, heads, d_k, generator=gen, device=dev, dtype=f32)
    v = torch.randn(T, heads, d_v, generator=gen, device=dev, dtype=f32)
    b_logit = torch.randn(T, heads, generator=gen, device=dev, dtype=f32)
    g_noise = torch.randn(T, heads, d_k, generator=gen, device=dev, dtype=f32)
    s0 = None
    if s0_std is not None:
        s0 = torch.randn(n, heads, d_k, d_v, generator=gen, device=dev, dtype=f32) * s0_std
    q = F.normalize(q, dim=-1) * (1.0 / math.sqrt(d_k))
    k = F.normalize(k, dim=-1)
    beta = torch.sigmoid(b_logit)
    if bounded_gate is None:
        log_alpha = -F.softplus(g_noise) * gate_scale
    else:
        log_alpha = bounded_gate * torch.sigmoid(2.0 * g_noise)
    cu = torch.zeros(n + 1, dtype=torch.int32)
    if n:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return {
        "q": q.to(dtype).contiguous(), "k": k.to(dtype).contiguous(),
        "v": v.to(dtype).contiguous(), "log_alpha": log_alpha.to(dtype).contiguous(),
        "beta": beta.to(dtype).contiguous(), "init_state": s0,
        "cu_seqlens": cu.to(dev), "seqlens": lengths,
    }


def make_raw_inputs(lengths, heads: int, seed: int, s0_std: float | None = 0.01, device="cpu",
                    dt_center: float = 0.0, d: int = D_K) -> dict:
    """Raw per-token projections for the input prologue, layout [T_tot, H, d], bf16.

    q_raw, k_raw, v_raw, g_raw and beta_logit are N(0, 1) (the short-convolution outputs and
    logits a layer would produce; the sources give no distribution).  A_log ~ 0.25 N(0, 1) per
    head and dt_bias ~ dt_center + N(0, 1) per (head, channel), fp32.  With the default centre
    0 the bounded gate's output spans its whole range (lower_bound, 0) and averages about
    lower_bound / 2 per token.  Also returns init_state, cu_seqlens and seqlens as
    ``make_inputs`` does."""
    lengths = [int(x) for x in lengths]
    if any(x < 0 for x in lengths):
        raise ValueError("bad lengths")
    n, T = len(lengths), sum(lengths)
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(seed)
    f32, bf = torch.float32, torch.bfloat16
    q = torch.randn(T, heads, d, generator=gen, device=dev, dtype=f32)
    k = torch.randn(T, heads, d, generator=gen, device=dev, dtype=f32)
    v = torch.randn(T, heads, d, generator=gen, device=dev, dtype=f32)
    b_logit = torch.randn(T, heads, generator=gen, device=dev, dtype=f32)
    g = torch.randn(T, heads, d, generator=gen, device=dev, dtype=f32)
    A_log = torch.randn(heads, generator=gen, device=dev, dtype=f32) * 0.25
    dt_bias = dt_center + torch.randn(heads, d, generator=gen, device=dev, dtype=f32)
    s0 = None
    if s0_std is not None:
        s0 = torch.randn(n, heads, d, d, generator=gen, device=dev, dtype=f32) * s0_std
    cu = torch.zeros(n + 1, dtype=torch.int32)
    if n:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return {
        "q_raw": q.to(bf).contiguous(), "k_raw": k.to(bf).contiguous(),
        "v_raw": v.to(bf).contiguous(), "g_raw": g.to(bf).contiguous(),
        "beta_logit": b_logit.to(bf).contiguous(), "A_log": A_log.contiguous(),
        "dt_bias": dt_bias.contiguous(), "init_state": s0, "cu_seqlens": cu.to(dev),
        "seqlens": lengths,
    }


def make_workload(w: Workload, device="cpu", heads: int | None = None,
                  lengths=None) -> dict:
    """Inputs of workload ``w`` (optionally with fewer heads or other lengths)."""
    return make_inputs(w.lengths if lengths is None else lengths,
                       w.heads if heads is None else heads, w.dtype, w.seed,
                       gate_scale=w.gate_scale, s0_std=w.s0_std, device=device)


def make_decode_inputs(n: int, heads: int, dtype: torch.dtype, seed: int,
                       state_std: float = 0.02, gate_scale: float = 0.1, device="cpu",
                       d_k: int = D_K, d_v: int = D_V) -> dict:
    """One token per (sequence, head): q, k, v, log_alpha [N,H,d], beta [N,H], state fp32."""
    x = make_inputs([1] * n, heads, dtype, seed, gate_scale=gate_scale, s0_std=state_std,
                    device=device, d_k=d_k, d_v=d_v)
    x["state"] = x.pop("init_state")
    return x
