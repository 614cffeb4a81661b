"""The C-ABI library loads, exports every symbol include/kda.h declares, and its host-side
logic (argument checks, work plan) behaves as documented.  No GPU needed: nothing here
launches a kernel — every call below is rejected or answered on the host."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from kimi_delta_attention_03_gb300 import build, binding
    build.build()
    return binding.load_library()


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(kda_\w+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    from kimi_delta_attention_03_gb300 import binding
    declared = _declared_functions()
    assert declared, "no declarations found"
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
        assert name in binding.SIGNATURES, f"{name} has no binding signature"


def test_version_and_status_strings(lib):
    assert lib.kda_version() >= 1
    assert lib.kda_status_string(0) == b"KDA_OK"
    assert lib.kda_status_string(-6) == b"KDA_ERR_DECAY_RANGE"
    assert lib.kda_status_string(12345) == b"KDA_ERR_UNKNOWN"


def _desc(lens, H=4, dtype=torch.bfloat16, d=128):
    from kimi_delta_attention_03_gb300 import binding
    return binding.make_desc(lens, H, dtype, d)


def test_plan_counts_chunks_per_sequence(lib):
    from kimi_delta_attention_03_gb300 import binding
    lens = [0, 1, 63, 64, 65, 8192, 130]
    info = binding.fwd_plan(lens, 4)
    assert info["chunk_size"] == 64
    assert info["chunks"] == sum((L + 63) // 64 for L in lens)
    assert info["work_items"] >= len(lens)


def test_plan_splits_long_sequences_by_length_only(lib):
    """The segment count is picked among 128-chunk segments and k * 152 / H segments (k = 1, 2,
    3; at least 64 chunks each) by the wave cost seg * (40 ceil(2H(n-1) / 152) + 43 ceil(Hn /
    152)), seg = ceil(chunks / n); segments of seg chunks, the last shorter."""
    from kimi_delta_attention_03_gb300 import binding
    H = 3
    # 1024 chunks: whole.  1025 chunks: n = 9 (128-chunk) costs 114 * 83 = 9462, n = 16 (the cap
    # 1025 // 64) costs 65 * 83 = 5395 -> 16 segments of 65.  4096 chunks: n = 32 costs
    # 128 * 123 = 15744, n = 50 (152 // 3) costs 82 * 123 = 10086, n = 64 (the cap) costs
    # 64 * 206 = 13184 -> segments of 82, 50 of them.
    lens = [65536, 65537, 262144, 5]
    info = binding.fwd_plan(lens, H)
    assert info["segment_chunks"] == 82
    assert info["split_sequences"] == 2
    assert info["work_items"] == 1 + 16 + 50 + 1
    slots = 16 + 50
    assert info["workspace_bytes"] == 3 * slots * H * 128 * 128 * 4
    assert binding.fwd_workspace_bytes(lens, H) == info["workspace_bytes"]
    # the plan of a sequence does not depend on its neighbours
    assert binding.fwd_plan([65537], H)["work_items"] == 16
    assert binding.fwd_plan([65537], H)["segment_chunks"] == 65
    assert binding.fwd_plan([100, 200], H)["workspace_bytes"] == 0
    assert binding.fwd_plan([100, 200], H)["segment_chunks"] == 0
    # 262,144 tokens with 16 heads (the long-sequence workload): 19 segments of 216 chunks
    # (576 + 304 items, about four and two waves), against 32 of 128 (992 + 512)
    info = binding.fwd_plan([262144], 16)
    assert (info["work_items"], info["segment_chunks"]) == (19, 216)


def test_segment_plan_covers_every_sequence_without_empty_segments(lib):
    """For lengths across the split threshold and head counts from 1 to 512: a split sequence has
    at least two segments of at least 64 chunks, the segments cover its chunks with a non-empty
    last one ((n - 1) * seg < chunks <= n * seg), and its plan is the same packed with others."""
    from kimi_delta_attention_03_gb300 import binding
    lengths = [65536, 65537, 65600, 70000, 100000, 131072, 262144, 262145, 400000, 1048576,
               3_000_000]
    for H in (1, 2, 3, 8, 16, 32, 64, 96, 152, 153, 512):
        for L in lengths:
            info = binding.fwd_plan([L], H)
            chunks = (L + 63) // 64
            n, seg = info["work_items"], info["segment_chunks"]
            if chunks <= 1024:
                assert (n, seg, info["split_sequences"]) == (1, 0, 0)
                continue
            assert info["split_sequences"] == 1 and n >= 2 and seg >= 64, (L, H, n, seg)
            assert (n - 1) * seg < chunks <= n * seg, (L, H, n, seg)
            assert info["workspace_bytes"] == 3 * n * H * 128 * 128 * 4
        packed = binding.fwd_plan([5] + lengths + [7], H)
        alone = sum(binding.fwd_plan([L], H)["work_items"] for L in lengths)
        assert packed["work_items"] == alone + 2


def test_checkpoint_count(lib):
    from kimi_delta_attention_03_gb300 import binding
    lens = [0, 63, 64, 511, 512, 1000, 1024]
    assert binding.fwd_checkpoint_count(lens, 2, 512) == 0 + 0 + 0 + 0 + 1 + 1 + 2
    assert binding.fwd_checkpoint_count(lens, 2, 64) == 0 + 0 + 1 + 7 + 8 + 15 + 16
    desc = binding.make_desc(lens, 2, torch.bfloat16)
    for bad in (0, -64, 100, 32):  # a positive multiple of the 64-token chunk only
        assert lib.kda_fwd_checkpoint_count(ctypes.byref(desc), bad) == -1


def test_host_argument_checks(lib):
    from kimi_delta_attention_03_gb300 import binding
    P = ctypes.c_void_p
    fake = P(0x1000)
    st = lambda d, **kw: lib.kda_fwd_chunked(
        ctypes.byref(d), kw.get("q", fake), fake, fake, fake, fake, None, fake,
        kw.get("out", P(0x2000)), None, None, 0, None)
    assert st(_desc([4, 5], d=64)) == -2                    # unsupported head dim
    assert st(_desc([4, 5], dtype=torch.float16)) == -2     # unsupported dtype
    d = _desc([4, 5])
    d.total_tokens = 10
    assert st(d) == -1                                      # lengths do not sum to T_tot
    assert st(_desc([4, -1])) == -1                         # negative length
    assert st(_desc([4, 5]), q=None) == -1                  # null input
    assert st(_desc([4, 5]), out=fake) == -1                # out aliases an input
    assert lib.kda_fwd_plan(None, None) == -1
    assert lib.kda_fwd_workspace_bytes(None) == 0
    # decode: total_tokens must equal num_seqs, every host length must be 1
    dd = _desc([1, 1, 1])
    dd.total_tokens = 4
    assert lib.kda_decode_step(ctypes.byref(dd), fake, fake, fake, fake, fake, P(0x3000),
                               P(0x2000), None) == -1
    dd = _desc([1, 2])
    dd.total_tokens = 2
    assert lib.kda_decode_step(ctypes.byref(dd), fake, fake, fake, fake, fake, P(0x3000),
                               P(0x2000), None) == -1


def test_host_call_workspace_and_checks(lib):
    """kda_fwd_host_workspace_bytes: states, every part's cumulative lengths and three slots of
    the largest part; kda_fwd_chunked_host's host-side rejections (no CUDA call is reached)."""
    P = ctypes.c_void_p
    fake = P(0x1000)
    size = lambda d, parts: lib.kda_fwd_host_workspace_bytes(ctypes.byref(d), parts)
    # 4 x 8192 tokens, 32 heads, 8 parts: the last part holds 1/32 of the tokens (256 per
    # sequence) and the first seven share the rest, rounded up to chunks: boundaries 1152, 2304,
    # 3456, 4544, 5696, 6848, 7936, so the largest part has 4 x 1,152 rows
    d = _desc([8192] * 4, H=32)
    row = 32 * 128 * 2
    slot = 5 * 4608 * row + 4608 * 32 * 2
    assert size(d, 8) == 4 * 32 * 65536 + 256 + 3 * slot
    assert size(d, 0) == size(d, 8)
    assert size(d, 1) == 4 * 32 * 65536 + 256 + 3 * (5 * 32768 * row + 32768 * 32 * 2)
    # one part asked for, but no part spans more than 65,536 tokens of a sequence:
    # parts [0, 65536) and [65536, 70000), the first with 65,636 rows
    d2 = _desc([70000, 100], H=1)
    assert size(d2, 1) == 2 * 65536 + 256 + 3 * (5 * 65636 * 256 + 131328)
    assert size(_desc([4, 5]), -1) == 0 and size(_desc([4, 5]), 65) == 0
    assert lib.kda_fwd_host_workspace_bytes(None, 0) == 0

    def call(d, ws, nbytes, parts=0, out=P(0x2000)):
        return lib.kda_fwd_chunked_host(ctypes.byref(d), fake, fake, fake, fake, fake, None, out,
                                        None, parts, ws, nbytes, None)
    big = 1 << 30
    assert call(_desc([4, 5]), None, 0) == -3                    # no workspace
    assert call(_desc([4, 5]), P(0x100100), 16) == -3            # workspace too small
    assert call(_desc([4, 5]), P(0x100101), big) == -3           # workspace misaligned
    assert call(_desc([4, 5]), P(0x100100), big, parts=65) == -1  # too many parts
    assert call(_desc([4, 5]), P(0x100100), big, out=fake) == -1  # out aliases an input
    assert call(_desc([4, 5], d=64), P(0x100100), big) == -1     # unsupported head dim


def test_checkpoint_and_window_argument_checks(lib):
    # refused on the host before any device pointer is touched
    P = ctypes.c_void_p
    fake = P(0x1000)
    ck = lambda d, every, states=P(0x4000): lib.kda_fwd_chunked_ckpt(
        ctypes.byref(d), fake, fake, fake, fake, fake, None, fake, P(0x2000), None, every,
        states, None, 0, None)
    assert ck(_desc([512, 100]), 0) == -1                       # no interval
    assert ck(_desc([512, 100]), 100) == -1                     # not a multiple of 64
    assert ck(_desc([512, 100], dtype=torch.float32), 256) == -2  # bf16 only
    assert ck(_desc([512, 100]), 256, states=None) == -1        # checkpoints but no buffer
    assert ck(_desc([512, 100]), 256, states=fake) == -1        # buffer aliases an input
    win = lambda d, state=P(0x3000): lib.kda_decode_window(
        ctypes.byref(d), fake, fake, fake, fake, fake, fake, state, P(0x2000), None, None)
    assert win(_desc([4, 65])) == -1                            # runs of at most 64 tokens
    assert win(_desc([4, 5]), state=None) == -1                 # no state
    d = _desc([4, 5])
    d.host_seqlens = None
    assert win(d) == -1                                         # run lengths are required


def test_prologue_argument_checks(lib):
    from kimi_delta_attention_03_gb300.binding import KdaPrologueParams
    P = ctypes.c_void_p
    fake, fake2 = P(0x1000), P(0x5000)
    ok = dict(A_log=0x7000, dt_bias=None, lower_bound=-5.0, q_scale=0.125)

    def prm(**kw):
        a = dict(ok, **kw)
        return KdaPrologueParams(a["A_log"], a["dt_bias"], a["lower_bound"], a["q_scale"])

    def fused(d, p):
        return lib.kda_fwd_chunked_prologue(ctypes.byref(d), p, fake, fake, fake, fake, fake,
                                            None, fake, P(0x2000), None, None, 0, None)
    d = _desc([128, 64])
    assert fused(d, None) == -1                                          # no parameters
    assert fused(d, ctypes.byref(prm(A_log=None))) == -1                 # no A_log
    assert fused(d, ctypes.byref(prm(dt_bias=0x7004))) == -1             # misaligned dt_bias
    assert fused(d, ctypes.byref(prm(lower_bound=0.0))) == -1            # bound must be < 0
    assert fused(d, ctypes.byref(prm(lower_bound=-100.0))) == -1         # beyond the range
    assert fused(d, ctypes.byref(prm(lower_bound=float("nan")))) == -1
    assert fused(d, ctypes.byref(prm(q_scale=0.0))) == -1
    assert fused(d, ctypes.byref(prm(q_scale=float("inf")))) == -1
    assert fused(_desc([128, 64], dtype=torch.float32), ctypes.byref(prm())) == -2  # bf16 only

    def alone(d, p, outs=(0x2000, 0x2400, 0x2800, 0x2c00, 0x3000), ins=None):
        ins = ins or (0x1000, 0x1400, 0x1800, 0x1c00, 0x2000 - 0x100)
        return lib.kda_prologue(ctypes.byref(d), p, *[P(x) for x in ins],
                                *[None if x is None else P(x) for x in outs], None)
    p = ctypes.byref(prm())
    assert alone(_desc([64]), None) == -1
    assert alone(_desc([64]), p, outs=(0x1000, 0x2400, 0x2800, 0x2c00, 0x3000)) == -1  # aliases
    assert alone(_desc([64]), p, outs=(0x2000, 0x2000, 0x2800, 0x2c00, 0x3000)) == -1  # repeats
    assert alone(_desc([64]), p, outs=(0x2000, 0x2400, None, 0x2c00, 0x3000)) == -1    # missing
    assert alone(_desc([64]), p, outs=(0x2008, 0x2400, 0x2800, 0x2c00, 0x3000)) == -1  # unaligned
    assert alone(_desc([64], dtype=torch.float32), p) == -2
    assert alone(_desc([0]), p) == 0                     # nothing to do: no launch, no error
    # decode step and window on raw projections
    step = lambda d, pp: lib.kda_decode_step_prologue(ctypes.byref(d), pp, fake, fake, fake, fake,
                                                       fake, P(0x3000), P(0x2000), None)
    assert step(_desc([1, 1]), None) == -1
    assert step(_desc([1, 1]), ctypes.byref(prm(q_scale=-1.0))) == -1
    assert step(_desc([1, 1], dtype=torch.float32), ctypes.byref(prm())) == -2
    assert lib.kda_decode_step_prologue(ctypes.byref(_desc([1, 1])), ctypes.byref(prm()),
                                        P(0x1008), fake, fake, fake, fake, P(0x3000), P(0x2000),
                                        None) == -1       # q_raw not 16-byte aligned
    win = lambda d, pp: lib.kda_decode_window_prologue(ctypes.byref(d), pp, fake, fake, fake, fake,
                                                        fake, fake, P(0x3000), P(0x2000), None,
                                                        None)
    assert win(_desc([4, 5]), None) == -1
    assert win(_desc([4, 5]), ctypes.byref(prm(lower_bound=1.0))) == -1
    assert win(_desc([4, 5], dtype=torch.float32), ctypes.byref(prm())) == -2
    assert win(_desc([4, 65]), ctypes.byref(prm())) == -1   # runs of at most 64 tokens
    assert lib.kda_decode_window_prologue(ctypes.byref(_desc([4, 5])), ctypes.byref(prm()), fake,
                                          P(0x1004), fake, fake, fake, fake, P(0x3000),
                                          P(0x2000), None, None) == -1  # k_raw not aligned
    # the short convolution in front of the prologue
    from kimi_delta_attention_03_gb300.binding import KdaConvParams
    cv = lambda **kw: KdaConvParams(kw.get("w_q", 0x8000), 0x8400, 0x8800, kw.get("cin", None),
                                    kw.get("cout", None))
    conv = lambda d, pp, c: lib.kda_prologue_conv(
        ctypes.byref(d), pp, c, P(0x9000), P(0x1000), P(0x1400), P(0x1800), P(0x1c00), P(0x1f00),
        P(0x2000), P(0x2400), P(0x2800), P(0x2c00), P(0x3000), None)
    assert conv(_desc([64, 3]), ctypes.byref(prm()), None) == -1              # no conv parameters
    assert conv(_desc([64, 3]), ctypes.byref(prm()), ctypes.byref(cv(w_q=None))) == -1
    assert conv(_desc([64, 3]), ctypes.byref(prm()), ctypes.byref(cv(w_q=0x8004))) == -1  # unaligned
    assert conv(_desc([64, 3]), ctypes.byref(prm()), ctypes.byref(cv(cout=0x1000))) == -1  # aliases
    assert conv(_desc([64, 3], dtype=torch.float32), ctypes.byref(prm()), ctypes.byref(cv())) == -2
    d = _desc([64, 3])
    d.host_seqlens = None
    assert conv(d, ctypes.byref(prm()), ctypes.byref(cv())) == -1             # lengths required


def test_binding_refuses_cpu_tensors(lib):
    import kimi_delta_attention_03_gb300 as kda
    x = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kda.fwd_chunked(x, x, x, x, torch.zeros(4, 2, dtype=torch.bfloat16),
                        torch.tensor([0, 4], dtype=torch.int32), [4])


def test_backward_host_checks(lib):
    """The backward's workspace size and the argument checks it makes before any launch."""
    from kimi_delta_attention_03_gb300 import binding
    P = ctypes.c_void_p
    lens, H = [0, 5, 33, 2048], 3
    desc = binding.make_desc(lens, H, torch.bfloat16)
    # the sequences' chunk offsets and a stop flag (rounded up to 64 entries), then per 16-token
    # chunk and head the tiles T, P, At (16 x 16 each), the chunk's start state (128 x 128) and
    # its R = V - K_f S (16 x 128), all 4-byte words
    chunks = sum((n + 15) // 16 for n in lens)
    index = ((len(lens) + 2 + 63) // 64) * 64
    need = lib.kda_bwd_workspace_bytes(ctypes.byref(desc))
    assert need == (index + chunks * H * (3 * 16 * 16 + 128 * 128 + 16 * 128)) * 4
    assert lib.kda_bwd_workspace_bytes(None) == 0
    ins = [P(0x1000 + 0x100 * i) for i in range(5)]          # q, k, v, log_alpha, beta
    cu, d_out = P(0x2000), P(0x2100)
    outs = [P(0x3000 + 0x100 * i) for i in range(6)]          # dq, dk, dv, dg, dbeta, dinit
    ws = P(0x10000)

    def call(outs=outs, ws=ws, ws_bytes=need, d_out=d_out):
        return lib.kda_bwd(ctypes.byref(desc), *ins, None, cu, d_out, None, *outs, ws,
                           ws_bytes, None)
    assert call(outs=outs[:5] + [None]) == -1                 # no initial-state gradient buffer
    assert call(outs=[ins[0]] + outs[1:]) == -1               # dq aliases q
    assert call(outs=[outs[0], outs[0]] + outs[2:]) == -1     # two outputs alias
    assert call(d_out=None) == -1                             # no output gradient
    assert call(outs=[P(0x3004)] + outs[1:]) == -1            # output not 16-byte aligned
    assert lib.kda_bwd(ctypes.byref(desc), P(0x1008), *ins[1:], None, cu, d_out, None, *outs, ws,
                       need, None) == -1                      # q not 16-byte aligned
    assert call(ws_bytes=need - 1) == -3                      # workspace too small
    assert call(ws=None) == -3                                # no workspace
    assert call(ws=P(0x10008)) == -3                          # workspace not 16-byte aligned
