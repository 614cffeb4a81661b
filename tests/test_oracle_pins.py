"""Pins of the fp64 oracle against what the pages and the mathematics fix.

The pages print no KDA output values, so the oracle is pinned by exact rational brute force
of the closed form, by special cases that reduce to textbook operators, by invariants, and
by structural facts the pages state.  Each test names the passage it rests on.  A plausible
slip in the oracle (a dropped term, a wrong sign, decay applied after the erase, a transposed
state, an off-by-one in the sequence walk) fails at least one of them; see
``test_planted_mistakes_are_caught``.
"""
import json
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------------------
# exact rational brute force of the closed form (T <= 8, d = 4)
# --------------------------------------------------------------------------------------
def _fmat_mul(a, b):
    n, m, p = len(a), len(b), len(b[0])
    return [[sum((a[i][x] * b[x][j] for x in range(m)), Fraction(0)) for j in range(p)]
            for i in range(n)]


def _fmat_add(a, b):
    return [[a[i][j] + b[i][j] for j in range(len(a[0]))] for i in range(len(a))]


def _eye(d):
    return [[Fraction(int(i == j)) for j in range(d)] for i in range(d)]


def _transition(alpha, beta, k):
    """M_t = (I - beta k k^T) Diag(alpha): the report's KDA transition ("How Kimi K3 Engineered
    Its Way to the Frontier", section "How KDA updates its state")."""
    d = len(k)
    m = [[(Fraction(int(i == j)) - beta * k[i] * k[j]) for j in range(d)] for i in range(d)]
    return [[m[i][j] * alpha[j] for j in range(d)] for i in range(d)]


def brute_force(alphas, betas, ks, vs, qs, s0):
    """S_t = (prod_{s=t..1} M_s) S0 + sum_j (prod_{s=t..j+1} M_s) beta_j k_j v_j^T, exactly;
    o_t = S_t^T q_t.  Products of transition matrices are expanded term by term."""
    T, d = len(ks), len(ks[0])
    Ms = [_transition(alphas[t], betas[t], ks[t]) for t in range(T)]
    outs, S_t = [], None
    for t in range(T):
        prod = _eye(d)
        for s in range(t, -1, -1):          # M_t M_{t-1} ... M_0
            prod = _fmat_mul(prod, Ms[s])
        S_t = _fmat_mul(prod, s0)
        for j in range(t + 1):
            pj = _eye(d)
            for s in range(t, j, -1):       # M_t ... M_{j+1}
                pj = _fmat_mul(pj, Ms[s])
            w = [[betas[j] * ks[j][a] * vs[j][b] for b in range(len(vs[j]))] for a in range(d)]
            S_t = _fmat_add(S_t, _fmat_mul(pj, w))
        outs.append([sum((S_t[a][b] * qs[t][a] for a in range(d)), Fraction(0))
                     for b in range(len(S_t[0]))])
    return outs, S_t


def _rational_case(seed, T, d=4, dv=4):
    r = random.Random(seed)
    vec = lambda n: [Fraction(r.randint(-8, 8), 8) for _ in range(n)]
    alphas = [[Fraction(r.randint(1, 15), 16) for _ in range(d)] for _ in range(T)]
    betas = [Fraction(r.randint(1, 7), 8) for _ in range(T)]
    ks, vs, qs = [vec(d) for _ in range(T)], [vec(dv) for _ in range(T)], [vec(d) for _ in range(T)]
    s0 = [vec(dv) for _ in range(d)]
    return alphas, betas, ks, vs, qs, s0


@pytest.mark.parametrize("seed,T", [(1, 1), (2, 3), (3, 5), (4, 8), (5, 8)])
def test_P0_exact_rational_brute_force(seed, T):
    alphas, betas, ks, vs, qs, s0 = _rational_case(seed, T)
    exact_o, exact_s = brute_force(alphas, betas, ks, vs, qs, s0)
    f = lambda x: np.array(x, dtype=np.float64)
    q = f(qs)[:, None, :]
    k = f(ks)[:, None, :]
    v = f(vs)[:, None, :]
    g = np.log(f(alphas))[:, None, :]          # log alpha in fp64; alpha itself is rational
    b = f(betas)[:, None]
    o, s = oracle.recurrence(q, k, v, g, b, [0, T], state_in=f(s0)[None, None])
    eo, es = f(exact_o), f(exact_s)
    scale = max(1.0, float(np.abs(eo).max()), float(np.abs(es).max()))
    assert np.abs(o[:, 0, :] - eo).max() <= 1e-12 * scale
    assert np.abs(s[0, 0] - es).max() <= 1e-12 * scale


def test_P0_two_sequences_two_heads_packed():
    """Packing: two sequences and two heads, each unit equal to its own brute force."""
    cases = {(n, h): _rational_case(100 + 10 * n + h, T) for n, T in ((0, 3), (1, 5))
             for h in range(2)}
    lens = [3, 5]
    Ttot, d = sum(lens), 4
    q = np.zeros((Ttot, 2, d)); k = np.zeros_like(q); v = np.zeros_like(q); g = np.zeros_like(q)
    b = np.zeros((Ttot, 2)); s0 = np.zeros((2, 2, d, d))
    exp_o = np.zeros((Ttot, 2, d)); exp_s = np.zeros((2, 2, d, d))
    for (n, h), (al, be, ks, vs, qs, s) in cases.items():
        t0 = sum(lens[:n])
        T = lens[n]
        q[t0:t0 + T, h] = np.array(qs, dtype=float); k[t0:t0 + T, h] = np.array(ks, dtype=float)
        v[t0:t0 + T, h] = np.array(vs, dtype=float); g[t0:t0 + T, h] = np.log(np.array(al, dtype=float))
        b[t0:t0 + T, h] = np.array(be, dtype=float); s0[n, h] = np.array(s, dtype=float)
        eo, es = brute_force(al, be, ks, vs, qs, s)
        exp_o[t0:t0 + T, h] = np.array(eo, dtype=float); exp_s[n, h] = np.array(es, dtype=float)
    o, s = oracle.recurrence(q, k, v, g, b, [0, 3, 8], state_in=s0)
    assert np.abs(o - exp_o).max() <= 1e-12 * max(1.0, np.abs(exp_o).max())
    assert np.abs(s - exp_s).max() <= 1e-12 * max(1.0, np.abs(exp_s).max())


# --------------------------------------------------------------------------------------
# special cases named on the pages
# --------------------------------------------------------------------------------------
def _rand(shape, rng):
    return rng.standard_normal(shape)


def test_P1_beta_zero_freezes_state():
    """alpha = 1 and beta = 0: beta scales both the erase and the write ("How KDA updates its
    state": beta near 0 leaves the value in place), so S_t = S0 and o_t = S0^T q_t."""
    rng = np.random.default_rng(11)
    T, H, d = 37, 3, 16
    q = _rand((T, H, d), rng); k = _rand((T, H, d), rng); v = _rand((T, H, d), rng)
    g = np.zeros((T, H, d)); b = np.zeros((T, H)); s0 = _rand((1, H, d, d), rng)
    o, s = oracle.recurrence(q, k, v, g, b, [0, T], state_in=s0)
    assert np.array_equal(s, s0)
    expect = np.einsum("thi,hij->thj", q, s0[0])
    np.testing.assert_allclose(o, expect, rtol=1e-13, atol=1e-13)


def _orthonormal_keys(T, d, rng):
    qmat, _ = np.linalg.qr(rng.standard_normal((d, d)))
    return qmat[:T]


@pytest.mark.parametrize("general_beta", [False, True])
def test_P2_linear_attention_reduction(general_beta):
    """S0 = 0, alpha = 1, mutually orthonormal keys: the erase term k_t^T S_{t-1} vanishes and
    KDA reads o_t = sum_{i<=t} beta_i (q_t . k_i) v_i — plain linear attention ("How linear
    attention works without a cache") when beta = 1."""
    rng = np.random.default_rng(12 + general_beta)
    T, d = 96, 128
    k = _orthonormal_keys(T, d, rng)[:, None, :]
    q = _rand((T, 1, d), rng); v = _rand((T, 1, d), rng)
    g = np.zeros((T, 1, d))
    beta = rng.uniform(0.05, 0.95, (T, 1)) if general_beta else np.ones((T, 1))
    o, _ = oracle.recurrence(q, k, v, g, beta, [0, T])
    scores = np.tril(q[:, 0, :] @ k[:, 0, :].T) * beta[:, 0][None, :]
    expect = scores @ v[:, 0, :]
    np.testing.assert_allclose(o[:, 0, :], expect, rtol=1e-11, atol=1e-11)


def _gated_deltanet_decay_after(q, k, v, a_scalar, beta, s0):
    """Single-gate delta rule written with the decay AFTER the erase:
    S <- a (S - beta k (k^T S)) + beta k v^T.  For a scalar gate the order does not matter
    ("How KDA updates its state": Gated DeltaNet's scalar gives the same state either way)."""
    S = s0.copy()
    outs = []
    for t in range(q.shape[0]):
        kk = k[t]
        S = a_scalar[t] * (S - beta[t] * np.outer(kk, kk @ S)) + beta[t] * np.outer(kk, v[t])
        outs.append(S.T @ q[t])
    return np.array(outs), S


def _per_channel_decay_after(q, k, v, g, beta, s0):
    """Negative control: per-channel decay applied after the erase (the wrong order)."""
    S = s0.copy()
    for t in range(q.shape[0]):
        kk = k[t]
        S = S - beta[t] * np.outer(kk, kk @ S)
        S = np.exp(g[t])[:, None] * S + beta[t] * np.outer(kk, v[t])
    return S


def test_P3_scalar_gate_is_gated_deltanet_and_order_matters_per_channel():
    rng = np.random.default_rng(13)
    T, d = 50, 32
    q = _rand((T, d), rng); k = _rand((T, d), rng) / math.sqrt(d); v = _rand((T, d), rng)
    beta = rng.uniform(0.1, 0.9, T); s0 = _rand((d, d), rng) * 0.1
    a = np.exp(-rng.uniform(0.0, 0.3, T))
    g_scalar = np.repeat(np.log(a)[:, None], d, axis=1)
    o, s = oracle.recurrence(q[:, None], k[:, None], v[:, None], g_scalar[:, None], beta[:, None],
                             [0, T], state_in=s0[None, None])
    eo, es = _gated_deltanet_decay_after(q, k, v, a, beta, s0)
    np.testing.assert_allclose(o[:, 0], eo, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(s[0, 0], es, rtol=1e-11, atol=1e-11)
    # per-channel gate: decay-then-erase (KDA) differs from erase-then-decay
    g = -rng.uniform(0.0, 1.0, (T, d))
    _, s_kda = oracle.recurrence(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None],
                                 [0, T], state_in=s0[None, None])
    s_wrong = _per_channel_decay_after(q, k, v, g, beta, s0)
    assert np.abs(s_kda[0, 0] - s_wrong).max() > 1e-3


def test_P4_delta_rule_retrieval():
    """beta = 1 and a unit-norm key: after the write, a read with k_t returns v_t exactly
    ("How KDA updates its state": the next read for k_t returns what this token wrote)."""
    rng = np.random.default_rng(14)
    T, d = 12, 24
    q = _rand((T, 1, d), rng); v = _rand((T, 1, d), rng)
    k = _rand((T, 1, d), rng); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    g = -rng.uniform(0, 0.5, (T, 1, d)); b = np.ones((T, 1)); s0 = _rand((1, 1, d, d), rng)
    for t in range(T):
        _, s = oracle.recurrence(q[:t + 1], k[:t + 1], v[:t + 1], g[:t + 1], b[:t + 1],
                                 [0, t + 1], state_in=s0)
        np.testing.assert_allclose(k[t, 0] @ s[0, 0], v[t, 0], rtol=1e-12, atol=1e-12)


def _transition_np(g_t, b_t, k_t):
    d = k_t.shape[0]
    return (np.eye(d) - b_t * np.outer(k_t, k_t)) @ np.diag(np.exp(g_t))


def test_P5_segment_composition():
    """A segment's effect is (M, S~): a cumulative transition on the incoming state plus the
    state it builds from zero, and S_out = M S_in + S~ ("k3_training_and_infra_notes",
    section 4.1, KDA Context Parallelism).  Resuming from a saved state is bitwise exact."""
    rng = np.random.default_rng(15)
    T, T1, H, d = 40, 17, 2, 16
    q = _rand((T, H, d), rng); k = _rand((T, H, d), rng) / 4; v = _rand((T, H, d), rng)
    g = -rng.uniform(0, 0.2, (T, H, d)); b = rng.uniform(0, 1, (T, H))
    s0 = _rand((1, H, d, d), rng)
    o_all, s_all = oracle.recurrence(q, k, v, g, b, [0, T], state_in=s0)
    _, s_mid = oracle.recurrence(q[:T1], k[:T1], v[:T1], g[:T1], b[:T1], [0, T1], state_in=s0)
    o_2, s_2 = oracle.recurrence(q[T1:], k[T1:], v[T1:], g[T1:], b[T1:], [0, T - T1],
                                 state_in=s_mid)
    assert np.array_equal(s_all, s_2)
    assert np.array_equal(o_all[T1:], o_2)
    # independently formed (M, S~) of the second segment
    _, s_tilde = oracle.recurrence(q[T1:], k[T1:], v[T1:], g[T1:], b[T1:], [0, T - T1])
    for h in range(H):
        M = np.eye(d)
        for t in range(T1, T):
            M = _transition_np(g[t, h], b[t, h], k[t, h]) @ M
        np.testing.assert_allclose(M @ s_mid[0, h] + s_tilde[0, h], s_all[0, h],
                                   rtol=1e-11, atol=1e-11)


def test_P6_fixed_state_size_and_page_cache_figures():
    """S has no token axis: its shape is [N, H, d_k, d_v] whatever the length.  With the page's
    96 heads of 128x128 in bf16 that is 3 MiB per layer, and with 216 KiB of ShortConv caches
    221.55 MiB over 69 layers ("How Kimi K3 Engineered Its Way to the Frontier", section
    "What the hybrid saves")."""
    gold = json.load(open(os.path.join(GOLDEN, "kda_cache_size.json")))
    rng = np.random.default_rng(16)
    for T in (1, 3, 1000):
        d = 128
        x = [_rand((T, 1, d), rng) for _ in range(4)]
        _, s = oracle.recurrence(x[0], x[1], x[2], -np.abs(x[3]) * 0.01, np.full((T, 1), 0.5),
                                 [0, T])
        assert s.shape == (1, 1, 128, 128)
        per_head = s.shape[-1] * s.shape[-2]
    bytes_layer = gold["heads"] * per_head * gold["bytes_per_element_bf16"]
    assert bytes_layer == gold["state_bytes_per_layer"] == 3 * 1024 * 1024
    total = (bytes_layer + gold["conv_cache_bytes_per_layer"]) * gold["kda_layers"] / 2**20
    assert round(total, 2) == gold["total_fixed_cache_MiB"]


def test_packed_equals_separate_and_empty_sequences():
    rng = np.random.default_rng(17)
    lens = [5, 0, 9, 1, 0]
    T, H, d = sum(lens), 2, 8
    q = _rand((T, H, d), rng); k = _rand((T, H, d), rng) / 3; v = _rand((T, H, d), rng)
    g = -rng.uniform(0, 0.3, (T, H, d)); b = rng.uniform(0, 1, (T, H))
    s0 = _rand((len(lens), H, d, d), rng)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, s = oracle.recurrence(q, k, v, g, b, cu, state_in=s0)
    for n, L in enumerate(lens):
        lo, hi = cu[n], cu[n + 1]
        on, sn = oracle.recurrence(q[lo:hi], k[lo:hi], v[lo:hi], g[lo:hi], b[lo:hi], [0, L],
                                   state_in=s0[n:n + 1])
        assert np.array_equal(o[lo:hi], on)
        assert np.array_equal(s[n], sn[0])
        if L == 0:
            assert np.array_equal(s[n], s0[n])


def test_windows_select_rows():
    rng = np.random.default_rng(18)
    T, H, d = 30, 1, 8
    x = [_rand((T, H, d), rng) for _ in range(4)]
    b = rng.uniform(0, 1, (T, H))
    o, _ = oracle.recurrence(x[0], x[1], x[2], -np.abs(x[3]) * 0.1, b, [0, T])
    ow, _ = oracle.recurrence(x[0], x[1], x[2], -np.abs(x[3]) * 0.1, b, [0, T],
                              windows=[(2, 5), (20, 30)])
    assert np.array_equal(ow, np.concatenate([o[2:5], o[20:30]]))


def test_bad_arguments_rejected():
    x = np.zeros((3, 1, 4))
    with pytest.raises(ValueError):
        oracle.recurrence(x, x, x, x, np.zeros((3, 1)), [0, 2, 1, 3][:3])
    with pytest.raises(ValueError):
        oracle.recurrence(x, x, x, x, np.zeros((3, 1)), [0, 4])


def test_bf16_inputs_are_widened_exactly():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(19)
    T, H, d = 20, 2, 16
    xs = [torch.from_numpy(_rand((T, H, d), rng)).to(torch.bfloat16) for _ in range(3)]
    g = torch.from_numpy(-rng.uniform(0, 0.2, (T, H, d))).to(torch.bfloat16)
    b = torch.from_numpy(rng.uniform(0, 1, (T, H))).to(torch.bfloat16)
    o16, s16 = oracle.recurrence(*xs, g, b, [0, T])
    o64, s64 = oracle.recurrence(*[x.double() for x in xs], g.double(), b.double(), [0, T])
    assert np.array_equal(o16, o64) and np.array_equal(s16, s64)


# --------------------------------------------------------------------------------------
# planted mistakes: each mutant of the oracle's C source must fail at least one pin
# --------------------------------------------------------------------------------------
MUTANTS = {
    "forget dropped": ("S[(int64_t)i * dv + j] *= a;", "(void)a;"),
    "gate sign flipped": ("exp(widen(g, in_format, kbase + i))", "exp(-widen(g, in_format, kbase + i))"),
    "erase sign flipped": ("u[j] = widen(v, in_format, vbase + j) - u[j];",
                           "u[j] = widen(v, in_format, vbase + j) + u[j];"),
    "beta dropped": ("const double bk = b * kt[i];", "const double bk = kt[i];"),
    "state transposed in read": ("o[j] += qi * S[(int64_t)i * dv + j];",
                                 "o[j] += qi * S[(int64_t)j * dv + i];"),
    "erase uses query": ("kt[i] = widen(k, in_format, kbase + i);",
                         "kt[i] = widen(q, in_format, kbase + i);"),
    "last token dropped": ("t < cu_seqlens[n + 1]; ++t", "t < cu_seqlens[n + 1] - 1; ++t"),
}


def _pins_pass(lib) -> bool:
    """A compact run of P0 (two cases), P3 and P5 against a given build."""
    try:
        for seed, T in ((4, 8), (5, 6)):
            alphas, betas, ks, vs, qs, s0 = _rational_case(seed, T)
            eo, es = brute_force(alphas, betas, ks, vs, qs, s0)
            f = lambda x: np.array(x, dtype=np.float64)
            o, s = oracle.recurrence(f(qs)[:, None], f(ks)[:, None], f(vs)[:, None],
                                     np.log(f(alphas))[:, None], f(betas)[:, None], [0, T],
                                     state_in=f(s0)[None, None], lib=lib)
            if np.abs(o[:, 0] - f(eo)).max() > 1e-10 or np.abs(s[0, 0] - f(es)).max() > 1e-10:
                return False
        rng = np.random.default_rng(21)
        T, d = 20, 8
        q = _rand((T, d), rng); k = _rand((T, d), rng) / 3; v = _rand((T, d), rng)
        beta = rng.uniform(0.1, 0.9, T); s0 = _rand((d, d), rng)
        a = np.exp(-rng.uniform(0.0, 0.3, T))
        o, s = oracle.recurrence(q[:, None], k[:, None], v[:, None],
                                 np.repeat(np.log(a)[:, None], d, 1)[:, None], beta[:, None],
                                 [0, T], state_in=s0[None, None], lib=lib)
        eo, es = _gated_deltanet_decay_after(q, k, v, a, beta, s0)
        if np.abs(o[:, 0] - eo).max() > 1e-10:
            return False
        return True
    except ValueError:
        return False


def test_planted_mistakes_are_caught(tmp_path):
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")).read()
    assert _pins_pass(None), "unmodified oracle must pass the compact pins"
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, f"mutation site not unique: {name}"
        c = tmp_path / f"mut_{abs(hash(name))}.c"
        so = tmp_path / f"mut_{abs(hash(name))}.so"
        c.write_text(src.replace(old, new))
        subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o", str(so),
                        str(c), "-lm"], check=True)
        lib = oracle.load_variant(str(so))
        assert not _pins_pass(lib), f"planted mistake not caught: {name}"
