"""Pins for the binary64 oracle: each check comes from something other than the oracle itself.

* Philox4x32-10: the published known-answer vectors (tests/golden/philox4x32_10_kat.txt) and, where
  Triton is installed, its interpreter's Philox as an independent library witness.
* Canonical order and top-k: brute force over all k-subsets of tiny rows (the defining dominance
  property, no sorting).
* Top-p and min-p: exact rational arithmetic (fractions.Fraction) on tiny rows; closed forms for
  uniform rows (ceil(p * V)), a forced single huge logit (exactly one token) and two-level rows.
* LSE / log-probability: closed forms (uniform: -log V; two-value rows) and sum_v exp(logp_v) = 1.
* Gumbel-max law: chi-square of many draws against the renormalised truncated distribution, and the
  heavy-tailed Z-score construction of the Gumbel precision page.
"""
import itertools
import math
import os
import struct
import subprocess
import sys
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads
from oracle import philox as ph
from oracle import sampler as sm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------------------------
# Philox4x32-10
# ----------------------------------------------------------------------------------------------
def _kat_rows():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            v = [int(t, 16) for t in line.split()]
            rows.append((tuple(v[0:4]), tuple(v[4:6]), tuple(v[6:10])))
    return rows


def test_philox_known_answer_vectors():
    rows = _kat_rows()
    assert len(rows) == 3
    for ctr, key, out in rows:
        assert ph.philox4x32_10(ctr, key) == out
        vec = ph.philox4x32_10_np(*[np.array([c]) for c in ctr], *[np.array([k]) for k in key])
        assert tuple(int(a[0]) for a in vec) == out


def test_philox_vectorised_matches_scalar():
    rng = np.random.default_rng(7)
    ctr = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64)
    key = rng.integers(0, 2**32, size=(64, 2), dtype=np.uint64)
    vec = ph.philox4x32_10_np(ctr[:, 0], ctr[:, 1], ctr[:, 2], ctr[:, 3], key[:, 0], key[:, 1])
    for i in range(64):
        ref = ph.philox4x32_10(tuple(int(c) for c in ctr[i]), tuple(int(k) for k in key[i]))
        assert tuple(int(v[i]) for v in vec) == ref


def test_philox_token_word_layout():
    # token v takes word v & 3 of Philox((v >> 2, row, step_lo, step_hi), (seed_lo, seed_hi))
    seed, row, step = (0x1234_5678_9ABC_DEF0, 17, (5 << 32) | 9)
    toks = np.arange(0, 23)
    got = ph.token_words(toks, seed, row, step)
    for v in toks:
        ref = ph.philox4x32_10((v >> 2, row, step & 0xFFFFFFFF, step >> 32),
                               (seed & 0xFFFFFFFF, seed >> 32))[v & 3]
        assert int(got[v]) == ref


_TRITON_WITNESS = r"""
import sys, torch, triton, triton.language as tl
@triton.jit
def k(out_ptr, c_ptr, k0, k1, N: tl.constexpr):
    o = tl.arange(0, N)
    c0 = tl.load(c_ptr + 4 * o + 0); c1 = tl.load(c_ptr + 4 * o + 1)
    c2 = tl.load(c_ptr + 4 * o + 2); c3 = tl.load(c_ptr + 4 * o + 3)
    z = c0 * 0
    a, b, c, d = triton.language.random.philox_impl(c0, c1, c2, c3, k0.to(tl.uint32) + z,
                                                    k1.to(tl.uint32) + z, 10)
    tl.store(out_ptr + 4 * o + 0, a); tl.store(out_ptr + 4 * o + 1, b)
    tl.store(out_ptr + 4 * o + 2, c); tl.store(out_ptr + 4 * o + 3, d)
vals = [int(t) for t in sys.argv[1:]]
k0, k1, ctr = vals[0], vals[1], vals[2:]
n = len(ctr) // 4
c = torch.tensor(ctr, dtype=torch.int64).to(torch.uint32)
out = torch.zeros(4 * n, dtype=torch.uint32)
k[(1,)](out, c, k0, k1, N=n)
print(" ".join(str(int(v) & 0xFFFFFFFF) for v in out.tolist()))
"""


def test_philox_matches_triton_interpreter_witness():
    pytest.importorskip("triton")
    rng = np.random.default_rng(11)
    ctr = [int(v) for v in rng.integers(0, 2**32, size=32, dtype=np.uint64)]
    k0, k1 = 0xDEADBEEF, 0x01234567
    env = dict(os.environ, TRITON_INTERPRET="1")
    try:
        out = subprocess.run([sys.executable, "-c", _TRITON_WITNESS, str(k0), str(k1)] + [str(c) for c in ctr],
                             capture_output=True, text=True, env=env, timeout=300)
    except subprocess.TimeoutExpired:
        pytest.skip("triton interpreter timed out")
    if out.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + out.stderr.strip().splitlines()[-1][:200])
    got = [int(t) for t in out.stdout.split()]
    for i in range(8):
        assert tuple(got[4 * i:4 * i + 4]) == ph.philox4x32_10(tuple(ctr[4 * i:4 * i + 4]), (k0, k1))


# ----------------------------------------------------------------------------------------------
# keys, widening, canonical order, top-k
# ----------------------------------------------------------------------------------------------
def test_widen_bf16_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x461C, 0x0000, 0x8000, 0x7F80, 0x0001], dtype=np.uint16)
    x = sm.widen(bits, "bf16")
    assert x[0] == 1.0 and x[1] == -2.0 and x[2] == 9984.0
    assert x[3] == 0.0 and x[4] == 0.0 and math.copysign(1.0, x[4]) < 0
    assert math.isinf(x[5]) and x[6] == 2.0 ** -133


def test_order_key_is_monotone_and_merges_signed_zero():
    f = np.float32
    vals = [-np.inf, -np.finfo(f).max, -1.5, -1.0, -np.finfo(f).tiny, -f(1e-45), -0.0, 0.0, f(1e-45),
            np.finfo(f).tiny, 1.0, 1.5, np.finfo(f).max, np.inf]
    keys = [sm.order_key(float(f(v))) for v in vals]
    assert sm.order_key(-0.0) == sm.order_key(0.0) == 0x80000000
    for a, b, ka, kb in zip(vals, vals[1:], keys, keys[1:]):
        if float(a) == float(b):
            assert ka == kb
        else:
            assert ka < kb
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(4000) * np.exp(rng.uniform(-30, 30, 4000))).astype(np.float32)
    k = np.array([sm.order_key(float(v)) for v in x], dtype=np.uint64)
    assert np.array_equal(np.argsort(k, kind="stable"), np.argsort(x, kind="stable"))


def _dominates(x, a, b):
    return x[a] > x[b] or (x[a] == x[b] and a < b)


def _brute_topk_set(x, k):
    """The unique k-subset S with every member dominating every non-member (no sorting)."""
    n = len(x)
    found = [set(c) for c in itertools.combinations(range(n), k)
             if all(_dominates(x, a, b) for a in c for b in range(n) if b not in c)]
    assert len(found) == 1
    return found[0]


def _brute_order(x):
    """pi from nested top-k sets: pi[k-1] = topk(k) minus topk(k-1)."""
    prev, order = set(), []
    for k in range(1, len(x) + 1):
        cur = _brute_topk_set(x, k)
        (new,) = cur - prev
        order.append(new)
        prev = cur
    return order


def test_canonical_order_and_topk_brute_force():
    rng = np.random.default_rng(5)
    for trial in range(60):
        n = int(rng.integers(1, 9))
        levels = np.array([-1.0, -0.0, 0.0, 0.5, 2.0, -3.25], dtype=np.float32)
        x = levels[rng.integers(0, len(levels), n)] if trial % 2 else rng.standard_normal(n).astype(np.float32)
        x64 = x.astype(np.float64)
        order = _brute_order(list(x64))
        assert list(sm.canonical_order(x64)) == order
        for k in range(0, n + 2):
            st, out = sm.topk_select_row(x, n, k, n + 2)
            assert st == 0
            want = sorted(_brute_topk_set(list(x64), min(k, n))) if k > 0 else []
            assert list(out[:len(want)]) == want and all(v == -1 for v in out[len(want):])


def _bf16_value(bits):
    """A bfloat16 bit pattern as a Python float: the high half of an IEEE single."""
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def test_topk_select_bf16_brute_force_with_ties():
    """bf16 scores: values equal as bf16 tie even where their fp32 sources differed; -0 ties +0; the k-set is
    the unique dominating subset and comes out in ascending index order."""
    rng = np.random.default_rng(17)
    src = np.array([1.0, 1.001, 0.999, -0.0, 0.0, 2.5, 2.5078125, -1.25, np.inf, -np.inf], np.float32)
    for trial in range(60):
        n = int(rng.integers(1, 9))
        bits = workloads.f32_to_bf16_bits(src[rng.integers(0, len(src), n)])
        vals = [_bf16_value(b) for b in bits]
        for k in range(0, n + 2):
            st, out = sm.topk_select_row(bits, n, k, n + 2, dtype="bf16")
            assert st == 0
            want = sorted(_brute_topk_set(vals, min(k, n))) if k > 0 else []
            assert list(out[:len(want)]) == want and all(v == -1 for v in out[len(want):]), (trial, vals, k)
    # 1.0 and 1.001 are one bf16 value: the lowest indices win the tie
    bits = workloads.f32_to_bf16_bits(np.array([0.5, 1.001, 1.0, 1.0, 0.25], np.float32))
    assert list(sm.topk_select_row(bits, 5, 2, 2, dtype="bf16")[1]) == [1, 2]
    nan = workloads.f32_to_bf16_bits(np.array([1.0, np.nan], np.float32))
    assert sm.topk_select_row(nan, 2, 1, 1, dtype="bf16")[0] == sm.STATUS_NONFINITE


def test_topk_select_contract():
    x = np.array([3, 1, 3, 3, 2, np.nan, np.nan], dtype=np.float32)
    st, out = sm.topk_select_row(x, 5, 2, 4)
    assert st == 0 and list(out) == [0, 2, -1, -1]         # lowest-index ties, ascending, -1 pad
    st, out = sm.topk_select_row(x, 5, 9, 9)
    assert st == 0 and list(out) == [0, 1, 2, 3, 4, -1, -1, -1, -1]   # short row: all, then pad
    assert sm.topk_select_row(x, 6, 2, 4)[0] == sm.STATUS_NONFINITE     # NaN inside the length
    assert sm.topk_select_row(x, 5, 5, 4)[0] == sm.STATUS_INVALID_ARG   # k > k_max
    st, out = sm.topk_select_row(x, 5, 0, 3)
    assert st == 0 and list(out) == [-1, -1, -1]
    eq = np.zeros(100, dtype=np.float32)
    assert list(sm.topk_select_row(eq, 100, 37, 37)[1]) == list(range(37))     # all_equal -> [0, k)
    z = np.array([0.0, -0.0, 0.0, -0.0], dtype=np.float32)
    assert list(sm.topk_select_row(z, 4, 3, 3)[1]) == [0, 1, 2]          # signed zeros tie
    inf = np.array([-np.inf, 1.0, np.inf, -np.inf], dtype=np.float32)
    assert list(sm.topk_select_row(inf, 4, 3, 3)[1]) == [0, 1, 2]


def test_topk_matches_torch_set_on_distinct_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(9)
    x = rng.permutation(5000).astype(np.float32) * 0.25
    for k in (1, 50, 2048):
        _, out = sm.topk_select_row(x, x.size, k, k)
        ref = torch.topk(torch.from_numpy(x), k).indices.numpy()
        assert set(out.tolist()) == set(ref.tolist())


# ----------------------------------------------------------------------------------------------
# top-p, min-p: exact rational brute force and closed forms
# ----------------------------------------------------------------------------------------------
def _exact_kept(x, T, k, p, mp):
    """Kept count by exact rational prefix sums on the binary64 weights; None if within 1e-9 of a tie."""
    x = [float(v) for v in x]
    n = len(x)
    order = _brute_order(x)
    m = x[order[0]]
    w = [Fraction(math.exp((x[v] - m) / T)) for v in order]
    nk = k if 0 < k < n else n
    kept = nk
    if p < 1:
        target = Fraction(float(np.float32(p))) * sum(w[:nk])
        pref = Fraction(0)
        cp = nk
        for j in range(nk):
            if abs(pref - target) <= target * Fraction(1, 10**9) and j > 0:
                return None
            if pref >= target:
                cp = j
                break
            pref += w[j]
        kept = min(kept, cp)
    if mp > 0:
        mpf = Fraction(float(np.float32(mp)))
        kept = min(kept, sum(1 for wv in w if wv >= mpf))
    return max(1, kept)


def test_topp_minp_exact_rational_brute_force():
    rng = np.random.default_rng(21)
    checked = 0
    for trial in range(400):
        n = int(rng.integers(1, 11))
        if trial % 3 == 0:
            x = rng.integers(-3, 3, n).astype(np.float32) * np.float32(0.5)
        else:
            x = (rng.standard_normal(n) * 2).astype(np.float32)
        T = float(np.float32(rng.choice([0.5, 1.0, 1.7])))
        k = int(rng.integers(0, n + 2))
        p = float(np.float32(rng.choice([1.0, rng.uniform(0.05, 1.0)])))
        mp = float(np.float32(rng.choice([0.0, 0.0, rng.uniform(0.0, 1.0), 1.0])))
        want = _exact_kept(x.astype(np.float64), T, k, p, mp)
        if want is None:
            continue
        r = sm.sample_row(x, "f32", T, k, p, mp, seed=1, row_id=0, step=trial, keep_order=True)
        assert r.status == 0
        assert r.kept == want, (x, T, k, p, mp)
        assert r.kept_lo <= r.kept <= r.kept_hi
        assert list(r.order[:r.kept]) == _brute_order(list(x.astype(np.float64)))[:want]
        checked += 1
    assert checked > 300


def test_uniform_rows_keep_ceil_p_times_V():
    for n, p in [(1000, 0.9), (1000, 0.123), (4096, 0.5), (151936, 0.95)]:
        x = np.full(n, 0.75, dtype=np.float32)
        r = sm.sample_row(x, "f32", 1.0, 0, p, 0.0, seed=3, row_id=0, step=0)
        want = math.ceil(Fraction(float(np.float32(p))) * n)
        assert r.kept == want and r.idx_cut == want - 1
        assert abs(r.row_logsum - math.log(n)) < 1e-12
        assert abs(r.logprob + math.log(n)) < 1e-12
        assert not r.ambiguous
    # the bf16 +1e4 workload: every value rounds to 9984.0, kept = ceil(0.95f * 151936)
    b = workloads.c4(B=2)
    assert np.all(b.logits == 0x461C)
    r = sm.sample_row(b.logits[0], "bf16", 1.0, 0, 0.95, 0.0, seed=3, row_id=0, step=0)
    assert r.kept == 144340 and abs(r.logprob + math.log(151936)) < 1e-12


def test_topk_then_topp_uses_topk_renormalised_mass():
    x = np.zeros(100, dtype=np.float32)
    r = sm.sample_row(x, "f32", 1.0, 10, 0.5, 0.0)
    assert r.kept == 5                     # target = 0.5 * S_k = 5 (not 0.5 * S = 50 -> 10)
    r = sm.sample_row(x, "f32", 1.0, 10, 1.0, 0.0)
    assert r.kept == 10 and r.idx_cut == 9


@pytest.mark.parametrize("big", [1.0e4, 1.0e30])
def test_forced_single_huge_logit_keeps_exactly_one(big):
    x = np.zeros(1000, dtype=np.float32)
    x[377] = big
    for p in (0.5, 0.9, 0.99999994):
        for T in (0.5, 1.0, 1.5):
            r = sm.sample_row(x, "f32", T, 0, p, 0.0, seed=5, row_id=2, step=1)
            assert r.kept == 1 and r.token == 377 and r.logprob == 0.0 and not math.isnan(r.logprob)


def test_two_level_rows_min_p_top_p_logprob():
    x = np.array([0, -2, 0, -2, -2, 0, -2, -2], dtype=np.float32)      # 3 upper, 5 lower
    S = 3 + 5 * math.exp(-2)
    r = sm.sample_row(x, "f32", 1.0, 0, 1.0, 0.5)
    assert r.kept == 3
    assert sm.sample_row(x, "f32", 1.0, 0, 1.0, 0.1).kept == 8
    assert sm.sample_row(x, "f32", 1.0, 0, 1.0, 1.0).kept == 3          # w >= min_p keeps the max ties
    assert sm.sample_row(x, "f32", 1.0, 0, 0.5, 0.0).kept == math.ceil(0.5 * S)
    assert abs(sm.logprob_row(x, "f32", 1.0, 0) + math.log(S)) < 1e-12
    assert abs(sm.logprob_row(x, "f32", 1.0, 1) - (-2 - math.log(S))) < 1e-12
    S2 = 3 + 5 * math.exp(-1)
    assert abs(sm.logprob_row(x, "f32", 2.0, 1) - (-1 - math.log(S2))) < 1e-12
    st, m, ls = sm.softmax_lse_row(x, "f32", 2.0)
    assert st == 0 and m == 0.0 and abs(ls - math.log(S2)) < 1e-12


def test_greedy_returns_lowest_index_argmax():
    x = np.array([1, 5, 5, 2], dtype=np.float32)
    for T in (0.0, -1.0):
        r = sm.sample_row(x, "f32", T, 0, 0.3, 0.0, seed=9, row_id=0, step=4)
        assert r.token == 1 and r.kept == 1
        S = 2 + math.exp(-4) + math.exp(-3)
        assert abs(r.logprob - min(0.0, -math.log(S))) < 1e-12


def test_logprobs_normalise():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(300) * 3).astype(np.float32)
    lp = [sm.logprob_row(x, "f32", 0.7, t) for t in range(300)]
    assert abs(math.fsum(math.exp(v) for v in lp) - 1.0) < 1e-12


def test_invalid_and_nonfinite_rows():
    x = np.zeros(8, dtype=np.float32)
    assert sm.sample_row(x, "f32", 1.0, 0, 0.0, 0.0).status == sm.STATUS_INVALID_ARG
    assert sm.sample_row(x, "f32", 1.0, 0, float("nan"), 0.0).status == sm.STATUS_INVALID_ARG
    assert sm.sample_row(x, "f32", 1.0, 0, 0.5, 1.5).status == sm.STATUS_INVALID_ARG
    assert sm.sample_row(x, "f32", float("nan"), 0, 0.5, 0.0).status == sm.STATUS_INVALID_ARG
    y = x.copy()
    y[3] = np.inf
    assert sm.sample_row(y, "f32", 1.0, 0, 0.5, 0.0).status == sm.STATUS_NONFINITE
    y[3] = np.nan
    assert sm.sample_row(y, "f32", 1.0, 0, 0.5, 0.0).status == sm.STATUS_NONFINITE


def test_neumaier_scan_against_exact_prefix():
    # sub-ulp increments: a plain running sum never moves off 1.0; the compensated scan finds the exact
    # crossing (1 + 400 quarter-ulps == target), and the rounded fsum certificate cannot separate the
    # last two prefixes, so the boundary is reported ambiguous ([TOPP] step 6).
    tiny = 2.0 ** -54
    w = np.array([1.0] + [tiny] * 1000)
    target = 1.0 + 100 * 2.0 ** -52
    acc, exact = Fraction(0), None
    for i, v in enumerate(w):
        acc += Fraction(float(v))
        if acc >= Fraction(target):
            exact = i + 1
            break
    assert exact == 401
    naive = next((i + 1 for i, c in enumerate(np.cumsum(w)) if c >= target), len(w))
    assert naive == len(w)
    assert sm.neumaier_scan(w, target) == exact
    c, amb = sm.nucleus_count(w, target)
    assert c == exact and amb
    # a boundary separated by more than an ulp certifies cleanly
    w2 = np.array([0.5, 0.25, 0.125, 0.0625, 0.0625])
    c2, amb2 = sm.nucleus_count(w2, 0.8)
    assert c2 == 3 and not amb2


def test_invariants_on_random_rows():
    rng = np.random.default_rng(13)
    for trial in range(40):
        n = int(rng.integers(50, 3000))
        x = (rng.standard_normal(n) * rng.uniform(0.1, 5)).astype(np.float32)
        T = float(np.float32(rng.uniform(0.3, 2.0)))
        k = int(rng.integers(0, n + 5))
        p = float(np.float32(rng.uniform(0.1, 1.0)))
        r = sm.sample_row(x, "f32", T, k, p, 0.0, seed=7, row_id=trial, step=0, keep_order=True)
        x64 = x.astype(np.float64)
        w = np.exp((x64 - x64.max()) / T)
        order = r.order
        assert np.all(np.diff(x64[order]) <= 0)
        ties = np.diff(x64[order]) == 0
        assert np.all(np.diff(order)[ties] > 0)
        nk = k if 0 < k < n else n
        Sk = math.fsum(w[order[:nk]].tolist())
        target = p * Sk
        kept_mass = math.fsum(w[order[:r.kept]].tolist())
        less_one = math.fsum(w[order[:r.kept - 1]].tolist())
        assert kept_mass >= target * (1 - 1e-12) or r.kept == nk
        assert r.kept == 1 or less_one < target * (1 + 1e-12)
        assert not r.ambiguous
        assert r.token in set(order[:r.kept].tolist())
        mask = sm.kept_mask(r, n)
        assert mask.sum() == r.kept and np.all(mask[order[:r.kept]] == 1)


def test_no_ambiguous_boundaries_on_the_workloads():
    for b in (workloads.c1(), workloads.c2(B=4, V=20000), workloads.c4(B=2, V=5000),
              workloads.c5(B=4, V=20000)):
        for r in range(b.B):
            res = sm.sample_row(b.logits[r], b.dtype, b.temperature[r], b.top_k[r], b.top_p[r],
                                b.min_p[r], int(b.seed[r]), r, int(b.step[r]))
            assert res.status == 0 and not res.ambiguous


# ----------------------------------------------------------------------------------------------
# Gumbel-max sampling law
# ----------------------------------------------------------------------------------------------
def _chi2(obs, probs, n):
    exp = probs * n
    return float(np.sum((obs - exp) ** 2 / exp))


def test_gumbel_draws_follow_the_truncated_softmax():
    x = np.array([0.0, -0.5, -1.0, -1.5, 0.3, -3.0], dtype=np.float32)
    T = 0.8
    s = (x.astype(np.float64) - 0.3) / np.float64(np.float32(T))
    N = 200_000
    steps = np.arange(N, dtype=np.uint64)
    # full support
    cand = sm.canonical_order(x.astype(np.float64))
    tok = sm.draw_many(s, cand, seed=42, row_id=3, steps=steps)
    w = np.exp(s)
    obs = np.bincount(tok, minlength=6).astype(np.float64)
    assert _chi2(obs, w / w.sum(), N) < 40.0            # 5 dof: p ~ 1e-7
    # top-3 support, renormalised
    cand3 = cand[:3]
    tok3 = sm.draw_many(s, cand3, seed=42, row_id=3, steps=steps)
    assert set(np.unique(tok3).tolist()) == set(cand3.tolist())
    w3 = w[cand3]
    obs3 = np.array([(tok3 == v).sum() for v in cand3], dtype=np.float64)
    assert _chi2(obs3, w3 / w3.sum(), N) < 35.0         # 2 dof
    # the per-step scalar draw agrees with the vectorised one
    for st in range(5):
        assert sm.draw(s, cand, 42, 3, st)[0] == tok[st]


def test_heavy_tailed_z_scores():
    # counts in {1,2,3}, one dominant count; logits = log(counts) (Gumbel precision page's test)
    V = 64
    counts = workloads.heavy_tail_counts(V, seed=1234, head_log_gap=6.0)
    x = np.log(counts.astype(np.float64)).astype(np.float32)
    s = x.astype(np.float64) - float(x.max())
    N = 100_000
    tok = sm.draw_many(s, np.arange(V), seed=1234, row_id=0, steps=np.arange(N, dtype=np.uint64))
    total = counts.sum()
    p0 = counts[0] / total

    def z(obs, exp):
        return (obs - exp) / math.sqrt(exp * (1 - exp / N))

    assert abs(z((tok == 0).sum(), p0 * N)) < 10.0
    assert abs(z((tok >= 1).sum(), (1 - p0) * N)) < 10.0


def test_uniform_map_is_the_cell_midpoint():
    top = 2**32 - 1
    u0, u1 = sm.uniform_from_word(np.array([0, top]))
    assert 0.0 < u0 < 1.0 and 0.0 < u1 < 1.0
    b = np.random.default_rng(4).integers(0, 2**32, size=10000, dtype=np.uint64)
    assert np.all(sm.uniform_from_word(b) + sm.uniform_from_word(np.uint64(top) - b) == 1.0)
    assert np.all(np.isfinite(sm.gumbel_from_uniform(sm.uniform_from_word(np.array([0, 1, top - 1, top])))))


def test_gumbel_noise_inverts_the_gumbel_cdf():
    u = np.array([1e-9, 1e-4, 0.1, 0.5, 0.9, 0.999, 1 - 1e-9])
    g = sm.gumbel_from_uniform(u)
    assert np.all(np.diff(g) < 0)                       # larger u -> smaller noise
    assert np.allclose(np.exp(-np.exp(-g)), 1.0 - u, rtol=1e-12, atol=0)


def test_argmax_ties_go_to_the_lowest_index():
    cand = np.array([7, 3, 9, 1])
    assert sm.argmax_lowest(np.array([2.0, 5.0, 5.0, 1.0]), cand)[0] == 3
    assert sm.argmax_lowest(np.array([5.0, 5.0, 5.0, 5.0]), cand)[0] == 1
    assert list(sm.argmax_lowest(np.array([[1.0, 0.0, 1.0, 0.0], [0.0, 2.0, 0.0, 2.0]]), cand)) == [7, 1]


# ----------------------------------------------------------------------------------------------
# Top-N log-probability lists
# ----------------------------------------------------------------------------------------------
def test_topn_list_dominates_everything_after_it_on_tiny_rows():
    """The defining property, checked pairwise (no sorting): every listed token precedes every later one and
    every unlisted one in the order (logit descending, index ascending)."""
    rng = np.random.default_rng(11)
    for trial in range(300):
        n = int(rng.integers(1, 9))
        x = (rng.integers(-3, 4, size=n) / 2.0).astype(np.float32)   # many ties
        N = int(rng.integers(1, 10))
        st, m, ls, idx, lp = sm.topn_logprobs_row(x, "f32", 1.0, N)
        assert st == 0
        listed = [int(v) for v in idx if v >= 0]
        assert len(listed) == min(N, n)
        assert all(v == -1 for v in idx[len(listed):]) and all(math.isnan(v) for v in lp[len(listed):])

        def before(a, b):
            return x[a] > x[b] or (x[a] == x[b] and a < b)

        for i, a in enumerate(listed):
            for b in listed[i + 1:]:
                assert before(a, b), (trial, x, listed)
            for b in set(range(n)) - set(listed):
                assert before(a, b), (trial, x, listed)


def test_topn_logprobs_closed_forms():
    # uniform row: the first N indices, each with log-probability -log V
    V = 1000
    st, m, ls, idx, lp = sm.topn_logprobs_row(np.zeros(V, np.float32), "f32", 1.0, 20)
    assert st == 0 and list(idx) == list(range(20))
    assert np.allclose(lp, -math.log(V), atol=1e-12, rtol=0)
    # two levels: n_a tokens at a, n_b at b; log p(a-token) = -log(n_a + n_b e^{(b - a)/T}) in closed form
    a, b, n_a, n_b, T = 1.5, -0.25, 3, 17, 0.75
    x = np.full(n_a + n_b, b, np.float32)
    pos = [4, 9, 13]
    x[pos] = a
    st, m, ls, idx, lp = sm.topn_logprobs_row(x, "f32", T, 5)
    assert list(idx[:3]) == pos and list(idx[3:]) == [0, 1]
    want_a = -math.log(n_a + n_b * math.exp((float(np.float32(b)) - float(np.float32(a))) / float(np.float32(T))))
    want_b = want_a + (float(np.float32(b)) - float(np.float32(a))) / float(np.float32(T))
    assert abs(lp[0] - want_a) < 1e-12 and abs(lp[4] - want_b) < 1e-12
    # the whole row listed: probabilities sum to one and the list is non-increasing
    x = np.random.default_rng(5).normal(0, 2, 257).astype(np.float32)
    st, m, ls, idx, lp = sm.topn_logprobs_row(x, "f32", 1.3, 257)
    assert abs(math.fsum(np.exp(lp).tolist()) - 1.0) < 1e-12
    assert np.all(np.diff(lp) <= 0)
    # greedy temperature reads as T = 1; a non-finite logit is a row error
    assert sm.topn_logprobs_row(x, "f32", 0.0, 3)[4][0] == sm.topn_logprobs_row(x, "f32", 1.0, 3)[4][0]
    x[7] = np.inf
    assert sm.topn_logprobs_row(x, "f32", 1.0, 3)[0] == sm.STATUS_NONFINITE


# ----------------------------------------------------------------------------------------------
# Processed (kept-set renormalised) log-probabilities
# ----------------------------------------------------------------------------------------------
def test_kept_logprobs_against_exact_rational_kept_sets():
    """On tiny rows the kept set comes from exact rational prefix sums; the processed probabilities of
    the kept tokens are their weights over the kept weights' sum, every other token has probability 0."""
    rng = np.random.default_rng(31)
    checked = 0
    for trial in range(200):
        n = int(rng.integers(1, 10))
        x = (rng.standard_normal(n) * 2).astype(np.float32)
        T = float(np.float32(rng.choice([0.5, 1.0, 1.7])))
        k = int(rng.integers(0, n + 2))
        p = float(np.float32(rng.choice([1.0, rng.uniform(0.05, 1.0)])))
        mp = float(np.float32(rng.choice([0.0, rng.uniform(0.0, 0.5)])))
        want = _exact_kept(x.astype(np.float64), T, k, p, mp)
        if want is None:
            continue
        order = _brute_order(list(x.astype(np.float64)))
        keep = set(order[:want])
        xs = x.astype(np.float64)
        z = sum(math.exp((xs[v] - xs.max()) / T) for v in keep)
        for t in range(n):
            st, lp, lo, hi, rank = sm.kept_logprob_row(x, "f32", T, k, p, mp, t)
            assert st == 0
            if t in keep:
                assert abs(math.exp(lp) - math.exp((xs[t] - xs.max()) / T) / z) < 1e-12, (x, t)
            else:
                assert lp == -math.inf
        checked += 1
    assert checked > 150


def test_kept_logprob_closed_forms():
    # uniform row, top-p p: ceil(p V) tokens kept, each at -log(ceil(p V)); the rest at -inf
    V, p = 1000, 0.3
    kept = math.ceil(Fraction(float(np.float32(p))) * V)
    x = np.zeros(V, np.float32)
    assert sm.kept_logprob_row(x, "f32", 1.0, 0, p, 0.0, kept - 1)[1] == pytest.approx(-math.log(kept), abs=1e-12)
    assert sm.kept_logprob_row(x, "f32", 1.0, 0, p, 0.0, kept)[1] == -math.inf
    # top-k alone on distinct logits: s_t - log sum over the k largest
    x = np.array([0.5, 3.0, -1.0, 2.0, 1.0], np.float32)
    want = 2.0 - math.log(math.exp(3.0) + math.exp(2.0) + math.exp(1.0))
    assert sm.kept_logprob_row(x, "f32", 1.0, 3, 1.0, 0.0, 3)[1] == pytest.approx(want, abs=1e-12)
    assert sm.kept_logprob_row(x, "f32", 1.0, 3, 1.0, 0.0, 0)[1] == -math.inf
    # greedy: the first maximum alone, probability one
    y = np.array([1.0, 4.0, 4.0, 2.0], np.float32)
    assert sm.kept_logprob_row(y, "f32", 0.0, 0, 0.9, 0.0, 1)[1] == 0.0
    assert sm.kept_logprob_row(y, "f32", 0.0, 0, 0.9, 0.0, 2)[1] == -math.inf
    # nothing filtered: the processed log-probability is the full-row one
    assert sm.kept_logprob_row(x, "f32", 0.8, 0, 1.0, 0.0, 4)[1] == pytest.approx(
        sm.logprob_row(x, "f32", 0.8, 4), abs=1e-12)
    # error rows and tokens outside the row
    assert sm.kept_logprob_row(y, "f32", 1.0, 0, 1.0, 0.0, 4)[0] == sm.STATUS_INVALID_ARG
    y[2] = np.nan
    assert sm.kept_logprob_row(y, "f32", 1.0, 0, 1.0, 0.0, 1)[0] == sm.STATUS_NONFINITE


# ----------------------------------------------------------------------------------------------
# The parity tolerances the oracle reports: the 1e-6 band of top-p / min-p and near-tie draws
# ----------------------------------------------------------------------------------------------
BAND = Fraction(1, 10**6)


def _band_counts_exact(w_sorted, nk, target):
    """(kept_lo, kept, kept_hi) of a top-p cut by exact rational prefixes: rank j is kept iff the mass
    before it is below the target; ranks whose prefix lies within 1e-6 * S_k of the target may go either
    way (the tolerance of the stage's contract, read in probability units)."""
    Sk = sum(w_sorted[:nk])
    pref, lo, mid, hi = Fraction(0), 0, 0, 0
    for j in range(nk):
        lo += pref < target - BAND * Sk
        mid += pref < target
        hi += pref <= target + BAND * Sk
        pref += w_sorted[j]
    return max(1, lo), max(1, mid), max(1, hi)


@pytest.mark.parametrize("n,k,T", [(1000, 0, 1.0), (12, 0, 1.0), (12, 9, 0.7), (40, 25, 1.3)])
def test_topp_band_bounds_at_half_and_twice_the_tolerance(n, k, T):
    """The target p * S_k is placed 0.5e-6 * S_k and 2e-6 * S_k on either side of a prefix mass (p rounded to
    fp32, the exact offset recomputed in rationals): inside the band the boundary token may go either way
    (kept_lo < kept_hi), outside it the three counts agree. A band of the wrong width, or a sign slip in
    either bound, moves one of the eight cases."""
    rng = np.random.default_rng(n * 100 + k)
    if n == 1000:
        x = np.zeros(n, dtype=np.float32)                       # uniform: prefixes are the integers
    else:
        x = (rng.uniform(-2.0, 0.0, n)).astype(np.float32)     # every weight >= e^-2/T of the max
    x64 = [float(v) for v in x]
    order = sorted(range(n), key=lambda v: (-x64[v], v))
    m = x64[order[0]]
    Tf = float(np.float32(T))
    w = [Fraction(math.exp((x64[v] - m) / Tf)) for v in order]
    nk = k if 0 < k < n else n
    Sk = sum(w[:nk])
    checked = 0
    for j in (1, nk // 2, nk - 2):
        Pj = sum(w[:j])                                         # mass before rank j
        for delta, pattern in ((Fraction(1, 2 * 10**6), (j, j + 1, j + 1)), (Fraction(-1, 2 * 10**6), (j, j, j + 1)),
                               (Fraction(2, 10**6), (j + 1, j + 1, j + 1)), (Fraction(-2, 10**6), (j, j, j))):
            p = float(np.float32(float((Pj + delta * Sk) / Sk)))
            off = (Fraction(p) * Sk - Pj) / Sk                   # realised offset, exact
            assert abs(off - delta) < Fraction(1, 10**7)
            want = _band_counts_exact(w, nk, Fraction(p) * Sk)
            assert want == pattern                              # the construction lands where intended
            r = sm.sample_row(x, "f32", T, k, p, 0.0)
            assert (r.kept_lo, r.kept, r.kept_hi) == want, (j, float(delta), (r.kept_lo, r.kept, r.kept_hi), want)
            assert not r.ambiguous
            checked += 1
    assert checked == 12


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_minp_band_bounds_at_half_and_twice_the_tolerance(T):
    """min_p placed at w_j (1 -+ 0.5e-6) and w_j (1 -+ 2e-6) for the weight w_j of rank j: a weight within
    1e-6 * min_p of min_p may go either way, one further out may not."""
    n = 16
    x = np.linspace(-3.0, 0.0, n).astype(np.float32)[::-1].copy()  # distinct, decreasing: rank j = index j
    Tf = float(np.float32(T))
    w = [math.exp((float(v) - float(x[0])) / Tf) for v in x]
    for j in (1, 7, 14):
        for rel, pattern in ((0.5e-6, (j, j, j + 1)), (-0.5e-6, (j, j + 1, j + 1)),
                             (2e-6, (j, j, j)), (-2e-6, (j + 1, j + 1, j + 1))):
            mp = float(np.float32(w[j] * (1.0 + rel)))
            r = sm.sample_row(x, "f32", T, 0, 1.0, mp)
            assert (r.kept_lo, r.kept, r.kept_hi) == pattern, (j, rel, (r.kept_lo, r.kept, r.kept_hi))


def _two_token_row(g_a, g_b, gap):
    """fp32 logits (0, x_b) whose perturbed scores (x - max) + g differ by about ``gap`` in favour of token 0;
    returns the row and the realised scores, computed exactly from the rounded x_b."""
    xb = np.float32(g_a - g_b - gap)
    x = np.array([0.0, xb], dtype=np.float32)
    m = max(0.0, float(xb))
    sa, sb = (0.0 - m) + g_a, (float(xb) - m) + g_b
    return x, sa, sb


def test_near_tie_flag_is_one_part_in_a_million_of_the_best_score():
    """Two-token rows built from the pinned Philox words and Gumbel map, with the runner-up 0.5e-6 or 2e-6
    (relative to max(1, |best|)) below the winner: only the first is a near tie. Draws with |best| well above
    1 separate the relative reading from an absolute 1e-6."""
    seed, rid = 77, 5
    steps = np.arange(4000, dtype=np.uint64)
    g = sm.gumbel_from_uniform(sm.uniform_from_word(ph.token_words(np.array([0, 1]), seed, rid, steps)))
    found = {"small": 0, "large": 0}
    for st in range(len(steps)):
        g_a, g_b = float(g[st, 0]), float(g[st, 1])
        if not (0.05 < g_a - g_b < 0.9):                       # x_b in (0, 1): fp32 spacing below 6e-8
            continue
        # the winner's score is g_b + gap (token 1 holds the maximum logit)
        kind = "large" if g_b > 3.0 else ("small" if abs(g_b) < 0.9 else None)
        if kind is None or found[kind] >= 3:
            continue
        scale = max(1.0, abs(g_b))
        for rel, want in ((0.5e-6, True), (2e-6, False)):
            x, sa, sb = _two_token_row(g_a, g_b, rel * scale)
            realised = (sa - sb) / max(1.0, abs(sa))
            assert 0.8 * rel < realised < 1.2 * rel             # the fp32 logit kept the intended gap
            r = sm.sample_row(x, "f32", 1.0, 0, 1.0, 0.0, seed=seed, row_id=rid, step=st)
            assert r.token == 0 and abs(r.best - sa) < 1e-12 and abs(r.second - sb) < 1e-12
            assert r.near_tie is want, (st, g_b, rel, realised)
            if kind == "large" and want:
                assert sa - sb > 1e-6                           # an absolute 1e-6 band would miss it
        found[kind] += 1
        if found["small"] >= 3 and found["large"] >= 3:
            break
    assert found == {"small": 3, "large": 3}
