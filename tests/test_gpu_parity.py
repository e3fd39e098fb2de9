"""GPU parity: every entry point of libvsamp.so against the binary64 oracle, on the seeded workloads (at
sizes the oracle finishes in seconds and at the full benchmark size) and on edge cases."""
import math
import os

import numpy as np
import pytest

import workloads
from oracle import sampler as osm

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import parity_util  # noqa: E402
from parity_util import (LOGP_TOL, TieCounter, check_cut, check_sample, oracle_row, run_cut, run_sample, t,  # noqa: E402
                         to_device)


@pytest.fixture(scope="module")
def ts():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g

    g.build()
    import top_sampling_gb300 as ts_mod

    return ts_mod


@pytest.fixture(scope="module")
def dev():
    return torch.device("cuda:0")


def _sample_batch(name, x, dtype="f32", T=1.0, k=0, p=1.0, mp=0.0, seed=7, step=0):
    B, V = x.shape
    f = lambda v, dt: np.full(B, v, dtype=dt) if np.isscalar(v) else np.asarray(v, dtype=dt)
    return workloads.SampleBatch(name, dtype, x, V, f(T, np.float32), f(k, np.int32), f(p, np.float32),
                                 f(mp, np.float32), f(seed, np.uint64), f(step, np.uint64))


# ------------------------------------------------------------------------------------------------
# the five workloads
# ------------------------------------------------------------------------------------------------
def test_c1_all_entry_points(ts, dev):
    b = workloads.c1()
    ties = TieCounter()
    tok, lp, st, stats = run_sample(ts, b, dev)
    check_sample(b, range(b.B), tok, lp, st, stats, ties)
    cut, mask, cstats = run_cut(ts, b, dev)
    check_cut(b, range(b.B), cut, mask, cstats)
    x = to_device(b.logits, b.dtype, dev)
    m, ls, lst = ts.vsamp_softmax_lse(x, temperature=t(b.temperature, dev))
    m, ls = m.cpu().numpy(), ls.cpu().numpy()
    for r in range(b.B):
        st_o, m_o, ls_o = osm.softmax_lse_row(b.logits[r], b.dtype, b.temperature[r])
        assert m[r] == np.float32(m_o) and abs(ls[r] - ls_o) <= LOGP_TOL
    idx, sst = ts.vsamp_topk_select(x, 50)
    idx = idx.cpu().numpy()
    for r in range(b.B):
        assert np.array_equal(idx[r], osm.topk_select_row(b.logits[r], b.V, 50, 50)[1])
    # log-probabilities of given tokens, from statistics and recomputed
    toks = torch.tensor([3, 31999, 0, 12345], dtype=torch.int32, device=dev)
    lp1, _ = ts.vsamp_logprob(x, toks, temperature=t(b.temperature, dev))
    mm, lss, _ = ts.vsamp_softmax_lse(x, temperature=t(b.temperature, dev))
    lp2, _ = ts.vsamp_logprob(x, toks, temperature=t(b.temperature, dev), row_max=mm, row_logsum=lss)
    for r in range(b.B):
        want = osm.logprob_row(b.logits[r], b.dtype, b.temperature[r], int(toks[r]))
        assert abs(float(lp1[r]) - want) <= LOGP_TOL and abs(float(lp2[r]) - want) <= LOGP_TOL
    ties.check()


def test_c2_dominant_token_rows(ts, dev):
    b = workloads.c2()
    ties = TieCounter()
    tok, lp, st, stats = run_sample(ts, b, dev)
    check_sample(b, range(b.B), tok, lp, st, stats, ties)
    cut, mask, cstats = run_cut(ts, b, dev, want_mask=True)
    check_cut(b, range(0, b.B, 2), cut, mask, cstats)
    ties.check()


def test_c2_one_million_draws_z_test(ts, dev):
    """C2's own distribution test: 15,625 steps x 64 rows = 1e6 draws under the workload's per-row mix of
    temperature, top-k, top-p and min-p. The oracle gives each row's kept set and renormalised law; the hits
    of the dominant tokens and the draws outside them are compared with their expectations (|Z| < 10, the
    Gumbel precision page's bound; where the law leaves no variance the count must be exact)."""
    b = workloads.c2()
    B, steps = b.B, 15625
    p_dom = np.zeros(B)
    for r in range(B):
        ref = oracle_row(b, r)
        assert ref.status == 0 and not ref.ambiguous
        kept = ref.order[:ref.kept]
        w = np.exp(ref.s[kept] - ref.s[kept].max())
        p_dom[r] = float(w[kept == int(b.meta["dominant"][r])].sum() / w.sum())
    x = to_device(b.logits, b.dtype, dev)
    dom = t(b.meta["dominant"].astype(np.int32), dev)
    kw = dict(temperature=t(b.temperature, dev), top_k=t(b.top_k, dev), top_p=t(b.top_p, dev),
              min_p=t(b.min_p, dev), seed=t(b.seed, dev), want_logprob=False)
    hits = torch.zeros(B, dtype=torch.int64, device=dev)
    bad = torch.zeros(B, dtype=torch.int64, device=dev)
    for s in range(steps):
        tok, _, st, _ = parity_util.sample_fn(ts)(x, step=torch.full((B,), s, dtype=torch.int64, device=dev), **kw)
        hits += (tok == dom)
        bad += (st != 0) | (tok < 0)
    torch.cuda.synchronize()
    hits, bad = hits.cpu().numpy(), bad.cpu().numpy()
    assert not bad.any()
    N = B * steps
    e_hit = float((steps * p_dom).sum())
    var = float((steps * p_dom * (1.0 - p_dom)).sum())
    tail = N - int(hits.sum())
    for r in np.flatnonzero(p_dom == 1.0):          # a one-token law: every draw is the dominant token
        assert hits[r] == steps, f"row {r}: {hits[r]} of {steps}"
    if var > 0:
        z_hit = (hits.sum() - e_hit) / math.sqrt(var)
        z_tail = (tail - (N - e_hit)) / math.sqrt(var)
        assert abs(z_hit) < 10 and abs(z_tail) < 10, (z_hit, z_tail)
    else:
        assert tail == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_c3_topk_select_ties(ts, dev, dtype):
    """All 128 rows bit-exact; the 256 score levels (q - 128) / 16 are exact in bf16 too."""
    b = workloads.c3()
    scores = b.scores if dtype == "f32" else workloads.f32_to_bf16_bits(b.scores)
    x = to_device(scores, dtype, dev)
    idx, st = ts.vsamp_topk_select(x, t(b.k, dev), k_max=b.k_max, lengths=t(b.lengths, dev))
    idx, st = idx.cpu().numpy(), st.cpu().numpy()
    for r in range(b.B):
        s_o, want = osm.topk_select_row(scores[r], int(b.lengths[r]), int(b.k[r]), b.k_max, dtype=dtype)
        assert st[r] == s_o
        assert np.array_equal(idx[r], want), f"row {r} (len {b.lengths[r]})"
    # repeated calls are bit-identical
    idx2, _ = ts.vsamp_topk_select(x, t(b.k, dev), k_max=b.k_max, lengths=t(b.lengths, dev))
    assert np.array_equal(idx, idx2.cpu().numpy())


def test_c4_full_size_bf16(ts, dev):
    """The benchmark workload at full size, in the benchmark's launch configuration."""
    b = workloads.c4()
    tok, lp, st, stats = run_sample(ts, b, dev)
    want_kept = math.ceil(0.949999988079071044921875 * 151936)
    assert want_kept == 144340
    assert np.all(st == 0)
    assert np.all(stats[:, 2] == want_kept)
    assert np.all((tok >= 0) & (tok < want_kept))
    assert np.all(np.abs(lp - (-math.log(151936))) <= LOGP_TOL)
    ties = TieCounter()
    check_sample(b, range(0, b.B, 16), tok, lp, st, stats, ties)
    ties.check()


def test_c4_full_size_cut_mask_and_statistics(ts, dev):
    """The C4 cut with its 38.9 MB mask, and the row statistics, at full size: every row keeps the 144,340
    lowest indices (uniform rows), element by element; sampled rows against the oracle's kept prefix; the
    maximum 9984.0 and log S = log 151,936 on every row."""
    b = workloads.c4()
    cut, mask, cstats = run_cut(ts, b, dev, want_mask=True)
    assert np.all(cut[:, 3] == 0) and np.all(cut[:, 2] == 144340) and np.all(cut[:, 1] == 144339)
    assert mask[:, :144340].all() and not mask[:, 144340:].any()
    check_cut(b, range(0, b.B, 32), cut, mask, cstats)
    x = to_device(b.logits, b.dtype, dev)
    m, ls, st = ts.vsamp_softmax_lse(x, temperature=t(b.temperature, dev))
    m, ls, st = m.cpu().numpy(), ls.cpu().numpy(), st.cpu().numpy()
    assert np.all(st == 0) and np.all(m == np.float32(9984.0))
    assert np.all(np.abs(ls - math.log(151936)) <= LOGP_TOL)
    for r in range(0, b.B, 64):
        st_o, m_o, ls_o = osm.softmax_lse_row(b.logits[r], b.dtype, b.temperature[r])
        assert m[r] == np.float32(m_o) and abs(ls[r] - ls_o) <= LOGP_TOL


def test_c5_near_uniform_rows(ts, dev):
    b = workloads.c5(B=64)
    ties = TieCounter()
    tok, lp, st, stats = run_sample(ts, b, dev)
    rows = sorted(set(range(0, 64, 4)) | set(int(r) for r in b.meta["dup_rows"]))
    check_sample(b, rows, tok, lp, st, stats, ties)
    cut, mask, cstats = run_cut(ts, b, dev, want_mask=True)
    check_cut(b, rows[:8], cut, mask, cstats)
    ties.check()


def test_c5_full_size_statistics(ts, dev):
    """Row maxima and log-sum-exp at the full C5 size (512 x 262,144 fp32) against the oracle on sampled rows,
    including the rows with a duplicated maximum."""
    b = workloads.c5()
    x = to_device(b.logits, b.dtype, dev)
    m, ls, st = ts.vsamp_softmax_lse(x, temperature=t(b.temperature, dev))
    m, ls, st = m.cpu().numpy(), ls.cpu().numpy(), st.cpu().numpy()
    assert np.all(st == 0)
    for r in sorted(set(range(0, 512, 37)) | set(int(v) for v in b.meta["dup_rows"])):
        st_o, m_o, ls_o = osm.softmax_lse_row(b.logits[r], b.dtype, b.temperature[r])
        assert m[r] == np.float32(m_o) and abs(ls[r] - ls_o) <= LOGP_TOL, r


def test_c5_full_batch_properties(ts, dev):
    b = workloads.c5()
    tok, lp, st, stats = run_sample(ts, b, dev)
    assert np.all(st == 0)
    # min-p is inactive (all weights within 1e-3 of the maximum), top-k keeps 4096, top-p 0.99 of those
    assert np.all((stats[:, 2] >= 4000) & (stats[:, 2] <= 4096))
    ties = TieCounter()
    check_sample(b, list(range(0, 512, 64)) + [int(r) for r in b.meta["dup_rows"]], tok, lp, st, stats, ties)
    ties.check()


# ------------------------------------------------------------------------------------------------
# edge cases
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 2, 3, 5, 7, 8, 9, 31, 33, 257, 1000, 4099])
def test_small_and_ragged_rows(ts, dev, dtype, V):
    rng = np.random.default_rng(V)
    B = 6
    x = (rng.integers(-4, 4, size=(B, V)) * 0.5).astype(np.float32) if V % 2 else \
        (rng.standard_normal((B, V)) * 2).astype(np.float32)
    if dtype == "bf16":
        x = workloads.f32_to_bf16_bits(x)
    k = rng.integers(0, V + 2, size=B)
    p = np.array([1.0, 0.9, 0.5, 0.3, 0.999, 0.05], dtype=np.float32)
    mp = np.array([0.0, 0.0, 0.1, 0.5, 1.0, 0.0], dtype=np.float32)
    T = np.array([1.0, 0.7, 1.3, 0.0, 2.0, 1.0], dtype=np.float32)
    b = _sample_batch("ragged", x, dtype, T, k, p, mp, seed=np.arange(B) + 100, step=np.arange(B))
    ties = TieCounter()
    tok, lp, st, stats = run_sample(ts, b, dev)
    check_sample(b, range(B), tok, lp, st, stats, ties)
    cut, mask, cstats = run_cut(ts, b, dev)
    check_cut(b, range(B), cut, mask, cstats)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_padded_stride_and_unaligned_rows(ts, dev, dtype):
    rng = np.random.default_rng(3)
    B, V, ld = 5, 1003, 1040
    xf = np.full((B, ld), np.nan, dtype=np.float32)
    xf[:, :V] = rng.standard_normal((B, V)).astype(np.float32) * 3
    x = workloads.f32_to_bf16_bits(xf) if dtype == "bf16" else xf
    b = _sample_batch("pad", x, dtype, 1.0, 40, 0.8, 0.0)
    b.V = V
    ties = TieCounter()
    tok, lp, st, stats = run_sample(ts, b, dev, V=V)
    check_sample(b, range(B), tok, lp, st, stats, ties)
    # an unaligned view (row start shifted by one element): the plain-load path
    full = to_device(x, dtype, dev)
    view = full[:, 1:V + 1]
    b2 = _sample_batch("unaligned", np.ascontiguousarray(x[:, 1:V + 1]), dtype, 1.0, 40, 0.8, 0.0)
    tok2, lp2, st2, stats2 = run_sample(ts, b2, dev, x=view)
    assert np.all(stats2[:, 3] & 32)    # rows were loaded with plain loads
    check_sample(b2, range(B), tok2, lp2, st2, stats2, ties)


def test_nonfinite_and_invalid_rows(ts, dev):
    x = np.zeros((8, 100), dtype=np.float32)
    x[0, 5] = np.nan
    x[1, 7] = np.inf
    x[2, 9] = -np.inf
    b = _sample_batch("bad", x, "f32", T=[1, 1, 1, 1, np.nan, 1, 1, 1], p=[1, 1, 1, 0.0, 0.5, 1, np.nan, 0.5],
                      mp=[0, 0, 0, 0, 0, 1.5, 0, 0])
    tok, lp, st, stats = run_sample(ts, b, dev)
    assert list(st) == [4, 4, 4, 1, 1, 1, 1, 0]
    assert np.all(tok[:7] == -1) and np.all(np.isnan(lp[:7])) and tok[7] >= 0
    cut, mask, _ = run_cut(ts, b, dev)
    assert list(cut[:, 3]) == [4, 4, 4, 1, 1, 1, 1, 0] and not mask[:7].any()


def test_greedy_ties_signed_zero_and_forced_rows(ts, dev):
    V = 1000
    x = np.zeros((6, V), dtype=np.float32)
    x[0, [10, 20, 30]] = 5.0                 # tied maxima, greedy -> 10
    x[1, :] = np.where(np.arange(V) % 2, -0.0, 0.0)   # signed zeros tie
    x[2, 377] = 1e30                         # forced single huge logit
    x[3, 377] = 1e4
    x[4, [1, 2, 3]] = 2.0                    # min_p = 1 keeps the three maxima
    x[5, :] = 0.25                           # uniform
    b = _sample_batch("edge", x, "f32", T=[0.0, 1.0, 1.0, 0.5, 1.0, 1.0], k=[0, 37, 0, 0, 0, 0],
                      p=[0.3, 1.0, 0.999, 0.9, 1.0, 0.5], mp=[0, 0, 0, 0, 1.0, 0])
    ties = TieCounter()
    tok, lp, st, stats = run_sample(ts, b, dev)
    check_sample(b, range(6), tok, lp, st, stats, ties)
    assert tok[0] == 10 and tok[2] == 377 and tok[3] == 377 and lp[2] == 0.0
    assert stats[1, 2] == 37 and stats[4, 2] == 3 and stats[5, 2] == 500
    cut, mask, cstats = run_cut(ts, b, dev)
    check_cut(b, range(6), cut, mask, cstats)
    idx, _ = ts.vsamp_topk_select(to_device(x, "f32", dev), 37)
    assert list(idx.cpu().numpy()[1]) == list(range(37))


def test_topk_select_contract_edges(ts, dev):
    rng = np.random.default_rng(8)
    B, L = 6, 5000
    x = (rng.integers(0, 3, size=(B, L)) * 1.0).astype(np.float32)
    x[0, :4] = [np.inf, -np.inf, np.inf, -np.inf]
    x[1, 100:] = np.nan                      # beyond its length: never read
    lengths = np.array([L, 100, 50, 3000, 0, L + 1], dtype=np.int32)
    ks = np.array([64, 64, 64, 0, 10, 10], dtype=np.int32)
    idx, st = ts.vsamp_topk_select(torch.from_numpy(x).to(dev), t(ks, dev), k_max=64, lengths=t(lengths, dev),
                                   max_len=L)
    idx, st = idx.cpu().numpy(), st.cpu().numpy()
    for r in range(B):
        s_o, want = osm.topk_select_row(x[r], int(lengths[r]), int(ks[r]), 64) if 0 < lengths[r] <= L else \
            (osm.STATUS_INVALID_ARG, np.full(64, -1, dtype=np.int32))
        assert st[r] == s_o and np.array_equal(idx[r], want), r
    # k > k_max is a row error
    idx, st = ts.vsamp_topk_select(torch.from_numpy(x).to(dev), t(np.full(B, 65, np.int32), dev), k_max=64)
    want_st = [osm.topk_select_row(x[r], L, 65, 64)[0] for r in range(B)]
    assert list(st.cpu().numpy()) == want_st and 1 in want_st and np.all(idx.cpu().numpy() == -1)


def test_determinism_batch_and_cluster_invariance(ts, dev):
    b = workloads.c1(B=8, V=32000, seed=5)
    b.top_k[:] = [0, 50, 1000, 0, 7, 0, 3000, 1]
    b.top_p[:] = [0.9, 1.0, 0.7, 0.99, 0.5, 1.0, 0.95, 0.9]
    b.min_p[:] = [0.0, 0.05, 0.0, 0.0, 0.0, 0.2, 0.0, 0.0]
    ref = run_sample(ts, b, dev)
    for _ in range(2):
        again = run_sample(ts, b, dev)
        assert all(np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                                  c.view(np.uint32) if c.dtype == np.float32 else c) for a, c in zip(ref, again))
    # one row at a time (same counters): identical outputs
    for r in (0, 3, 6):
        one = workloads.SampleBatch("one", b.dtype, b.logits[r:r + 1], b.V, b.temperature[r:r + 1], b.top_k[r:r + 1],
                                    b.top_p[r:r + 1], b.min_p[r:r + 1], b.seed[r:r + 1], b.step[r:r + 1])
        o = run_sample(ts, one, dev, row_id=np.array([r], dtype=np.uint32))
        assert o[0][0] == ref[0][r] and o[1][0].view(np.uint32) == ref[1][r].view(np.uint32)
    # cluster size does not change any output bit
    old = os.environ.get("VSAMP_CLUSTER")
    try:
        for C in (1, 2, 4, 8, 16):
            os.environ["VSAMP_CLUSTER"] = str(C)
            o = run_sample(ts, b, dev)
            assert np.array_equal(o[0], ref[0]) and np.array_equal(o[1].view(np.uint32), ref[1].view(np.uint32)), C
            assert np.array_equal(o[3][:, 2], ref[3][:, 2]), C
    finally:
        if old is None:
            os.environ.pop("VSAMP_CLUSTER", None)
        else:
            os.environ["VSAMP_CLUSTER"] = old


# ------------------------------------------------------------------------------------------------
# sampling law
# ------------------------------------------------------------------------------------------------
def test_heavy_tailed_z_scores_one_million_draws(ts, dev):
    """The Gumbel precision page's test: one token 18 log-units above counts in {1, 2, 3}."""
    V = 151936
    counts = workloads.heavy_tail_counts(V, seed=1234)
    row = workloads.heavy_tail_logits(V, seed=1234)
    B, steps = 2000, 500
    x = torch.from_numpy(row).to(dev).unsqueeze(0).repeat(B, 1).contiguous()
    seeds = torch.full((B,), 1234, dtype=torch.int64, device=dev)
    rid = torch.arange(B, dtype=torch.int32, device=dev)
    hits0 = tail = 0
    first = None
    for s in range(steps):
        tok, _, st, _ = parity_util.sample_fn(ts)(x, seed=seeds, step=torch.full((B,), s, dtype=torch.int64, device=dev),
                                        row_id=rid, want_logprob=False)
        if first is None:
            first = tok.cpu().numpy()
        hits0 += int((tok == 0).sum())
        tail += int((tok >= 1).sum())
    N = B * steps
    total = counts.sum()
    p0 = counts[0] / total
    z0 = (hits0 - p0 * N) / math.sqrt(N * p0 * (1 - p0))
    zt = (tail - (1 - p0) * N) / math.sqrt(N * p0 * (1 - p0))
    assert abs(z0) < 10 and abs(zt) < 10, (z0, zt)
    # same counters as the oracle on a sample of the draws
    s_row = osm.widen(row, "f32")
    s_row = s_row - s_row.max()
    for r in range(0, B, 100):
        ref_tok = osm.draw(s_row, osm.canonical_order(s_row), 1234, r, 0)[0]
        assert first[r] == ref_tok


def test_small_vocab_chi_square(ts, dev):
    x = np.array([0.0, -0.5, -1.0, -1.5, 0.3, -3.0, -0.2, -0.9], dtype=np.float32)
    T = 0.8
    B, steps = 100_000, 10
    xt = torch.from_numpy(x).to(dev).unsqueeze(0).repeat(B, 1).contiguous()
    temp = torch.full((B,), T, dtype=torch.float32, device=dev)
    counts = np.zeros(8)
    for s in range(steps):
        tok, _, _, _ = parity_util.sample_fn(ts)(xt, temperature=temp, seed=torch.full((B,), 99, dtype=torch.int64, device=dev),
                                       step=torch.full((B,), s, dtype=torch.int64, device=dev), want_logprob=False)
        counts += np.bincount(tok.cpu().numpy(), minlength=8)
    s = (x.astype(np.float64) - 0.3) / np.float64(np.float32(T))
    w = np.exp(s)
    exp = w / w.sum() * B * steps
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    assert chi2 < 45.0, chi2        # 7 dof: p ~ 1e-7
