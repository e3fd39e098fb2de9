"""GPU checks of vsamp_sample_rejection, the dual-pivot rejection sampler ("Sorting-free top-k/top-p/min-p sampling
with dual-pivot rejection kernels #901", Regression guard: the sampled support equals the filtered set, and
frequencies inside it pass a chi-square test against the renormalised truncated distribution over >= 1e6 draws;
Task: an adversarial near-uniform 152K-token row that exercises the round cap and its fallback). The rejection
rounds consume other random numbers than the Gumbel-max draw, so the comparison with the binary64 oracle is of the
law (the oracle's kept prefix and its weights), not of individual tokens."""
import math
import os

import numpy as np
import pytest

import workloads
from oracle import sampler as osm

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from parity_util import LOGP_TOL, t, to_device  # noqa: E402


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


def _law(row, dtype, T, k, p, mp):
    """The oracle's kept prefix and its renormalised probabilities."""
    ref = osm.sample_row(row, dtype, T, k, p, mp, keep_order=True)
    assert ref.status == 0 and not ref.ambiguous and ref.kept_lo == ref.kept_hi
    kept = ref.order[:ref.kept]
    w = np.exp(ref.s[kept] - ref.s[kept].max())
    return kept, w / w.sum()


def _draws(ts, dev, row, dtype, T, k, p, mp, B=100_000, steps=10, seed=11):
    xt = to_device(np.repeat(row[None, :], B, axis=0), dtype, dev)
    counts = np.zeros(row.shape[0], dtype=np.int64)
    kw = dict(temperature=T, top_k=k, top_p=p, min_p=mp, want_logprob=False)
    rid = torch.arange(B, dtype=torch.int32, device=dev)
    for s in range(steps):
        tok, _, st, _ = ts.vsamp_sample_rejection(xt, seed=seed, step=s, row_id=rid, **kw)
        assert int(st.ne(0).sum()) == 0
        counts += np.bincount(tok.cpu().numpy(), minlength=row.shape[0])
    return counts


CASES = [
    # (name, logits, T, top_k, top_p, min_p)
    ("top_k", np.array([0.0, -0.5, 0.3, -1.0, 0.3, -3.0, -0.2, -0.9, 0.1, -2.0], np.float32), 0.8, 4, 1.0, 0.0),
    ("top_k_ties", np.array([1.0, 0.5, 1.0, 0.5, 0.5, 0.5, -1.0, 0.5], np.float32), 1.0, 4, 1.0, 0.0),
    ("top_p", np.array([0.0, -0.5, 0.3, -1.0, 0.35, -3.0, -0.2, -0.9, 0.1, -2.0], np.float32), 1.3, 0, 0.7, 0.0),
    ("min_p", np.array([0.0, -0.5, 0.3, -1.0, 0.35, -3.0, -0.2, -0.9, 0.1, -2.0], np.float32), 1.0, 0, 1.0, 0.4),
    ("joint", np.array([0.0, -0.5, 0.3, -1.0, 0.35, -3.0, -0.2, -0.9, 0.1, -2.0], np.float32), 0.9, 6, 0.8, 0.0),
    ("joint_all", np.array([2.0, 1.5, 1.5, 1.0, 0.2, 0.2, -0.4, -1.0, 0.9, 1.5], np.float32), 1.1, 7, 0.9, 0.1),
]


@pytest.mark.parametrize("name,row,T,k,p,mp", CASES, ids=[c[0] for c in CASES])
def test_support_and_chi_square_over_a_million_draws(ts, dev, name, row, T, k, p, mp):
    kept, prob = _law(row, "f32", T, k, p, mp)
    counts = _draws(ts, dev, row, "f32", T, k, p, mp)
    N = int(counts.sum())
    assert N == 1_000_000
    outside = np.setdiff1d(np.flatnonzero(counts), kept)
    assert outside.size == 0, f"{name}: sampled outside the kept set: {outside}"
    assert set(np.flatnonzero(counts).tolist()) == set(kept.tolist()), name       # every kept token is drawn
    exp = prob * N
    chi2 = float(((counts[kept] - exp) ** 2 / exp).sum())
    dof = max(1, kept.size - 1)
    assert chi2 < dof + 10 * math.sqrt(2 * dof) + 20, (name, chi2, dof)         # ~1e-6 tail for these dof


@pytest.mark.parametrize("name,row,T,k,p,mp", CASES[:3], ids=[c[0] for c in CASES[:3]])
def test_the_cap_fallback_draws_the_same_law(ts, dev, name, row, T, k, p, mp):
    """With the round cap lowered to one, most rows take the cap's exact cut: support and law are unchanged."""
    old = os.environ.get("VSAMP_REJECT_ROUNDS")
    os.environ["VSAMP_REJECT_ROUNDS"] = "1"
    try:
        kept, prob = _law(row, "f32", T, k, p, mp)
        counts = _draws(ts, dev, row, "f32", T, k, p, mp, B=50_000, steps=4)
        xt = to_device(row[None, :].repeat(64, 0), "f32", dev)
        _, _, _, stats = ts.vsamp_sample_rejection(xt, temperature=T, top_k=k, top_p=p, min_p=mp, seed=3,
                                                   step=torch.arange(64, dtype=torch.int64, device=dev), want_stats=True)
        torch.cuda.synchronize()
        assert int((stats[:, 3] & 64).ne(0).sum()) > 0                           # the cap was reached
    finally:
        if old is None:
            os.environ.pop("VSAMP_REJECT_ROUNDS", None)
        else:
            os.environ["VSAMP_REJECT_ROUNDS"] = old
    N = int(counts.sum())
    assert np.setdiff1d(np.flatnonzero(counts), kept).size == 0
    exp = prob * N
    chi2 = float(((counts[kept] - exp) ** 2 / exp).sum())
    dof = max(1, kept.size - 1)
    assert chi2 < dof + 10 * math.sqrt(2 * dof) + 20, (name, chi2, dof)


@pytest.mark.parametrize("which", ["c1", "c2", "c4", "c5"])
def test_workload_draws_lie_in_the_kept_set(ts, dev, which):
    """Every draw of the workloads (several steps) lies in the oracle's kept prefix; log-probabilities are the
    full-row ones; repeated calls are identical."""
    b = {"c1": workloads.c1, "c2": lambda: workloads.c2(B=16), "c4": lambda: workloads.c4(B=16),
         "c5": lambda: workloads.c5(B=16)}[which]()
    x = to_device(b.logits, b.dtype, dev)
    kw = dict(temperature=t(b.temperature, dev), top_k=t(b.top_k, dev), top_p=t(b.top_p, dev),
              min_p=t(b.min_p, dev), seed=t(b.seed, dev))
    refs = [osm.sample_row(b.logits[r], b.dtype, b.temperature[r], b.top_k[r], b.top_p[r], b.min_p[r],
                           keep_order=True) for r in range(b.B)]
    for s in range(8):
        step = torch.full((b.B,), s, dtype=torch.int64, device=dev)
        tok, lp, st, stats = ts.vsamp_sample_rejection(x, step=step, want_stats=True, **kw)
        tok2, _, _, _ = ts.vsamp_sample_rejection(x, step=step, **kw)
        torch.cuda.synchronize()
        tok, lp, st, tok2 = tok.cpu().numpy(), lp.cpu().numpy(), st.cpu().numpy(), tok2.cpu().numpy()
        assert np.array_equal(tok, tok2)
        for r in range(b.B):
            ref = refs[r]
            assert st[r] == 0 and not ref.ambiguous
            assert tok[r] in set(ref.order[:ref.kept_hi].tolist()), (which, r, s)
            want = osm.logprob_row(b.logits[r], b.dtype, b.temperature[r], int(tok[r]))
            assert abs(float(lp[r]) - want) <= LOGP_TOL


def test_adversarial_near_uniform_row_reports_its_rounds(ts, dev):
    """The page's adversarial case: 152K near-uniform logits (N(0, 1e-4^2)) under top-k, top-p and min-p. Every
    row ends (within the cap or by its fallback, which stats reports), and every draw lies in the kept set."""
    rng = np.random.default_rng(17)
    B, V = 32, 151936
    x = rng.normal(0.0, 1e-4, size=(B, V)).astype(np.float32)
    k = np.array([1, 40, 4096, 0] * 8, np.int32)
    p = np.array([1.0, 0.9, 0.99, 0.5] * 8, np.float32)
    mp = np.array([0.0, 0.0, 0.01, 0.9999] * 8, np.float32)
    xt = to_device(x, "f32", dev)
    tok, _, st, stats = ts.vsamp_sample_rejection(xt, top_k=t(k, dev), top_p=t(p, dev), min_p=t(mp, dev), seed=5,
                                                  want_stats=True)
    torch.cuda.synchronize()
    tok, st, stats = tok.cpu().numpy(), st.cpu().numpy(), stats.cpu().numpy()
    assert np.all(st == 0)
    rounds = stats[:, 1]
    capped = int(np.count_nonzero(stats[:, 3] & 64))
    print(f"rounds per row: min {rounds.min()} median {int(np.median(rounds))} max {rounds.max()}; cap reached {capped}")
    assert np.all((rounds >= 1) & (rounds <= 32))
    for r in range(0, B, 3):
        ref = osm.sample_row(x[r], "f32", 1.0, k[r], p[r], mp[r], keep_order=True)
        assert tok[r] in set(ref.order[:ref.kept_hi].tolist()), r


def test_greedy_and_error_rows(ts, dev):
    x = np.zeros((5, 300), np.float32)
    x[0, [40, 7, 99]] = 3.0
    x[1, 5] = np.nan
    x[3, 2] = 1.0
    T = np.array([0.0, 1.0, np.nan, 1.0, -2.0], np.float32)
    tok, lp, st, _ = ts.vsamp_sample_rejection(to_device(x, "f32", dev), temperature=t(T, dev), top_p=0.5, seed=2)
    torch.cuda.synchronize()
    tok, lp, st = tok.cpu().numpy(), lp.cpu().numpy(), st.cpu().numpy()
    assert list(st) == [0, osm.STATUS_NONFINITE, osm.STATUS_INVALID_ARG, 0, 0]
    assert tok[0] == 7 and tok[4] == 0 and tok[1] == -1 and tok[2] == -1 and math.isnan(lp[1])
    assert abs(float(lp[0]) - osm.logprob_row(x[0], "f32", 1.0, 7)) <= LOGP_TOL
