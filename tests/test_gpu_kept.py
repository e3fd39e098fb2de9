"""GPU parity of vsamp_kept_logprob (log-probabilities renormalised over the cut's kept set) against the
binary64 oracle: -inf exactly for tokens outside the kept set, within 1e-5 for kept tokens. Where the CUDA cut
keeps a count inside the 1e-6 band, the oracle is evaluated at that count."""
import math

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


def _batch(name, x, dtype="f32", T=1.0, k=0, p=1.0, mp=0.0):
    B, V = x.shape
    f = lambda v, dt: np.full(B, v, dtype=dt) if np.isscalar(v) else np.asarray(v, dtype=dt)
    return workloads.SampleBatch(name, dtype, x, V, f(T, np.float32), f(k, np.int32), f(p, np.float32),
                                 f(mp, np.float32), np.zeros(B, np.uint64), np.zeros(B, np.uint64))


def _tokens(b, rows, rng):
    """Per row: the first maximum, the last kept token, the first token outside the cut and a random one."""
    out = [np.zeros(b.B, np.int32) for _ in range(4)]
    for r in range(b.B):
        out[3][r] = rng.integers(0, b.V)
    for r in rows:
        res = osm.sample_row(b.logits[r, :b.V], b.dtype, b.temperature[r], b.top_k[r], b.top_p[r], b.min_p[r],
                             keep_order=True)
        if res.status != 0:
            continue
        out[0][r] = res.order[0]
        out[1][r] = res.order[res.kept - 1]
        out[2][r] = res.order[min(res.kept, res.n - 1)]
    return out


def _check(ts, dev, b, rows, seed=0):
    x = to_device(b.logits, b.dtype, dev)
    kw = dict(temperature=t(b.temperature, dev), top_k=t(b.top_k, dev), top_p=t(b.top_p, dev),
              min_p=t(b.min_p, dev), V=b.V)
    cut, _, _ = ts.vsamp_topp_minp_mask(x, want_mask=False, **kw)
    cut = cut.cpu().numpy()
    for r in rows:   # an ambiguous oracle boundary stops the comparison ([TOPP] step 6)
        assert not osm.sample_row(b.logits[r, :b.V], b.dtype, b.temperature[r], b.top_k[r], b.top_p[r],
                                  b.min_p[r]).ambiguous, f"row {r}: oracle_boundary_ambiguous"
    for tokens in _tokens(b, rows, np.random.default_rng(seed)):
        out, st = ts.vsamp_kept_logprob(x, t(tokens, dev), **kw)
        torch.cuda.synchronize()
        out, st = out.cpu().numpy(), st.cpu().numpy()
        for r in rows:
            row = b.logits[r, :b.V]
            args = (row, b.dtype, b.temperature[r], b.top_k[r], b.top_p[r], b.min_p[r], int(tokens[r]))
            s0, lp0, lo, hi, rank = osm.kept_logprob_row(*args)
            assert st[r] == s0, f"row {r}: status {st[r]} != {s0}"
            if s0 != 0:
                assert np.isnan(out[r])
                continue
            kept = int(cut[r, 2])
            assert lo <= kept <= hi, f"row {r}: kept {kept} outside [{lo}, {hi}]"
            _, lp1, _, _, _ = osm.kept_logprob_row(*args, kept=kept)
            if lp1 == -math.inf:
                assert out[r] == -np.inf, f"row {r} token {tokens[r]} (rank {rank}): {out[r]} != -inf"
            else:
                assert abs(float(out[r]) - lp1) <= LOGP_TOL, f"row {r} token {tokens[r]}: {out[r]} vs {lp1}"


def test_c1_rows(ts, dev):
    b = workloads.c1()
    _check(ts, dev, b, range(b.B))


def test_c2_dominant_token_rows(ts, dev):
    b = workloads.c2()
    _check(ts, dev, b, range(0, b.B, 4))


def test_c4_tied_rows(ts, dev):
    b = workloads.c4()
    _check(ts, dev, b, range(0, b.B, 32))


def test_c5_near_uniform_rows(ts, dev):
    b = workloads.c5(B=64)
    rows = sorted(set(range(0, 64, 8)) | set(int(r) for r in b.meta["dup_rows"]))
    _check(ts, dev, b, rows)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 7, 33, 1000, 4099])
def test_small_ragged_rows_greedy_and_min_p(ts, dev, dtype, V):
    rng = np.random.default_rng(V)
    B = 6
    a = rng.normal(0.0, 2.0, size=(B, V)).astype(np.float32)
    a[1] = (rng.integers(-4, 5, size=V) / 2.0).astype(np.float32)    # ties
    logits = workloads.f32_to_bf16_bits(a) if dtype == "bf16" else a
    b = _batch("small", logits, dtype, T=[1.0, 0.8, 0.0, 1.3, 1.0, -1.0], k=[0, 5, 0, 40, 0, 3],
               p=[0.9, 1.0, 0.5, 0.7, 1.0, 0.95], mp=[0.0, 0.0, 0.0, 0.1, 0.3, 0.0])
    _check(ts, dev, b, range(B))


def test_error_rows(ts, dev):
    rng = np.random.default_rng(9)
    B, V = 4, 3000
    a = rng.normal(0.0, 1.0, size=(B, V)).astype(np.float32)
    a[0, 5] = np.inf
    b = _batch("err", a, T=[1.0, np.nan, 1.0, 1.0], p=[0.9, 0.9, 0.0, 0.9])
    x = to_device(b.logits, "f32", dev)
    tok = np.array([1, 1, 1, V + 3], np.int32)
    out, st = ts.vsamp_kept_logprob(x, t(tok, dev), temperature=t(b.temperature, dev), top_p=t(b.top_p, dev))
    out, st = out.cpu().numpy(), st.cpu().numpy()
    assert list(st) == [osm.STATUS_NONFINITE, osm.STATUS_INVALID_ARG, osm.STATUS_INVALID_ARG,
                        osm.STATUS_INVALID_ARG]
    assert np.all(np.isnan(out))
