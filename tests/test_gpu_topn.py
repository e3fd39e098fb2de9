"""GPU parity of vsamp_topn_logprobs (top-N log-probability lists) against the binary64 oracle: the list's
indices bit-exact, log-probabilities within 1e-5, empty lists on error rows, and invariance of a row's list
to the batch around it."""
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


def _check_rows(logits, dtype, temps, N, rows, idx, lp, st, V=None):
    for r in rows:
        row = logits[r] if V is None else logits[r, :V]
        s_o, m_o, ls_o, idx_o, lp_o = osm.topn_logprobs_row(row, dtype, temps[r], N)
        assert st[r] == s_o, f"row {r}: status {st[r]} != {s_o}"
        assert np.array_equal(idx[r], idx_o), f"row {r}: {idx[r][:8]} != {idx_o[:8]}"
        valid = idx_o >= 0
        assert np.all(np.isnan(lp[r][~valid]))
        assert np.all(np.abs(lp[r][valid] - lp_o[valid]) <= LOGP_TOL), f"row {r}"


def _run(ts, x, N, temps, dev, V=None):
    oi, ol, m, ls, st = ts.vsamp_topn_logprobs(x, N, temperature=t(temps, dev), V=V)
    torch.cuda.synchronize()
    return oi.cpu().numpy(), ol.cpu().numpy(), st.cpu().numpy()


@pytest.mark.parametrize("N", [1, 20, 257])
def test_c1_rows(ts, dev, N):
    b = workloads.c1()
    idx, lp, st = _run(ts, to_device(b.logits, b.dtype, dev), N, b.temperature, dev, V=b.V)
    _check_rows(b.logits, b.dtype, b.temperature, N, range(b.B), idx, lp, st, V=b.V)


def test_c2_dominant_token_rows(ts, dev):
    b = workloads.c2()
    idx, lp, st = _run(ts, to_device(b.logits, b.dtype, dev), 20, b.temperature, dev, V=b.V)
    _check_rows(b.logits, b.dtype, b.temperature, 20, range(0, b.B, 4), idx, lp, st, V=b.V)


def test_c4_full_size_all_tied_rows(ts, dev):
    """Every logit of the bf16 rows rounds to the same value: the list is the first N indices, each at -log V."""
    b = workloads.c4()
    idx, lp, st = _run(ts, to_device(b.logits, b.dtype, dev), 20, b.temperature, dev, V=b.V)
    assert np.all(st == 0)
    assert np.all(idx == np.arange(20, dtype=np.int32)[None, :])
    assert np.all(np.abs(lp - (-math.log(151936))) <= LOGP_TOL)
    _check_rows(b.logits, b.dtype, b.temperature, 20, range(0, b.B, 32), idx, lp, st, V=b.V)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,N", [(1, 1), (1, 20), (7, 20), (31, 31), (100, 64), (4097, 20), (10000, 4096)])
def test_small_ragged_and_tied_rows(ts, dev, dtype, V, N):
    rng = np.random.default_rng(1000 + V + N)
    B = 6
    a = (rng.integers(-6, 7, size=(B, V)) / 4.0).astype(np.float32)   # many exact ties
    a[1] = rng.normal(0.0, 3.0, size=V).astype(np.float32)
    a[2, : V // 2] = -0.0                                             # -0 equals +0 in the order
    a[2, V // 2:] = 0.0
    logits = workloads.f32_to_bf16_bits(a) if dtype == "bf16" else a
    temps = np.array([1.0, 0.7, 1.0, 0.0, 2.5, -1.0], dtype=np.float32)
    idx, lp, st = _run(ts, to_device(logits, dtype, dev), N, temps, dev)
    _check_rows(logits, dtype, temps, N, range(B), idx, lp, st)
    assert np.all(idx[:, min(N, V):] == -1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_padded_stride(ts, dev, dtype):
    rng = np.random.default_rng(77)
    B, V, ld = 5, 3001, 3072
    a = rng.normal(0.0, 2.0, size=(B, ld)).astype(np.float32)
    a[:, V:] = 1e30   # beyond the row: never read
    logits = workloads.f32_to_bf16_bits(a) if dtype == "bf16" else a
    temps = np.full(B, 0.9, np.float32)
    idx, lp, st = _run(ts, to_device(logits, dtype, dev), 20, temps, dev, V=V)
    _check_rows(logits, dtype, temps, 20, range(B), idx, lp, st, V=V)


def test_error_rows_give_empty_lists(ts, dev):
    rng = np.random.default_rng(5)
    B, V = 4, 5000
    a = rng.normal(0.0, 1.0, size=(B, V)).astype(np.float32)
    a[0, 17] = np.nan
    a[1, 4000] = np.inf
    temps = np.array([1.0, 1.0, np.nan, np.inf], dtype=np.float32)
    idx, lp, st = _run(ts, to_device(a, "f32", dev), 20, temps, dev)
    assert list(st) == [osm.STATUS_NONFINITE, osm.STATUS_NONFINITE, osm.STATUS_INVALID_ARG,
                        osm.STATUS_INVALID_ARG]
    assert np.all(idx == -1) and np.all(np.isnan(lp))
    _check_rows(a, "f32", temps, 20, range(B), idx, lp, st)


def test_list_does_not_depend_on_the_batch(ts, dev):
    b = workloads.c1(B=8)
    x = to_device(b.logits, b.dtype, dev)
    idx, lp, st = _run(ts, x, 20, b.temperature, dev)
    for r in (0, 5):
        i1, l1, s1 = _run(ts, x[r:r + 1].contiguous(), 20, b.temperature[r:r + 1], dev)
        assert np.array_equal(i1[0], idx[r]) and np.array_equal(l1[0].view(np.uint32), lp[r].view(np.uint32))
    i2, l2, s2 = _run(ts, x, 20, b.temperature, dev)
    assert np.array_equal(i2, idx) and np.array_equal(l2.view(np.uint32), lp.view(np.uint32))
