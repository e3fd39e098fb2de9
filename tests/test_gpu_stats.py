"""GPU parity of the streaming row-statistics kernel behind vsamp_softmax_lse and the recomputing vsamp_logprob:
(m, log S) and log-probabilities against the binary64 oracle, agreement with the cluster row kernel
(VSAMP_STATS_ROW=1) on the same rows, invariance to the number of CTAs per row, and its edges: partial last
pieces, unaligned rows (plain loads), rows longer than the kernel takes (the row kernel then runs), non-finite
rows, bad temperatures and tokens."""
import os

import numpy as np
import pytest

import workloads
from oracle import sampler as osm

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from parity_util import LOGP_TOL, t, to_device  # noqa: E402

STATUS_OK, STATUS_INVALID_ARG, STATUS_NONFINITE = osm.STATUS_OK, osm.STATUS_INVALID_ARG, osm.STATUS_NONFINITE


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


class _env:
    """Environment variables set for the duration of a block."""

    def __init__(self, **kv):
        self.kv = kv

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in self.kv}
        os.environ.update({k: str(v) for k, v in self.kv.items()})

    def __exit__(self, *a):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _lse(ts, x, temp, dev, V=None):
    m, ls, st = ts.vsamp_softmax_lse(x, temperature=t(np.asarray(temp, np.float32), dev), V=V)
    torch.cuda.synchronize()
    return m.cpu().numpy(), ls.cpu().numpy(), st.cpu().numpy()


def _check_oracle(rows, dtype, temp, m, ls, st):
    for r in range(len(rows)):
        s_o, m_o, ls_o = osm.softmax_lse_row(rows[r], dtype, float(temp[r]))
        assert st[r] == s_o, r
        if s_o == STATUS_OK:
            assert m[r] == np.float32(m_o), r
            assert abs(float(ls[r]) - ls_o) <= LOGP_TOL, (r, float(ls[r]), ls_o)


@pytest.mark.parametrize("name,rows", [("c4", 16), ("c2", 8), ("c5", 4), ("c1", 4)])
def test_workload_rows_match_the_oracle_and_the_row_kernel(ts, dev, name, rows):
    b = getattr(workloads, name)()
    lg = np.ascontiguousarray(b.logits[:rows])
    temp = b.temperature[:rows]
    x = to_device(lg, b.dtype, dev)
    m, ls, st = _lse(ts, x, temp, dev)
    _check_oracle(lg, b.dtype, temp, m, ls, st)
    with _env(VSAMP_STATS_ROW=1):
        m2, ls2, st2 = _lse(ts, x, temp, dev)
    assert np.array_equal(st, st2)
    assert np.array_equal(m.view(np.uint32), m2.view(np.uint32))
    assert np.max(np.abs(ls - ls2)) <= 4e-6


def test_ctas_per_row_do_not_change_any_bit(ts, dev):
    rng = np.random.default_rng(11)
    for dtype, V in (("f32", 151936), ("bf16", 262144 + 333), ("f32", 40000 + 7)):
        x32 = (rng.normal(0.0, 3.0, size=(6, V))).astype(np.float32)
        lg = workloads.f32_to_bf16_bits(x32) if dtype == "bf16" else x32
        temp = np.array([1.0, 0.7, 1.3, 0.0, 2.0, 0.5], np.float32)
        x = to_device(lg, dtype, dev)
        ref = _lse(ts, x, temp, dev)
        for C in (1, 2, 3, 5, 8):
            with _env(VSAMP_STATS_C=C):
                o = _lse(ts, x, temp, dev)
            assert np.array_equal(o[2], ref[2]), C
            assert np.array_equal(o[0].view(np.uint32), ref[0].view(np.uint32)), C
            assert np.array_equal(o[1].view(np.uint32), ref[1].view(np.uint32)), C
        for cfg in (1, 2):
            with _env(VSAMP_STATS_CFG=cfg):
                o = _lse(ts, x, temp, dev)
            assert np.array_equal(o[1].view(np.uint32), ref[1].view(np.uint32)), cfg
        _check_oracle(lg[:2], dtype, temp[:2], ref[0][:2], ref[1][:2], ref[2][:2])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_partial_pieces_and_unaligned_rows(ts, dev, dtype):
    rng = np.random.default_rng(12)
    V = 5 * 2048 + 17 if dtype == "bf16" else 7 * 1024 + 13
    x32 = rng.normal(0.0, 2.0, size=(3, V + 9)).astype(np.float32)
    lg = workloads.f32_to_bf16_bits(x32) if dtype == "bf16" else x32
    temp = np.array([1.0, 0.9, 1.1], np.float32)
    full = to_device(lg, dtype, dev)
    # padded stride, aligned rows: bulk copies and a partial last piece
    m, ls, st = _lse(ts, full, temp, dev, V=V)
    _check_oracle(np.ascontiguousarray(lg[:, :V]), dtype, temp, m, ls, st)
    # rows shifted by one element: every piece by plain loads
    view = full[:, 1:V + 1]
    m2, ls2, st2 = _lse(ts, view, temp, dev)
    _check_oracle(np.ascontiguousarray(lg[:, 1:V + 1]), dtype, temp, m2, ls2, st2)


def test_rows_longer_than_the_kernel_takes(ts, dev):
    rng = np.random.default_rng(13)
    V = 400 * 1024 + 5                       # 401 pieces of fp32: the cluster row kernel runs
    lg = rng.normal(0.0, 1.0, size=(2, V)).astype(np.float32)
    temp = np.array([1.0, 0.8], np.float32)
    m, ls, st = _lse(ts, to_device(lg, "f32", dev), temp, dev)
    _check_oracle(lg, "f32", temp, m, ls, st)


def test_status_edges(ts, dev):
    rng = np.random.default_rng(14)
    V = 30000
    lg = rng.normal(0.0, 1.0, size=(6, V)).astype(np.float32)
    lg[0, 1234] = np.nan
    lg[1, 29999] = np.inf
    temp = np.array([1.0, 1.0, np.nan, np.inf, 0.0, 1.0], np.float32)
    m, ls, st = _lse(ts, to_device(lg, "f32", dev), temp, dev)
    assert list(st[:4]) == [STATUS_NONFINITE, STATUS_NONFINITE, STATUS_INVALID_ARG, STATUS_INVALID_ARG]
    assert np.isnan(m[:4]).all() and np.isnan(ls[:4]).all()
    # T <= 0 reads as T = 1
    at_one = _lse(ts, to_device(lg[4:5], "f32", dev), np.array([1.0], np.float32), dev)
    assert st[4] == STATUS_OK and ls[4].view(np.uint32) == at_one[1][0].view(np.uint32)
    _check_oracle(lg[4:], "f32", temp[4:], m[4:], ls[4:], st[4:])


def test_logprob_recomputes_the_statistics(ts, dev):
    b = workloads.c4()
    lg = np.ascontiguousarray(b.logits[:6])
    x = to_device(lg, b.dtype, dev)
    toks = np.array([0, 17, b.V - 1, -1, b.V, 4242], np.int32)
    temp = np.array([1.0, 0.5, 2.0, 1.0, 1.0, 0.0], np.float32)
    lp, st = ts.vsamp_logprob(x, t(toks, dev), temperature=t(temp, dev))
    lp, st = lp.cpu().numpy(), st.cpu().numpy()
    assert st[3] == STATUS_INVALID_ARG and st[4] == STATUS_INVALID_ARG
    assert np.isnan(lp[3]) and np.isnan(lp[4])
    for r in (0, 1, 2, 5):
        assert st[r] == STATUS_OK
        want = osm.logprob_row(lg[r], b.dtype, float(temp[r]), int(toks[r]))
        assert abs(float(lp[r]) - want) <= LOGP_TOL, r
    with _env(VSAMP_STATS_ROW=1):
        lp2, st2 = ts.vsamp_logprob(x, t(toks, dev), temperature=t(temp, dev))
    assert np.array_equal(st, st2.cpu().numpy())
    ok = st == STATUS_OK
    assert np.max(np.abs(lp[ok] - lp2.cpu().numpy()[ok])) <= 4e-6
