"""GPU parity of the vocabulary-sharded entry points (vsamp_shard_partial + the owned vsamp_shard_merge): R shards
of each row on one device, merged from the rank-ordered records, against the unsharded entry points and the
binary64 oracle. Max and arg-max decompose over shards ("[WS2][Logprob] Deterministic SM90 linear_logp ...",
Tensor parallelism: rank order + owned merge), so the drawn token must equal the unsharded draw exactly; with
shard boundaries on piece boundaries every output must be bit-identical to vsamp_sample_ws for every R."""
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


def _unfiltered(b):
    """The batch with top-k, top-p and min-p off: the sharded draw is over the full distribution."""
    b.top_k[:] = 0
    b.top_p[:] = 1.0
    b.min_p[:] = 0.0
    return b


def _kw(b, dev):
    return dict(temperature=t(b.temperature, dev), seed=t(b.seed, dev), step=t(b.step, dev))


def _bits(a):
    a = a.cpu().numpy()
    return a.view(np.int32) if a.dtype == np.float32 else a


WORKLOADS = [("c1", lambda: workloads.c1()), ("c2", lambda: workloads.c2(B=16)),
             ("c4", lambda: workloads.c4(B=16)), ("c5", lambda: workloads.c5(B=16))]


@pytest.mark.parametrize("name,make", WORKLOADS)
@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_piece_aligned_shards_are_bit_identical_to_the_unsharded_streaming_sampler(ts, dev, name, make, R):
    b = _unfiltered(make())
    x = to_device(b.logits, b.dtype, dev)
    kw = _kw(b, dev)
    tok_ws, lp_ws, st_ws, _ = ts.vsamp_sample_ws(x, **kw)
    tok_c, _, _, _ = ts.vsamp_sample(x, **kw)
    m_ref, ls_ref, _ = ts.vsamp_softmax_lse(x, temperature=kw["temperature"])
    m, ls, tok, lp, _, st = ts.vsamp_sample_sharded(x, R, **kw)
    torch.cuda.synchronize()
    assert int(st.ne(0).sum()) == 0 and int(st_ws.ne(0).sum()) == 0
    assert np.array_equal(_bits(tok), _bits(tok_ws)), (name, R)
    assert np.array_equal(_bits(lp), _bits(lp_ws)), (name, R)              # same pieces, same fold: same bits
    assert np.array_equal(_bits(tok), _bits(tok_c)), (name, R)             # the cluster path draws the same token
    assert np.array_equal(_bits(m), _bits(m_ref))
    assert float((ls - ls_ref).abs().max()) <= LOGP_TOL


@pytest.mark.parametrize("name,make", WORKLOADS)
def test_any_shard_count_draws_the_same_token(ts, dev, name, make):
    """Vector-aligned (not piece-aligned) boundaries: the fold's last bits may move, the token may not."""
    b = _unfiltered(make())
    x = to_device(b.logits, b.dtype, dev)
    kw = _kw(b, dev)
    tok_ws, lp_ws, _, _ = ts.vsamp_sample_ws(x, **kw)
    for R in (2, 3, 5, 8):
        m, ls, tok, lp, _, st = ts.vsamp_sample_sharded(x, R, align_to_pieces=False, **kw)
        torch.cuda.synchronize()
        assert int(st.ne(0).sum()) == 0
        assert np.array_equal(_bits(tok), _bits(tok_ws)), (name, R)
        assert float((lp - lp_ws).abs().max()) <= LOGP_TOL


@pytest.mark.parametrize("name,make", WORKLOADS)
def test_merged_draw_and_logprobs_against_the_oracle(ts, dev, name, make):
    b = _unfiltered(make())
    x = to_device(b.logits, b.dtype, dev)
    kw = _kw(b, dev)
    rng = np.random.default_rng(5)
    target = rng.integers(0, b.V, size=b.B).astype(np.int32)
    m, ls, tok, lp, tlp, st = ts.vsamp_sample_sharded(x, 4, target=t(target, dev), **kw)
    torch.cuda.synchronize()
    tok, lp, tlp, ls = tok.cpu().numpy(), lp.cpu().numpy(), tlp.cpu().numpy(), ls.cpu().numpy()
    near = 0
    for r in range(b.B):
        ref = osm.sample_row(b.logits[r], b.dtype, b.temperature[r], 0, 1.0, 0.0, int(b.seed[r]), r, int(b.step[r]))
        assert not ref.ambiguous
        if ref.near_tie:
            near += 1
        else:
            assert tok[r] == ref.token, (name, r)
        assert abs(float(lp[r]) - osm.logprob_row(b.logits[r], b.dtype, b.temperature[r], int(tok[r]))) <= LOGP_TOL
        assert abs(float(tlp[r]) - osm.logprob_row(b.logits[r], b.dtype, b.temperature[r], int(target[r]))) <= LOGP_TOL
        assert abs(float(ls[r]) - ref.row_logsum) <= LOGP_TOL
    assert near == 0


def test_greedy_rows_errors_and_unowned_targets(ts, dev):
    rng = np.random.default_rng(3)
    B, V = 6, 8192
    x = (rng.integers(-4, 4, size=(B, V)) * 0.5).astype(np.float32)
    x[0, [5000, 6000, 7000]] = 9.0          # greedy: the first of tied maxima, in another shard than index 0
    x[2, 4321] = np.nan
    x[3, 17] = np.inf
    T = np.array([0.0, 1.0, 1.0, 1.0, np.nan, -1.0], dtype=np.float32)
    xd = torch.from_numpy(x).to(dev)
    temp = t(T, dev)
    m, ls, tok, lp, _, st = ts.vsamp_sample_sharded(xd, 4, temperature=temp, seed=7)
    torch.cuda.synchronize()
    st, tok, lp = st.cpu().numpy(), tok.cpu().numpy(), lp.cpu().numpy()
    assert list(st) == [0, 0, osm.STATUS_NONFINITE, osm.STATUS_NONFINITE, osm.STATUS_INVALID_ARG, 0]
    assert tok[0] == 5000 and tok[5] == int(np.argmax(x[5])) and lp[0] == pytest.approx(
        osm.logprob_row(x[0], "f32", 1.0, 5000), abs=LOGP_TOL)
    assert np.all(tok[2:5] == -1) and np.all(np.isnan(lp[2:5]))
    ref = osm.sample_row(x[1], "f32", 1.0, 0, 1.0, 0.0, 7, 1, 0)
    assert tok[1] == ref.token or ref.near_tie
    # a target outside the vocabulary is owned by no shard: a row error
    tgt = t(np.array([1, V + 5, 1, 1, 1, 1], np.int32), dev)
    _, _, _, _, tlp, st2 = ts.vsamp_sample_sharded(xd, 4, temperature=temp, seed=7, target=tgt)
    torch.cuda.synchronize()
    assert int(st2[1]) == osm.STATUS_INVALID_ARG and math.isnan(float(tlp[1]))
    assert int(st2[0]) == 0 and abs(float(tlp[0]) - osm.logprob_row(x[0], "f32", 1.0, 1)) <= LOGP_TOL


def test_shard_calls_are_deterministic_and_refuse_bad_arguments(ts, dev):
    b = _unfiltered(workloads.c1(B=3))
    x = to_device(b.logits, b.dtype, dev)
    kw = _kw(b, dev)
    first = [a.clone() for a in ts.vsamp_sample_sharded(x, 4, **kw) if a is not None]
    again = [a for a in ts.vsamp_sample_sharded(x, 4, **kw) if a is not None]
    torch.cuda.synchronize()
    assert all(np.array_equal(_bits(a), _bits(c)) for a, c in zip(first, again))
    with pytest.raises(ts.VsampError):                      # v0 not a multiple of the fp32 vector (4 logits)
        ts.vsamp_shard_partial(x[:, 2:1000], 2, 1, **kw)
    with pytest.raises(ts.VsampError):                      # fewer record slots than the shard's pieces
        ts.vsamp_shard_partial(x[:, 0:4096], 0, 2, **kw)
