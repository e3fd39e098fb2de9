"""vsamp_topk_select at the shapes of the sparse-attention indexer ("[Kernel] Make persistent_topk deterministic":
Test plan, the short-row regression and the wide-row fallback runs): TopK 512/1024/2048, rows of a few hundred
tokens up to 474,112, random, tie-heavy, all-equal and narrow-range keys. Every output is compared with the
binary64 oracle bit for bit, and repeated calls must be identical."""
import numpy as np
import pytest

import workloads
from oracle import sampler as osm

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from parity_util import t  # noqa: E402


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


def _keys(rng, kind, n):
    if kind == "random":
        return rng.standard_normal(n).astype(np.float32)
    if kind == "ties":        # 64 levels: thousands of equal keys at any threshold
        return (rng.integers(0, 64, n) / 8.0).astype(np.float32)
    if kind == "equal":
        return np.full(n, 0.75, np.float32)
    if kind == "narrow":      # every key in one coarse bin: 1 + j * 2^-23 for j < 4096
        return (1.0 + rng.integers(0, 4096, n) * 2.0 ** -23).astype(np.float32)
    raise ValueError(kind)


def _run_and_check(ts, dev, x, lengths, k, repeats=2, dtype="f32"):
    """fp32 keys x, selected as fp32 or as their bfloat16 roundings (dtype "bf16")."""
    B, ld = x.shape
    if dtype == "bf16":
        x = workloads.f32_to_bf16_bits(x)
        xd = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        xd = torch.from_numpy(x).to(dev)
    outs = []
    for _ in range(repeats):
        idx, st = ts.vsamp_topk_select(xd, k, k_max=k, lengths=t(lengths, dev), max_len=ld)
        torch.cuda.synchronize()
        outs.append((idx.cpu().numpy(), st.cpu().numpy()))
    for idx, st in outs[1:]:
        assert np.array_equal(idx, outs[0][0]) and np.array_equal(st, outs[0][1])
    idx, st = outs[0]
    for r in range(B):
        s_o, want = osm.topk_select_row(x[r], int(lengths[r]), k, k, dtype=dtype)
        assert st[r] == s_o, f"row {r}"
        assert np.array_equal(idx[r], want), f"row {r} (length {lengths[r]}, k {k})"


@pytest.mark.parametrize("k", [512, 1024, 2048])
def test_short_rows_are_padded(ts, dev, k):
    """Rows of 256-2048 tokens: a row no longer than k returns its indices in order, then -1."""
    rng = np.random.default_rng(k)
    lengths = np.linspace(256, 2048, 33).astype(np.int32)
    x = np.stack([_keys(rng, "random", 2048) for _ in range(33)])
    _run_and_check(ts, dev, x, lengths, k)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows", [1, 8, 64])
@pytest.mark.parametrize("k", [512, 2048])
@pytest.mark.parametrize("kind", ["random", "ties"])
def test_indexer_lengths(ts, dev, rows, k, kind, dtype):
    """Rows {1, 8, 64} x lengths {1k, 4k, 8k, 20k, 40k} x k {512, 2048} x {random, tie-heavy}, fp32 and bf16."""
    rng = np.random.default_rng(rows * 7 + k)
    lens = np.array([1024, 4096, 8192, 20480, 40960], dtype=np.int32)
    lengths = lens[np.arange(rows) % lens.size]
    x = np.stack([_keys(rng, kind, 40960) for _ in range(rows)])
    _run_and_check(ts, dev, x, lengths, k, dtype=dtype)


@pytest.mark.parametrize("kind", ["equal", "narrow"])
def test_all_equal_and_narrow_range(ts, dev, kind):
    """All keys equal give exactly [0, k); keys inside one coarse histogram bin lose no candidate."""
    rng = np.random.default_rng(3)
    lengths = np.array([4096, 20000, 40960, 2048], dtype=np.int32)
    x = np.stack([_keys(rng, kind, 40960) for _ in range(4)])
    _run_and_check(ts, dev, x, lengths, 2048)
    if kind == "equal":
        idx, _ = ts.vsamp_topk_select(torch.from_numpy(x).to(dev), 2048, lengths=t(lengths, dev))
        idx = idx.cpu().numpy()
        assert np.array_equal(idx[0], np.arange(2048))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ties", [2047, 4096, 16385])
def test_pivot_tie_populations(ts, dev, ties, dtype):
    """k - 1 keys above one level that is shared by `ties` keys: the lowest-index one of them is taken."""
    rng = np.random.default_rng(ties)
    n, k = 40960, 2048
    x = rng.uniform(-2.0, -1.0, n).astype(np.float32)
    pos = rng.permutation(n)
    x[pos[:k - 1]] = rng.uniform(1.0, 2.0, k - 1).astype(np.float32)
    x[pos[k - 1:k - 1 + ties]] = 0.5
    if dtype == "bf16":   # keep the populations exact after rounding: above 1.0, at 0.5, below -1.0
        x[pos[:k - 1]] = 1.5
        x[pos[k - 1 + ties:]] = -1.5
    _run_and_check(ts, dev, x[None, :].copy(), np.array([n], np.int32), k, dtype=dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("width", [355588, 400000, 474112])
@pytest.mark.parametrize("k", [512, 2048])
def test_wide_rows(ts, dev, width, k, dtype):
    """Contiguous rows (stride = length) of 355,588 to 474,112 keys: random, tie-heavy, all-equal."""
    rng = np.random.default_rng(width + k)
    x = np.stack([_keys(rng, kind, width) for kind in ("random", "ties", "equal", "random")])
    _run_and_check(ts, dev, x, np.full(4, width, np.int32), k, dtype=dtype)


# ------------------------------------------------------------------------------------------------
# the uncached path: rows longer than a thread-block cluster holds on chip ("[Kernel] Make persistent_topk
# deterministic", the wide-row fallback runs), and the same path forced on the shapes above
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("width", [1 << 20, 2 << 20])
def test_rows_beyond_on_chip_capacity(ts, dev, width, dtype):
    """1 M and 2 M keys per row (past the on-chip capacity for fp32; 2 M also for bf16): random, tie-heavy and
    all-equal rows, bit-exact, where the on-chip select would refuse the row."""
    lim = ts.device_info(0)
    cap = lim.max_row_f32 if dtype == "f32" else lim.max_row_bf16
    rng = np.random.default_rng(width)
    x = np.stack([_keys(rng, kind, width) for kind in ("random", "ties", "equal")])
    for k in (512, 2048):
        _run_and_check(ts, dev, x, np.full(3, width, np.int32), k, repeats=2, dtype=dtype)
    if width <= cap:
        pytest.skip(f"{width} keys fit on chip ({cap}): the on-chip path ran")


@pytest.fixture
def forced_stream():
    import os

    old = os.environ.get("VSAMP_SELECT_STREAM")
    os.environ["VSAMP_SELECT_STREAM"] = "1"
    yield
    if old is None:
        os.environ.pop("VSAMP_SELECT_STREAM", None)
    else:
        os.environ["VSAMP_SELECT_STREAM"] = old


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("k", [512, 2048])
@pytest.mark.parametrize("kind", ["random", "ties", "equal", "narrow"])
def test_uncached_path_on_indexer_shapes(ts, dev, forced_stream, k, kind, dtype):
    rng = np.random.default_rng(k + len(kind))
    lens = np.array([256, 1024, 4096, 20480, 40960, 2048], dtype=np.int32)
    x = np.stack([_keys(rng, kind, 40960) for _ in range(lens.size)])
    _run_and_check(ts, dev, x, lens, k, dtype=dtype)


def test_uncached_path_contract_edges(ts, dev, forced_stream):
    rng = np.random.default_rng(8)
    B, L = 6, 5000
    x = (rng.integers(0, 3, size=(B, L)) * 1.0).astype(np.float32)
    x[0, :4] = [np.inf, -np.inf, np.inf, -np.inf]
    x[1, 100:] = np.nan                      # beyond its length: never read
    x[2, 10] = np.nan                        # inside: a row error
    lengths = np.array([L, 100, 50, 3000, 0, L + 1], dtype=np.int32)
    ks = np.array([64, 64, 64, 0, 10, 10], dtype=np.int32)
    idx, st = ts.vsamp_topk_select(torch.from_numpy(x).to(dev), t(ks, dev), k_max=64, lengths=t(lengths, dev),
                                   max_len=L)
    idx, st = idx.cpu().numpy(), st.cpu().numpy()
    for r in range(B):
        s_o, want = osm.topk_select_row(x[r], int(lengths[r]), int(ks[r]), 64) if 0 < lengths[r] <= L else \
            (osm.STATUS_INVALID_ARG, np.full(64, -1, dtype=np.int32))
        assert st[r] == s_o and np.array_equal(idx[r], want), r
    idx, st = ts.vsamp_topk_select(torch.from_numpy(x).to(dev), t(np.full(B, 65, np.int32), dev), k_max=64)
    want_st = [osm.topk_select_row(x[r], L, 65, 64)[0] for r in range(B)]
    assert list(st.cpu().numpy()) == want_st and np.all(idx.cpu().numpy() == -1)


def test_uncached_path_on_the_quantised_workload(ts, dev, forced_stream):
    b = workloads.c3(B=32)
    x = torch.from_numpy(b.scores).to(dev)
    idx, st = ts.vsamp_topk_select(x, t(b.k, dev), k_max=b.k_max, lengths=t(b.lengths, dev))
    idx, st = idx.cpu().numpy(), st.cpu().numpy()
    for r in range(b.B):
        s_o, want = osm.topk_select_row(b.scores[r], int(b.lengths[r]), int(b.k[r]), b.k_max)
        assert st[r] == s_o and np.array_equal(idx[r], want), r
