"""vsamp_sample_static, the split-vocabulary draw on the library's fixed device scratch array (no
allocation), against vsamp_sample_ws on the same inputs: bit-identical outputs on two calls in a row and
across shapes, and a batch beyond the array refused before any device work. The file name sorts last so
the test also runs after every other GPU test in one session."""
import re

import numpy as np
import pytest

import parity_util
import workloads

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ts():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as g

    g.build()
    import top_sampling_gb300 as ts_mod

    ts_mod.load()
    return ts_mod


@pytest.fixture(scope="module")
def dev():
    return torch.device("cuda:0")


def _draw(fn, b, x, dev, step):
    t = parity_util.t
    return fn(x, temperature=t(b.temperature, dev), top_k=t(b.top_k, dev), top_p=t(b.top_p, dev),
              min_p=t(b.min_p, dev), seed=t(b.seed, dev), step=t(np.full(b.B, step, np.uint64), dev), V=b.V,
              want_stats=True)


def _host(out):
    tok, lp, st, stats = out
    return tok.cpu().numpy(), lp.cpu().numpy().view(np.int32), st.cpu().numpy(), stats.cpu().numpy()


def test_header_and_binding_agree_on_the_scratch_limit():
    import top_sampling_gb300 as ts_mod

    src = open(parity_util.__file__.replace("tests/parity_util.py", "include/vsamp.h")).read()
    m = re.search(r"#define VSAMP_STATIC_SCRATCH_BYTES (\d+)", src)
    assert m and int(m.group(1)) == ts_mod.VSAMP_STATIC_SCRATCH_BYTES
    m = re.search(r"VSAMP_ERR_SCRATCH_LIMIT = (\d+)", src)
    assert m and int(m.group(1)) == ts_mod.VSAMP_ERR_SCRATCH_LIMIT


@pytest.mark.gpu
def test_static_scratch_matches_the_workspace_entry_point_on_two_calls_in_a_row(ts, dev):
    # three shapes one after another: fp32 rows with per-row filters, bf16 rows with large logits, a small batch
    for b in (workloads.c2(B=16), workloads.c4(B=32), workloads.c1()):
        x = parity_util.to_device(b.logits, b.dtype, dev)
        want = [_host(_draw(ts.vsamp_sample_ws, b, x, dev, step)) for step in (0, 1)]
        torch.cuda.synchronize()
        got = [_draw(ts.vsamp_sample_static, b, x, dev, step) for step in (0, 1)]   # back to back
        torch.cuda.synchronize()
        for step in (0, 1):
            g, w = _host(got[step]), want[step]
            assert (w[2] == 0).all(), (b.name, step)
            for name, a, e in zip(("token", "logprob bits", "row_status", "stats"), g, w):
                np.testing.assert_array_equal(a, e, err_msg=f"{b.name} step {step}: {name}")


@pytest.mark.gpu
def test_static_scratch_calls_leave_free_device_memory_unchanged(ts, dev):
    """The property the entry point exists for: after a first call (which looks up the array's address),
    further calls with caller-owned outputs change no device allocation."""
    b = workloads.c2(B=16)
    x = parity_util.to_device(b.logits, b.dtype, dev)
    t = parity_util.t
    args = dict(temperature=t(b.temperature, dev), top_k=t(b.top_k, dev), top_p=t(b.top_p, dev),
                min_p=t(b.min_p, dev), seed=t(b.seed, dev), step=t(b.step, dev), V=b.V,
                token=torch.empty(b.B, dtype=torch.int32, device=dev),
                logprob=torch.empty(b.B, dtype=torch.float32, device=dev),
                row_status=torch.empty(b.B, dtype=torch.int32, device=dev),
                stats=torch.empty((b.B, 4), dtype=torch.int32, device=dev), want_stats=True)
    ts.vsamp_sample_static(x, **args)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    for _ in range(5):
        ts.vsamp_sample_static(x, **args)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0, (free0, free1)
    assert int(args["row_status"].ne(0).sum()) == 0


@pytest.mark.gpu
def test_static_scratch_refuses_a_batch_beyond_its_size(ts, dev):
    lib = ts.load()
    V = 151936
    size = lambda b: int(lib.vsamp_sample_workspace_size(ts.VSAMP_BF16, b, V))
    per_row, fixed = size(2) - size(1), 2 * size(1) - size(2)   # the size is fixed + per_row * B
    B = (ts.VSAMP_STATIC_SCRATCH_BYTES - fixed) // per_row + 1
    assert size(B) > ts.VSAMP_STATIC_SCRATCH_BYTES >= size(B - 1)
    # full-size buffers although the call is refused on the host before any launch
    x = torch.empty((B, V), dtype=torch.bfloat16, device=dev)
    token = torch.full((B,), -7, dtype=torch.int32, device=dev)
    with pytest.raises(ts.VsampError) as e:
        ts.vsamp_sample_static(x, token=token, want_logprob=False)
    assert e.value.status == ts.VSAMP_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert int(token.ne(-7).sum()) == 0
    # one row fewer than the limit allows is accepted
    B_ok = B - 1
    tok, _, st, _ = ts.vsamp_sample_static(x[:B_ok].zero_(), want_logprob=False)
    torch.cuda.synchronize()
    assert int(st.ne(0).sum()) == 0
    assert int(tok.lt(0).sum()) == 0
