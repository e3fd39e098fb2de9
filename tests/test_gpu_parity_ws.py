"""GPU parity of vsamp_sample_ws (split vocabulary, workspace): every sampling check of test_gpu_parity.py,
run again through the workspace entry point, plus the workspace contract (no initialisation needed, too small or
unaligned refused before launch)."""
import numpy as np
import pytest

import parity_util
import workloads
from test_gpu_parity import *  # noqa: F401,F403  (fixtures and the parity checks, re-run below)
from test_gpu_parity import dev, ts  # noqa: F401

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _through_the_workspace_entry_point():
    old = parity_util.SAMPLE_FN
    parity_util.SAMPLE_FN = "vsamp_sample_ws"
    yield
    parity_util.SAMPLE_FN = old


def test_workspace_needs_no_initialisation(ts, dev):
    """Every call writes what it reads: a workspace full of arbitrary bytes, or one left by calls of other shapes,
    gives the same outputs as a zero-filled one."""
    b = workloads.c1()
    x = parity_util.to_device(b.logits, b.dtype, dev)
    need = int(ts.load().vsamp_sample_workspace_size(ts.VSAMP_F32, b.logits.shape[0], b.V))
    kw = dict(temperature=parity_util.t(b.temperature, dev), top_k=parity_util.t(b.top_k, dev),
              top_p=parity_util.t(b.top_p, dev), seed=parity_util.t(b.seed, dev), want_stats=True)
    zero = torch.zeros(need, dtype=torch.uint8, device=dev)
    want = [a.cpu().numpy() for a in ts.vsamp_sample_ws(x, workspace=zero, **kw) if a is not None]
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    for fill in ("ones", "random", "reused"):
        if fill == "ones":
            ws = torch.full((need,), 255, dtype=torch.uint8, device=dev)
        elif fill == "random":
            ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device=dev, generator=g)
        else:   # a workspace last used by a call of another shape
            ws = torch.zeros(need, dtype=torch.uint8, device=dev)
            other = workloads.c1(B=2, V=5000, seed=3)
            ts.vsamp_sample_ws(parity_util.to_device(other.logits, other.dtype, dev), workspace=ws)
        for _ in range(2):
            got = [a.cpu().numpy() for a in ts.vsamp_sample_ws(x, workspace=ws, **kw) if a is not None]
            torch.cuda.synchronize()
            for a, e in zip(got, want):
                np.testing.assert_array_equal(a.view(np.int32), e.view(np.int32), err_msg=fill)


def test_workspace_too_small_or_unaligned_is_refused(ts, dev):
    b = workloads.c1()
    x = parity_util.to_device(b.logits, b.dtype, dev)
    need = int(ts.load().vsamp_sample_workspace_size(ts.VSAMP_F32, b.logits.shape[0], b.V))
    small = torch.zeros(need - 16, dtype=torch.uint8, device=dev)
    with pytest.raises(ts.VsampError) as e:
        ts.vsamp_sample_ws(x, workspace=small)
    assert e.value.status == ts.VSAMP_ERR_INVALID_ARG
    big = torch.zeros(need + 64, dtype=torch.uint8, device=dev)
    with pytest.raises(ts.VsampError) as e:
        ts.vsamp_sample_ws(x, workspace=big[1:])
    assert e.value.status == ts.VSAMP_ERR_INVALID_ARG
