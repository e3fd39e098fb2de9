"""GPU parity of vsamp_sample_ws (split vocabulary, workspace): every sampling check of test_gpu_parity.py,
run again through the workspace entry point, plus the workspace contract (left zero-filled, too small or
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


def test_workspace_is_left_zero_filled(ts, dev):
    b = workloads.c1()
    x = parity_util.to_device(b.logits, b.dtype, dev)
    need = int(ts.load().vsamp_sample_workspace_size(ts.VSAMP_F32, b.logits.shape[0], b.V))
    ws = torch.zeros(need + 64, dtype=torch.uint8, device=dev)
    for _ in range(3):
        tok, _, st, _ = ts.vsamp_sample_ws(x, temperature=parity_util.t(b.temperature, dev),
                                           top_k=parity_util.t(b.top_k, dev), top_p=parity_util.t(b.top_p, dev),
                                           seed=parity_util.t(b.seed, dev), workspace=ws)
        torch.cuda.synchronize()
        assert int(st.ne(0).sum()) == 0
        # the reserved header and the per-row counters and draw slots are back to zero
        assert int(ws[:256].ne(0).sum()) == 0
        plans = ws[256: 256 + 128 * b.logits.shape[0]].view(-1, 128)
        assert int(plans[:, :16].ne(0).sum()) == 0


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
