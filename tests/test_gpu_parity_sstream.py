"""GPU parity of the workspace-free streaming sampler (vsamp_sample with VSAMP_SAMPLE_STREAM=1: piece records and
draw codes gathered in the first CTA of a cluster, which finishes the row): every sampling check of
test_gpu_parity.py run again through it, and bit identity with vsamp_sample_ws, whose piece pass and row finish
are the same code over a workspace."""
import os

import numpy as np
import pytest

import parity_util
import workloads
from test_gpu_parity import *  # noqa: F401,F403  (fixtures and the parity checks, re-run below)
from test_gpu_parity import dev, ts  # noqa: F401

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _through_the_streaming_sampler():
    old = os.environ.get("VSAMP_SAMPLE_STREAM")
    os.environ["VSAMP_SAMPLE_STREAM"] = "1"
    yield
    if old is None:
        os.environ.pop("VSAMP_SAMPLE_STREAM", None)
    else:
        os.environ["VSAMP_SAMPLE_STREAM"] = old


@pytest.mark.parametrize("name,rows", [("c1", 4), ("c2", 16), ("c4", 32)])
def test_bit_identical_to_the_workspace_entry_point(ts, dev, name, rows):
    b = getattr(workloads, name)()
    x = parity_util.to_device(np.ascontiguousarray(b.logits[:rows]), b.dtype, dev)
    t = parity_util.t
    kw = dict(temperature=t(b.temperature[:rows], dev), top_k=t(b.top_k[:rows], dev), top_p=t(b.top_p[:rows], dev),
              min_p=t(b.min_p[:rows], dev), seed=t(b.seed[:rows], dev), step=t(b.step[:rows], dev), want_stats=True)
    a = [v.cpu().numpy() for v in ts.vsamp_sample(x, **kw)]
    w = [v.cpu().numpy() for v in ts.vsamp_sample_ws(x, **kw)]
    for got, want in zip(a, w):
        np.testing.assert_array_equal(got.view(np.int32), want.view(np.int32))
