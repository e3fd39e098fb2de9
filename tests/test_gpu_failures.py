"""Failure detection on the GPU without a fault: capacity limits and bounded device-side waits.

* A device that cannot hold the row: `VSAMP_SMEM_OPTIN_OVERRIDE` makes the library believe the
  device has less shared memory, so a row that no cluster can hold is refused before launch with
  VSAMP_ERR_UNSUPPORTED and nothing is written.
* A wait that runs out: `VSAMP_TEST_DROP_LOADS` arms each row load on its mbarrier but never issues the
  copy, so every load wait ends at its bound (`VSAMP_WAIT_CYCLES`, about a millisecond here); the rows
  report VSAMP_ERR_TIMEOUT with sentinel outputs and the context stays usable: the next call in the
  same process is checked against the oracle.

Each case runs in a child process because the library reads its device limits once per process.
"""
import json
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD_CAPACITY = textwrap.dedent("""
    import json, sys, torch
    import top_sampling_gb300 as ts
    ts.load()
    lim = ts.device_info(0)
    dev = torch.device("cuda:0")
    V = 151936
    x = torch.randn(2, V, device=dev)
    tok = torch.full((2,), 7, dtype=torch.int32, device=dev)
    try:
        ts.vsamp_sample(x, token=tok)
        status = 0
    except ts.VsampError as e:
        status = e.status
    torch.cuda.synchronize()
    print(json.dumps({"status": status, "max_row_f32": int(lim.max_row_f32), "tok": tok.cpu().tolist()}))
""")

CHILD_TIMEOUT = textwrap.dedent("""
    import json, os, sys, math, torch
    sys.path.insert(0, ".")
    import numpy as np
    import top_sampling_gb300 as ts, workloads
    from tests import parity_util as pu
    ts.load()
    dev = torch.device("cuda:0")
    b = workloads.c1()
    os.environ["VSAMP_TEST_DROP_LOADS"] = "1"
    os.environ["VSAMP_WAIT_CYCLES"] = "2000000"
    tok, lp, st, stats = pu.run_sample(ts, b, dev)
    del os.environ["VSAMP_TEST_DROP_LOADS"]
    del os.environ["VSAMP_WAIT_CYCLES"]
    first = {"status": st.tolist(), "tok": tok.tolist(), "lp_nan": [bool(math.isnan(v)) for v in lp]}
    tok2, lp2, st2, stats2 = pu.run_sample(ts, b, dev)
    ties = pu.TieCounter()
    pu.check_sample(b, range(b.logits.shape[0]), tok2, lp2, st2, stats2, ties)
    print(json.dumps({"first": first, "second_ok": True}))
""")


def _run(code, env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.gpu
def test_row_too_long_for_the_device_is_refused_before_launch():
    out = _run(CHILD_CAPACITY, {"VSAMP_SMEM_OPTIN_OVERRIDE": "16384"})
    assert out["max_row_f32"] < 151936
    assert out["status"] == 2                      # VSAMP_ERR_UNSUPPORTED
    assert out["tok"] == [7, 7]                    # nothing was enqueued


@pytest.mark.gpu
def test_load_wait_that_runs_out_reports_timeout_and_context_survives():
    out = _run(CHILD_TIMEOUT, {})
    first = out["first"]
    assert first["status"] == [5, 5, 5, 5]         # VSAMP_ERR_TIMEOUT on every row
    assert first["tok"] == [-1, -1, -1, -1]
    assert all(first["lp_nan"])
    assert out["second_ok"]
