"""The benchmark's reporting on CPU: the reference arm's JSON line, and the DRAM traffic that `bench.py` takes
from the committed machine-readable ncu record only while that record describes the current kernel sources."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_follows_the_profile_digest(tmp_path, monkeypatch):
    good = tmp_path / "good.json"
    good.write_text(json.dumps({"source_digest": bench._csrc_digest(), "dram_bytes_per_launch": 123456}))
    monkeypatch.setattr(bench, "PROFILE", str(good))
    assert bench._traffic() == 123456
    stale = tmp_path / "stale.json"
    stale.write_text(json.dumps({"source_digest": "0000000000000000", "dram_bytes_per_launch": 123456}))
    monkeypatch.setattr(bench, "PROFILE", str(stale))
    assert bench._traffic() is None
    monkeypatch.setattr(bench, "PROFILE", str(tmp_path / "missing.json"))
    assert bench._traffic() is None


def test_committed_profile_record_is_machine_readable():
    with open(os.path.join(ROOT, "profiles", "sample_kernel_c4.json")) as f:
        rec = json.load(f)
    assert len(rec["source_digest"]) == 16 and int(rec["dram_bytes_per_launch"]) > 0
    assert "ncu" in rec["command"] and "--clock-control none" in rec["command"]


def test_digest_covers_every_kernel_source(tmp_path, monkeypatch):
    # the digest changes with any file of the kernel sources (name or content)
    d0 = bench._csrc_digest()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "top_sampling_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "a.cu").write_text("x")
    d1 = bench._csrc_digest()
    (src / "a.cu").write_text("y")
    d2 = bench._csrc_digest()
    assert len({d0, d1, d2}) == 3


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["unit"] == "rows/s" and out["value"] > 0
    assert out["higher_is_better"] is True and out["n_gpus"] == 1 and out["steps"] == 1
    assert out["e2e"] == {"value": out["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] >= 1
    assert out["config"]["B"] == 256 and out["config"]["V"] == 151936
