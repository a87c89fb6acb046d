"""The benchmark's reference arm on CPU: `bench.py --impl reference` times the
float64 oracle on host cores and prints one JSON line with the keys the
benchmark contract names (metric, value, unit, steps, warm-up, the reference
tag, a CPU baseline describing the run and an end-to-end figure with no
host-device bytes). Also the helpers that tie roofline traffic to the
committed ncu summaries: a summary counts only while its recorded source
hash matches the kernel source."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload", ["llama8k", "prefill512"])
def test_reference_arm_prints_one_contract_line(workload):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload, "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["steps"] == 1 and d["n_gpus"] == 1 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_profile_traffic_needs_the_current_source(tmp_path, monkeypatch):
    """A summary's DRAM bytes count only while its recorded hash matches the
    kernel source it names."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "paged_kv_cache_209_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "pkv_decode.cu").write_text("// kernel v1\n")
    sha = bench.kernel_source_sha(("pkv_decode.cu",))
    assert len(sha) == 16
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "s.md").write_text(f"source_sha: {sha}   (note)\n\ndram_bytes_per_call: 123456\n")
    assert bench.profiled_traffic("s") == 123456
    assert bench.profiled_traffic("missing") is None
    (src / "pkv_decode.cu").write_text("// kernel v2\n")     # the kernel changed since the capture
    assert bench.profiled_traffic("s") is None
