"""bench.py prints one JSON line with the keys its readers rely on, for every
workload, for the study modes and for the reference arm (short runs)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("workload", ["c1", "c2", "c3", "c4", "c5"])
def test_bench_line_keys(workload):
    d = _run("--workload", workload, "--steps", "3", "--warmup", "3", "--e2e-steps", "1",
             "--no-cpu-baseline")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
                "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"].startswith(workload)
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] >= d["steps"]
    if workload == "c3":
        assert "sigma" in d["config"]


def test_cpu_baseline_and_reference_arm():
    d = _run("--workload", "c1", "--steps", "3", "--warmup", "3", "--e2e-steps", "1")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    r = _run("--impl", "reference", "--workload", "c1", "--steps", "2", "--warmup", "3")
    assert r["impl"] == "reference" and r["value"] > 0 and r["e2e"]["h2d_bytes_per_step"] == 0


@pytest.mark.parametrize("study", ["fanout", "csweep"])
def test_study_lines(study):
    d = _run("--study", study, "--batch", "16", "--study-draws", "1", "--study-rounds", "2",
             "--warmup", "3")
    assert d["study"] == study and len(d["rows"]) > 0
    for row in d["rows"]:
        assert 0.0 <= row["hit_rate"] <= 1.0
