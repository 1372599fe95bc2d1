"""The bench's JSON line: one short run of each arm, checked for the keys and
the consistency the measurement depends on (the numbers themselves are the
bench's business, not a test's)."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()
    yield


def _run(*args):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_carries_the_contract():
    d = _run("--steps", "2", "--warmup", "3", "--no-cpu-baseline", "--no-sweep")
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["dtype"] == "bf16" and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["config"]["workload"] == "dense_t8192" and "l2" in d["config"]
    calls = d["launch"]["calls_per_step"]
    # whole-job bytes over time: the value follows from the per-call time and the bytes
    assert d["value"] == pytest.approx(d["alg_bytes_per_call"] / (d["us_per_call"] * 1e-6) / 1e9, rel=0.02)
    assert d["ms_per_step"] == pytest.approx(d["us_per_call"] * calls / 1e3, rel=0.02)
    assert d["gpu_launches"] == 2 * calls * d["steps"]
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-3)
    assert rf["achieved"] == pytest.approx(rf["alg_bytes_per_launch"] / (rf["us_per_launch"] * 1e-6) / 1e9, rel=0.02)
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == "GB/s" and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = d["clocks"]
    assert c["sm_mhz"] > 0 and c["sm_max_mhz"] > 0 and isinstance(c["reasons"], list)


def test_reference_arm_line():
    d = _run("--impl", "reference", "--steps", "1", "--warmup", "3")
    ours = _run("--steps", "1", "--warmup", "3", "--no-cpu-baseline", "--no-sweep")
    assert d["impl"] == "reference" and d["config"] == ours["config"]
    assert d["metric"] == ours["metric"] and d["unit"] == ours["unit"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
