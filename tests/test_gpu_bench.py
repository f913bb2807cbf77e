"""bench.py end to end on the GPU (tiny workload, few steps): the JSON line
carries every field of the bench contract with sane values."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_on_gpu(cuda_device):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny", "--steps", "5",
                        "--warmup", "3", "--cpu-seconds", "1"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks", "eager"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["value"] > 0
    assert d["gpu_launches"] == 2 * 5
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert set(rf["kernels"]) == {"dispatch_kernel", "combine_kernel"}
    assert "traffic" in rf and (rf["traffic"] is None or rf["traffic"] > 0)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] > 0 and cb["sample"]
    if len(os.sched_getaffinity(0)) > 1:
        ca = d["cpu_baseline_all_cores"]
        assert ca["kind"] == "oracle" and ca["cores"] >= 1 and ca["value"] > 0 and "processes" in ca["sample"]
    assert rf["peak_kind"] and rf["frac_of_nominal"] == pytest.approx(rf["achieved"] / rf["nominal_peak"])
    assert d["launch"] == "stream order"
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"] and "source" in d["clocks"]
    p10, p90, mx = d["us_per_round_p10_p90_max"]
    assert 0 < p10 <= p90 <= mx
    assert d["config"]["workload"] == "tiny"
