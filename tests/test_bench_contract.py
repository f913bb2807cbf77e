"""CPU checks of bench.py's host logic: the reference arm's JSON line, the
argument rules, the non-zero ranks' silence under torchrun, and the
algorithmic byte count (its routed-pair count P against the oracle's
receive planes)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True,
                          text=True, env=e, timeout=300)


def test_reference_arm_line():
    r = _bench("--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3",
               "--reference-seconds", "3")
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["steps"] == 3 and line["warmup"] == 3 and line["value"] > 0
    assert line["config"]["workload"] == "tiny"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_nonzero_rank_is_silent():
    r = _bench("--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3",
               env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_below_three_is_rejected():
    r = _bench("--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "2")
    assert r.returncode != 0


@pytest.mark.parametrize("name", ["tiny", "qwen3_mask"])
def test_round_bytes_routed_pairs_match_oracle(name):
    import bench
    from ep_testutil import small
    wl = workloads.WORKLOADS[name]
    wl = wl if name == "tiny" else small(wl)
    inp = workloads.make_inputs(wl)
    b = bench.round_bytes(inp)
    disp = oracle.dispatch(wl.ep_size, wl.num_experts, wl.top_k, wl.tokens_per_rank, inp.num_tokens,
                           inp.hidden, inp.topk_ids, mask_enabled=wl.enable_rank_mask,
                           active_rank_mask=inp.active_rank_mask, payload=False)
    P = sum(int((ids != -1).any(axis=1).sum()) for ids in disp.recv_ids)
    assert b["P"] == P and b["N"] == inp.total_tokens
    ep, K, H, T = wl.ep_size, wl.top_k, wl.hidden, wl.tokens_per_rank
    hb = H * wl.elem_bytes
    G = wl.scale_cols
    w = 1 if inp.topk_weights is not None else 0
    N = inp.total_tokens
    assert b["total"] == (N * (hb + 4 * G + 4 * K + 4 * K * w) + P * (hb + 4 * G + 4 * K * w)
                          + ep * ep * T * 4 * K + P * 2 * H + 8 * N + N * 2 * H)


def test_kernel_fingerprint_ignores_comments_only():
    import bench
    code = 'int f(int x) { return x /* half */ >> 1; }  // shift\nconst char *s = "a//b";\n'
    same = '// a comment\nint f(int x)\n{\n    return x >> 1;\n}\nconst char *s = "a//b";'
    other = 'int f(int x) { return x >> 2; }\nconst char *s = "a//b";'
    assert bench._strip_comments(code) == bench._strip_comments(same)
    assert bench._strip_comments(code) != bench._strip_comments(other)
    assert '"a//b"' in bench._strip_comments(code)  # string literals are kept whole


class _FakeNvml:
    """Stands in for the NVML reader: a clock that drops once, a power-cap reason."""

    def __init__(self):
        self.n, self.closed = 0, False

    def sm_max_mhz(self):
        return 2070.0

    def sm_mhz(self):
        self.n += 1
        return 1900.0 if self.n == 3 else 2070.0

    def power_w(self):
        return 600.0 + self.n

    def reason_bits(self):
        return 0x4 if self.n == 3 else 0  # sw_power_cap

    def close(self):
        self.closed = True


def test_clock_poller_lines_and_summary():
    import io

    import bench
    fake, out = _FakeNvml(), io.StringIO()
    assert bench.clock_poller(fake, 0.0, out, lambda: fake.n >= 5) == 0
    lines = out.getvalue().splitlines()
    assert lines[0] == "ready" and len(lines) == 6 and fake.closed
    s = bench.ClockSampler.summarise(bench.ClockSampler.parse_nvml(lines[1:]), "nvml", 2.0)
    assert s["samples"] == 5 and s["sm_mhz"] == 2070.0 and s["sm_min_mhz"] == 1900.0
    assert s["sm_max_mhz"] == 2070.0 and s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 605.0


def test_clock_smi_lines_parse():
    import bench
    lines = ["0, 2070, 2070, 650.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "0, 1995, 2070, 700.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "garbage"]
    s = bench.ClockSampler.summarise(bench.ClockSampler.parse_smi(lines), "nvidia-smi", 50)
    assert s["samples"] == 2 and s["sm_min_mhz"] == 1995.0 and s["reasons"] == ["sw_power_cap"]


def test_clock_poller_process_reports_unavailable_without_nvml():
    # No GPU has this UUID (and here there is no NVML at all): the poller process
    # says so and exits 0, and the sampler then falls back to nvidia-smi.
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--clock-poller", "GPU-none", "0.002"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("unavailable")


def test_quantile():
    import bench
    assert bench._quantile([3, 1, 2, 5, 4], 0.5) == 3
    assert abs(bench._quantile([1, 2, 3, 4, 5], 0.1) - 1.4) < 1e-12
    assert bench._quantile([7], 0.9) == 7


def test_all_cores_oracle_leg_covers_distinct_token_slices():
    """The all-cores CPU baseline runs the unchanged oracle in one process per
    core, each on its own slice of tokens of every rank; the slices are
    disjoint and their bytes add up to the bytes of the tokens they cover."""
    import bench
    wl = workloads.WORKLOADS["tiny"]
    inp = workloads.make_inputs(wl)
    gbs, procs, desc, wall = bench.oracle_parallel(inp, 0.1, 4)
    assert gbs > 0 and wall > 0 and 1 <= procs <= len(os.sched_getaffinity(0))
    m = max(1, min(4, -(-wl.tokens_per_rank // len(os.sched_getaffinity(0)))))
    chunks = [bench._sample_inputs(inp, m, w * m) for w in range(procs)]
    assert sum(sum(c.num_tokens) for c in chunks) <= inp.total_tokens
    assert f"{procs} processes" in desc
    import torch
    for w, c in enumerate(chunks):  # slice w holds rows [w*m, w*m + count) of the full inputs
        for s in range(wl.ep_size):
            n = c.num_tokens[s]
            assert n == max(0, min(m, inp.num_tokens[s] - w * m))
            assert torch.equal(c.topk_ids[s], inp.topk_ids[s][w * m:w * m + n])
            assert torch.equal(c.hidden[s], inp.hidden[s][w * m:w * m + n])
