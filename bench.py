#!/usr/bin/env python
"""Throughput of rank-major MoE EP dispatch + combine on one GB300.

A step (a "round") is one ep_dispatch then one ep_combine of a whole EP group
of virtual ranks, on one stream, with the inputs resident in HBM. The
combine reads the backend combine-input buffers, filled once (untimed) with
stand-in expert outputs. L2 is flushed before each timed step, outside the
step's CUDA events (a 256 MB buffer written, then read back so the flush
leaves no dirty lines behind); the prefill workload's traffic is also far
larger than L2.

Timing: the round is captured once as one CUDA graph of the two API calls and
replayed (as a static-shape caller runs it), with CUDA events around each
replay; a second pass replays the calls as two graphs with an event between
them for the per-kernel times of the roofline.

Metric: algorithmic bytes per round / round time, in GB/s, and that as a
fraction of the measured HBM copy bandwidth. Algorithmic bytes per round,
with N tokens, P routed (token, rank) pairs, payload row H*b bytes, G scale
columns, K ids, w = 1 when weights are sent:
  dispatch reads  N*(H*b + 4G + 4K + 4K*w)
  dispatch writes P*(H*b + 4G + 4K*w) + ep*ep*T*4K   (routed rows + whole id plane)
  combine         P*2H (reads) + 8N (routing state) + N*2H (writes)

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                    [--pdl] [--partitions NPART]

--partitions NPART runs each round as NPART partitions of the group (ranks in
NPART contiguous blocks, each with its own workspace and communicator,
connected with one another): NPART dispatch launches, then NPART combine
launches per round, one after another, or side by side on a stream each with
--partition-streams.

Under torchrun (N > 1) every rank runs an independent replica of the same
workload on its own GPU (the EP group is simulated inside one GPU, so there
is nothing to exchange between GPUs); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

class NvmlReader:
    """Read-only clock, power and clock-event-reason queries on one GPU through
    the driver's NVML library (libnvidia-ml.so.1), called with ctypes."""

    # nvmlClocksEventReasons bits (public NVML API)
    REASON_BITS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
                   ("hw_thermal_slowdown", 0x40), ("hw_power_brake_slowdown", 0x80))
    CLOCK_SM = 1

    def __init__(self, uuid: str):
        import ctypes
        self._c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.lib, self.dev = lib, ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
            lib.nvmlShutdown()
            raise RuntimeError(f"no NVML device {uuid}")
        self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _uint(self, fn, *args):
        v = self._c.c_uint(0)
        if fn(self.dev, *args, self._c.byref(v)) != 0:
            raise RuntimeError(fn.__name__)
        return v.value

    def sm_mhz(self):
        return float(self._uint(self.lib.nvmlDeviceGetClockInfo, self.CLOCK_SM))

    def sm_max_mhz(self):
        return float(self._uint(self.lib.nvmlDeviceGetMaxClockInfo, self.CLOCK_SM))

    def power_w(self):
        return self._uint(self.lib.nvmlDeviceGetPowerUsage) / 1000.0

    def reason_bits(self):
        v = self._c.c_ulonglong(0)
        if self._reasons_fn(self.dev, self._c.byref(v)) != 0:
            raise RuntimeError("clock event reasons")
        return v.value

    def close(self):
        self.lib.nvmlShutdown()


def clock_poller(reader, period_s: float, out, stop) -> int:
    """Writes "ready" once, then one line "sm_mhz,sm_max_mhz,power_w,reason_bits"
    every period_s until stop() is true. Runs in its own process (below), so
    it never competes with the timed launches for the interpreter lock."""
    smax = reader.sm_max_mhz()
    out.write("ready\n")
    out.flush()
    while not stop():
        out.write(f"{reader.sm_mhz()},{smax},{reader.power_w()},{reader.reason_bits()}\n")
        time.sleep(period_s)
    out.flush()
    reader.close()
    return 0


if __name__ == "__main__" and sys.argv[1:2] == ["--clock-poller"]:
    import signal
    _stop = []
    signal.signal(signal.SIGTERM, lambda *_: _stop.append(1))
    try:
        _reader = NvmlReader(sys.argv[2])
    except Exception as e:  # no NVML here: the parent falls back to nvidia-smi
        print(f"unavailable: {e}", flush=True)
        sys.exit(0)
    sys.exit(clock_poller(_reader, float(sys.argv[3]), sys.stdout, lambda: bool(_stop)))


import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "dispatch+combine µs/round and routed-payload GB/s as % of GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth (7.9 TB/s), for context beside the measured peak
L2_FLUSH_BYTES = 256 << 20
# Sources whose code decides what the profiled kernels do: the kernels and
# their argument blocks.
KERNEL_SRCS = [os.path.join(ROOT, "combine_topk_ids_dest_gb300", "csrc", f)
               for f in ("ep_kernels.cu", "ep_internal.h")]


# ---------------------------------------------------------------------------
# bookkeeping
# ---------------------------------------------------------------------------
def routed_pairs(inp) -> int:
    """P: number of (token, destination rank) pairs of the workload."""
    wl = inp.wl
    ep, E, epr = wl.ep_size, wl.num_experts, wl.num_experts // wl.ep_size
    active = torch.tensor([(inp.active_rank_mask >> d) & 1 for d in range(ep)], dtype=torch.bool)
    P = 0
    for ids in inp.topk_ids:
        if ids.shape[0] == 0:
            continue
        ids = ids.to(torch.int64)
        ok = (ids >= 0) & (ids < E)
        owner = torch.where(ok, ids // epr, torch.zeros_like(ids))
        hit = torch.zeros(ids.shape[0], ep, dtype=torch.bool)
        hit.scatter_(1, owner, ok)
        if wl.enable_rank_mask:
            hit &= active
        P += int(hit.sum())
    return P


def round_bytes(inp) -> dict:
    wl = inp.wl
    N, P = inp.total_tokens, routed_pairs(inp)
    ep, K, H, T = wl.ep_size, wl.top_k, wl.hidden, wl.tokens_per_rank
    hb = H * wl.elem_bytes
    G = wl.scale_cols if inp.scale is not None else 0
    w = 1 if inp.topk_weights is not None else 0
    d_read = N * (hb + 4 * G + 4 * K + 4 * K * w)
    d_write = P * (hb + 4 * G + 4 * K * w) + ep * ep * T * 4 * K
    c_read = P * 2 * H + 8 * N
    c_write = N * 2 * H
    return dict(N=N, P=P, dispatch=d_read + d_write, combine=c_read + c_write,
                total=d_read + d_write + c_read + c_write, payload=P * (hb + 4 * G) + N * hb,
                h2d=N * (hb + 4 * G + 4 * K + 4 * K * w), d2h=N * 2 * H)


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no measured peak available)"


def _strip_comments(text: str) -> str:
    """C/C++ source without comments and with whitespace runs collapsed, so
    that editing a comment does not change the fingerprint of the code."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # string or character literal, copied whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_code_fingerprint() -> str:
    """sha256[:16] of the kernel sources' code (comments and layout ignored)."""
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        h.update(_strip_comments(open(path, encoding="utf-8").read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, with_source: bool = False):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, when
    that summary was taken on the current kernel code; else None. With
    `with_source`, (bytes, how they were obtained) or (None, None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    src = kernel_code_fingerprint()
    pat = re.compile(r"^(\S+)\s+workload=(\S+)\s+dram_bytes_per_launch=(\d+)\s+code_sha256=(\S+)"
                     r"(?:\s+scaled_from=T(\d+))?")
    found = (None, None)
    if os.path.exists(path):
        for line in open(path):
            m = pat.match(line.strip())
            if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == src:
                how = ("ncu capture of a full launch" if m.group(5) is None else
                       f"ncu capture at {m.group(5)} tokens per rank, scaled to a full launch by the "
                       "algorithmic bytes (profiles/dram_traffic.txt)")
                found = (int(m.group(3)), how)
                break
    return found if with_source else found[0]


class L2Flush:
    """Evicts L2 between timed steps: writes a 256 MB buffer (twice L2), and in
    "write+read" mode then reads it back, so that L2 holds clean lines and the
    next timed kernel does not pay for writing back the flush's dirty data."""

    def __init__(self, device, mode="write+read"):
        self.mode = mode
        self.buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.sink = torch.empty((), dtype=torch.int64, device=device)

    def __call__(self, i):
        self.buf.fill_(i & 0xFF)
        if self.mode == "write+read":
            torch.sum(self.buf.view(torch.int64), dim=0, out=self.sink)


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


class ClockSampler:
    """Samples SM clock, power and clock-event reasons while the timed region
    runs: every 2 ms through NVML in a separate process (this file run with
    --clock-poller), or, where NVML cannot be loaded, every 50 ms with
    nvidia-smi. Either sampler is started, and its first line awaited, before
    the region begins."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    NVML_PERIOD_S = 0.002
    SMI_PERIOD_MS = 50

    def __init__(self, device):
        self.proc, self.path, self.source = None, None, None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.sel = str(device.index or 0)

    def _start(self, cmd):
        if self.path:
            os.unlink(self.path)
        fd, self.path = tempfile.mkstemp(suffix=".clk")
        with os.fdopen(fd, "w") as fh:
            self.proc = subprocess.Popen(cmd, stdout=fh, stderr=subprocess.DEVNULL, stdin=subprocess.DEVNULL)
        t0 = time.time()
        while time.time() - t0 < 20 and self.proc.poll() is None and os.path.getsize(self.path) == 0:
            time.sleep(0.005)
        with open(self.path) as f:
            first = f.readline()
        return first

    def __enter__(self):
        try:
            if self.sel.startswith("GPU-"):
                first = self._start([sys.executable, os.path.abspath(__file__), "--clock-poller", self.sel,
                                     str(self.NVML_PERIOD_S)])
                if first.startswith("ready"):
                    self.source = "nvml"
                    return self
                self._stop()
            self._start(["nvidia-smi", "-i", self.sel, f"--query-gpu={self.FIELDS}",
                         "--format=csv,noheader,nounits", "-lms", str(self.SMI_PERIOD_MS)])
            self.source = "nvidia-smi"
        except Exception:
            self._stop()
        return self

    def _stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
                self.proc.wait()
            self.proc = None

    def __exit__(self, *exc):
        self._stop()

    @staticmethod
    def parse_nvml(lines):
        out = []
        for line in lines:
            f = line.strip().split(",")
            if len(f) != 4:
                continue
            try:
                sm, smax, pw, bits = float(f[0]), float(f[1]), float(f[2]), int(f[3])
            except ValueError:
                continue
            out.append((sm, smax, pw, {n for n, b in NvmlReader.REASON_BITS if bits & b}))
        return out

    @classmethod
    def parse_smi(cls, lines):
        out = []
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                vals = float(f[1]), float(f[2]), float(f[3])
            except ValueError:
                continue
            out.append(vals + ({n for n, v in zip(cls.NAMES, f[5:9]) if v.lower() == "active"},))
        return out

    @staticmethod
    def summarise(samples, source, period_ms):
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "source": source}
        sm = [x[0] for x in samples]
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm),
                "sm_max_mhz": max(x[1] for x in samples),
                "reasons": sorted(set().union(*(x[3] for x in samples))), "samples": len(samples),
                "power_w_max": max(x[2] for x in samples), "source": source, "period_ms": period_ms}

    def summary(self):
        if self.source is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source (NVML, nvidia-smi)"]}
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        if self.source == "nvml":
            return self.summarise(self.parse_nvml(lines), "nvml", 1e3 * self.NVML_PERIOD_S)
        return self.summarise(self.parse_smi(lines), "nvidia-smi", self.SMI_PERIOD_MS)


def _quantile(xs, q):
    """q-quantile of xs by linear interpolation between order statistics."""
    ys = sorted(xs)
    pos = q * (len(ys) - 1)
    lo = int(pos)
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (pos - lo)


def reduce_max(values, device=None):
    """Element-wise max over all ranks of the default process group (identity
    without one): the slowest replica sets the time of the whole job."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_gbs(bytes_per_round: int, rounds: int, world: int, max_total_ms: float) -> float:
    """GB/s of the whole job: every replica's bytes over the slowest replica's time."""
    return world * bytes_per_round * rounds / (max_total_ms / 1e3) / 1e9


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------
def _sample_inputs(inp, m: int, t0: int = 0):
    """Tokens [t0, t0+m) of every source rank (as many as it has), as a
    workload with tokens_per_rank m: the oracle's bounded sample of the full
    workload. Under the rank-major row rule such a slice of tokens is a
    problem of its own (its row s*m+j stands for full row s*T+t0+j)."""
    wl = inp.wl
    counts = [max(0, min(m, n - t0)) for n in inp.num_tokens]
    # copies, not views: a view would carry (and pickle) its whole storage
    sub = lambda lst: None if lst is None else [x[t0:t0 + c].clone() for x, c in zip(lst, counts)]
    swl = wl.replace(capacity=m, runtime_max=None, counts=("fixed",) + tuple(counts))
    return workloads.EpInputs(wl=swl, num_tokens=counts, hidden=sub(inp.hidden), scale=sub(inp.scale),
                              topk_ids=sub(inp.topk_ids), topk_weights=sub(inp.topk_weights),
                              active_rank_mask=inp.active_rank_mask)


def _oracle_chunk_timed(s):
    """Runs in a worker process: one chunk's oracle round, timed by the wall
    clock the parent shares; returns (start, end, algorithmic bytes)."""
    import numpy as np
    torch.set_num_threads(1)  # one core per process: torch's own thread pool would oversubscribe them
    wl = s.wl
    rows = torch.arange(wl.ep_size * wl.tokens_per_rank)
    eo = [workloads.expert_output_rows(1, d, rows, wl.hidden).view(torch.int16).numpy().view(np.uint16)
          for d in range(wl.ep_size)]
    t0 = time.time()
    _oracle_round(s, eo)
    return t0, time.time(), round_bytes(s)["total"]


def oracle_parallel(inp, seconds: float, m_single: int):
    """The unchanged single-threaded oracle on every host core at once: one
    spawn-started process per core, each on its own chunk of tokens (tokens
    [w*m, (w+1)*m) of every rank, m chosen so a chunk takes about `seconds`,
    at most the workload split evenly). GB/s = all chunks' bytes over the
    wall time from the first chunk's start to the last one's end."""
    import concurrent.futures as cf
    import multiprocessing as mp
    n = len(os.sched_getaffinity(0))
    T = inp.wl.tokens_per_rank
    m = max(1, min(m_single, -(-T // n)))
    chunks = [_sample_inputs(inp, m, w * m) for w in range(n) if w * m < max(inp.num_tokens)]
    with cf.ProcessPoolExecutor(max_workers=len(chunks), mp_context=mp.get_context("spawn")) as ex:
        list(ex.map(_oracle_chunk_timed, [_sample_inputs(inp, 1)] * len(chunks)))  # start and warm every worker
        res = list(ex.map(_oracle_chunk_timed, chunks))
    wall = max(r[1] for r in res) - min(r[0] for r in res)
    nbytes = sum(r[2] for r in res)
    desc = (f"{len(chunks)} processes at once, each the single-threaded C oracle on {m} tokens of every "
            f"source rank (tokens [w*{m}, (w+1)*{m}) in process w; {sum(sum(c.num_tokens) for c in chunks)} of "
            f"{inp.total_tokens} tokens)")
    return nbytes / wall / 1e9, len(chunks), desc, wall


def _oracle_round(s, eo):
    import oracle
    wl = s.wl
    oracle.dispatch(wl.ep_size, wl.num_experts, wl.top_k, wl.tokens_per_rank, s.num_tokens, s.hidden,
                    s.topk_ids, scale=s.scale, topk_weights=s.topk_weights,
                    mask_enabled=wl.enable_rank_mask, active_rank_mask=s.active_rank_mask)
    oracle.combine(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.tokens_per_rank, s.num_tokens,
                   s.topk_ids, eo, mask_enabled=wl.enable_rank_mask, active_rank_mask=s.active_rank_mask)


def oracle_sample(inp, seconds: float):
    """Picks the number of tokens per rank m whose oracle round takes about
    `seconds`; returns (sample inputs, expert outputs, bytes, description)."""
    import numpy as np
    wl = inp.wl
    T = wl.tokens_per_rank

    def prep(m):
        s = _sample_inputs(inp, m)
        rows = torch.arange(wl.ep_size * m)
        eo = [workloads.expert_output_rows(1, d, rows, wl.hidden).view(torch.int16).numpy().view(np.uint16)
              for d in range(wl.ep_size)]
        return s, eo

    m = 1
    while True:
        s, eo = prep(m)
        t0 = time.perf_counter()
        _oracle_round(s, eo)
        dt = time.perf_counter() - t0
        if dt >= seconds / 4 or m >= T:
            break
        m = min(T, max(m + 1, int(m * min(8.0, (seconds / 4) / max(dt, 1e-4)))))
    m = min(T, max(1, int(round(m * seconds / max(dt, 1e-4)))))
    s, eo = prep(m)
    b = round_bytes(s)
    desc = (f"first {m} of {T} tokens per source rank ({s.total_tokens} of {inp.total_tokens} tokens), "
            f"all {wl.ep_size} ranks, same ids/masks/payload; single-threaded C oracle")
    return s, eo, b, desc, m


def run_reference(args, rank, world):
    """The oracle timed as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    wl = workloads.by_name(args.workload)
    inp = workloads.make_inputs(wl)
    full = round_bytes(inp)
    # the whole arm takes about --reference-seconds for any step count (the
    # oracle's cost grows linearly with the sample, so GB/s does not depend on it)
    per_step = max(0.05, args.reference_seconds / max(1, args.steps + args.warmup))
    s, eo, b, desc, _ = oracle_sample(inp, per_step)
    for _ in range(args.warmup):
        _oracle_round(s, eo)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_round(s, eo)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    gbs = b["total"] * len(times) / tot / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32",
        "data": "synthetic", "config": workload_config(wl, full, args.l2_flush),
        "us_per_round_extrapolated": 1e6 * full["total"] / (gbs * 1e9),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc,
                         "host_cores_available": len(os.sched_getaffinity(0))},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(wl, b, l2_flush):
    """The workload, as both arms print it (same object for the same arguments)."""
    l2 = {"write": "L2 flushed before each timed step, outside its events: 256 MB written",
          "write+read": "L2 flushed before each timed step, outside its events: 256 MB written then "
                        "read back (clean, cold L2)"}[l2_flush]
    if b["total"] > (128 << 20):
        l2 += "; per-round traffic larger than L2"
    return {"workload": wl.name, "ep_size": wl.ep_size, "num_experts": wl.num_experts,
            "top_k": wl.top_k, "hidden": wl.hidden,
            "payload": wl.dtype + (f" + fp32 scales [n,{wl.scale_cols}]" if wl.scales else ""),
            "max_tokens_per_rank": wl.capacity, "tokens_per_rank": wl.tokens_per_rank,
            "ids": wl.ids, "rank_mask_drops": list(wl.dropped_ranks) if wl.dropped_ranks else None,
            "tokens": b["N"], "routed_pairs": b["P"], "bytes_per_round": b["total"], "l2": l2,
            "combine_input": "backend buffer, filled once with stand-in expert outputs (untimed)"}


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------
def run_ours(args, rank, world):
    import torch.distributed as dist
    from combine_topk_ids_dest_gb300 import EpComm, connect_partitions

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = workloads.by_name(args.workload)
    inp = workloads.make_inputs(wl)
    b = round_bytes(inp)
    dtype = wl.torch_dtype
    # one communicator, or (--partitions G) G partitions of the group, each with its own workspace
    G = args.partitions
    comms = [EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, dtype=dtype,
                    enable_rank_mask=wl.enable_rank_mask, device=dev, pdl=args.pdl, num_partitions=G, partition=g)
             for g in range(G)]
    if G > 1:
        connect_partitions(comms)
    mask = inp.active_rank_mask if wl.enable_rank_mask else None
    hid = [x.to(dev) for x in inp.hidden]
    ids = [x.to(dev) for x in inp.topk_ids]
    wts = None if inp.topk_weights is None else [x.to(dev) for x in inp.topk_weights]
    scl = None if inp.scale is None else [x.to(dev) for x in inp.scale]
    out = [torch.empty(n, wl.hidden, dtype=torch.bfloat16, device=dev) for n in inp.num_tokens]
    flush = L2Flush(dev, args.l2_flush)

    # with --partition-streams each partition's launches go to a stream of its
    # own, forked from and joined back into the current stream (as a graph
    # capture sees them), so partitions run side by side as on separate GPUs
    side = [torch.cuda.Stream(dev) for _ in comms] if args.partition_streams and G > 1 else None

    def each_partition(fn):
        if side is None:
            for c in comms:
                fn(c)
            return
        cur = torch.cuda.current_stream(dev)
        fork = torch.cuda.Event()
        fork.record(cur)
        joins = []
        for c, st in zip(comms, side):
            st.wait_event(fork)
            with torch.cuda.stream(st):
                fn(c)
                e = torch.cuda.Event()
                e.record(st)
                joins.append(e)
        for e in joins:
            cur.wait_event(e)

    def dispatch():
        each_partition(lambda c: c.dispatch(_part(hid, c), _part(ids, c), _part(wts, c),
                                            hidden_states_scale=_part(scl, c),
                                            runtime_max_tokens_per_rank=wl.runtime_max, active_rank_mask=mask))

    def combine():
        each_partition(lambda c: c.combine(output=_part(out, c), active_rank_mask=mask))

    # one untimed round to fill the combine-input buffers with expert outputs
    dispatch()
    rows = torch.arange(wl.ep_size * wl.tokens_per_rank, device=dev)
    for c in comms:
        for j, buf in enumerate(c.get_combine_input_buffer()):
            buf.copy_(workloads.expert_output_rows(1, c.first_rank + j, rows, wl.hidden, device=dev))
    del rows
    combine()
    launches_per_round = 2 * G if wl.ep_size * wl.tokens_per_rank > 0 else 0

    # The same API calls captured once in CUDA graphs (static shapes):
    # replaying them runs exactly the dispatch and combine kernels, without
    # the Python binding's per-call overhead in the measured device time. The
    # round is one graph (dispatch then combine, as a static-shape caller
    # replays it); the per-kernel times come from a second pass that replays
    # the two calls as separate graphs with an event between them.
    g_round, g_disp, g_comb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_round):
        dispatch()
        combine()
    with torch.cuda.graph(g_disp):
        dispatch()
    with torch.cuda.graph(g_comb):
        combine()

    def timed_rounds(run_dispatch, run_combine, steps, warmup, clocks=None):
        for i in range(warmup):
            flush(i)
            run_dispatch()
            if run_combine is not None:
                run_combine()
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        with (clocks if clocks is not None else _Null()):
            torch.cuda.synchronize(dev)
            for i in range(steps):
                flush(i + 1)
                ev[i][0].record()
                run_dispatch()
                ev[i][1].record()
                if run_combine is not None:
                    run_combine()
                    ev[i][2].record()
            torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        if run_combine is None:  # run_dispatch ran the whole round
            return None, None, [e[0].elapsed_time(e[1]) for e in ev]
        return ([e[0].elapsed_time(e[1]) for e in ev], [e[1].elapsed_time(e[2]) for e in ev],
                [e[0].elapsed_time(e[2]) for e in ev])

    clocks = ClockSampler(dev)
    _, _, t_round = timed_rounds(g_round.replay, None, args.steps, args.warmup, clocks)
    total_ms = sum(t_round)
    t_disp, t_comb, t_split = timed_rounds(g_disp.replay, g_comb.replay, args.steps, args.warmup)
    ed, ec, er = timed_rounds(dispatch, combine, args.steps, args.warmup)
    eager_ms = sum(er)

    # end to end through the public API from pinned host memory
    e2e_steps = max(4, min(args.steps, 20))
    e2e_ms, h2d_bytes, d2h_bytes = run_e2e(comms, inp, wl, dev, mask, e2e_steps)
    local_cpus = gpu_local_cpus(dev)

    total_ms, e2e_ms, eager_ms = reduce_max([total_ms, e2e_ms, eager_ms], device=dev)
    for c in comms:
        c.destroy()
    if rank != 0:
        return

    peak, peak_src = hbm_peak()
    ms = total_ms / args.steps
    gbs = whole_job_gbs(b["total"], args.steps, world, total_ms)
    disp_ms, comb_ms = statistics.mean(t_disp), statistics.mean(t_comb)
    kernels = {
        "dispatch_kernel": {"bytes": b["dispatch"], "ms": disp_ms},
        "combine_kernel": {"bytes": b["combine"], "ms": comb_ms},
    }
    top = max(kernels, key=lambda k: kernels[k]["ms"])
    per = {k: {"achieved": v["bytes"] / (v["ms"] / 1e3) / 1e9, "ms": v["ms"], "bytes": v["bytes"],
               "frac": v["bytes"] / (v["ms"] / 1e3) / 1e9 / peak, "share": v["ms"] / (disp_ms + comb_ms),
               "traffic": recorded_traffic(k, wl.name)} for k, v in kernels.items()}
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32", "data": "synthetic",
        "config": workload_config(wl, b, args.l2_flush),
        "us_per_round": 1e3 * ms, "us_per_round_median": 1e3 * statistics.median(t_round),
        "us_per_round_p10_p90_max": [1e3 * _quantile(t_round, 0.1), 1e3 * _quantile(t_round, 0.9),
                                     1e3 * max(t_round)],
        "pct_hbm_peak": 100.0 * b["total"] / (ms / 1e3) / 1e9 / peak,
        "pct_nominal_hbm": 100.0 * b["total"] / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS,
        "payload_gbs": b["payload"] / (ms / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "kernel": top, "achieved": per[top]["achieved"], "peak": peak,
                     "unit": "GB/s", "frac": per[top]["frac"], "traffic": per[top]["traffic"],
                     "traffic_source": recorded_traffic(top, wl.name, with_source=True)[1],
                     "peak_source": peak_src,
                     "peak_kind": "a measured copy bandwidth (equal bytes read and written); a kernel whose "
                                  "traffic is mostly reads or mostly writes can stream above it",
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": per[top]["achieved"] / NOMINAL_HBM_GBS,
                     "kernels": per},
        "e2e": {"value": whole_job_gbs(b["total"], 1, world, e2e_ms), "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "steps": e2e_steps,
                "path": "pinned host inputs (one packed buffer) -> one H2D copy -> EpComm.dispatch/combine "
                        "(C ABI) -> one D2H copy of the packed outputs; H2D, kernels and D2H of consecutive "
                        "steps overlap on three streams",
                "pinned_on": f"{len(local_cpus)} GPU-local CPUs" if local_cpus else "default placement"},
        "eager": {"value": whole_job_gbs(b["total"], args.steps, world, eager_ms), "unit": "GB/s",
                  "ms_per_step": eager_ms / args.steps,
                  "dispatch_ms": statistics.mean(ed), "combine_ms": statistics.mean(ec),
                  "path": "EpComm.dispatch/combine called from Python each round"},
        "timing": "round: CUDA-graph replay of the captured EpComm.dispatch + EpComm.combine calls (one "
                  "graph), events on the launching stream around it; kernels: the two calls replayed as "
                  "separate graphs in a second pass, events around each",
        "us_per_round_two_graphs": 1e3 * statistics.mean(t_split),
        "gpu_launches": launches_per_round * args.steps,
        "launch": "programmatic dependent launch (EP_LAUNCH_PDL)" if args.pdl else "stream order",
        "partitions": G, "partition_streams": side is not None,
        "clocks": clocks.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        s, eo, sb, desc, m = oracle_sample(inp, args.cpu_seconds)
        t0 = time.perf_counter()
        _oracle_round(s, eo)
        dt = time.perf_counter() - t0
        cpu_gbs = sb["total"] / dt / 1e9
        line["cpu_baseline"] = {"value": cpu_gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": desc, "seconds": dt,
                                "us_per_round_extrapolated": 1e6 * b["total"] / (cpu_gbs * 1e9),
                                "host_cores_available": len(os.sched_getaffinity(0))}
        if len(os.sched_getaffinity(0)) > 1:
            pgbs, cores, pdesc, wall = oracle_parallel(inp, args.cpu_seconds, m)
            line["cpu_baseline_all_cores"] = {
                "value": pgbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": pdesc,
                "seconds": wall, "us_per_round_extrapolated": 1e6 * b["total"] / (pgbs * 1e9)}
    print(json.dumps(line), flush=True)


def _packed(tensors, device=None, pin=False):
    """One contiguous buffer holding `tensors` back to back (32-byte aligned
    offsets, so the library's 32-byte access paths apply to every view) and
    per-tensor views into it."""
    import math
    offs, off = [], 0
    for t in tensors:
        offs.append(off)
        off += -(-t.numel() * t.element_size() // 32) * 32
    buf = torch.empty(max(off, 32), dtype=torch.uint8, device=device, pin_memory=pin)
    views = []
    for t, o in zip(tensors, offs):
        nb = t.numel() * t.element_size()
        views.append(buf[o:o + nb].view(t.dtype).view(t.shape))
    return buf, views


def gpu_local_cpus(dev):
    """CPUs the GPU's PCI device reports as local (sysfs), within this
    process's allowed set; None when unknown."""
    try:
        p = torch.cuda.get_device_properties(dev)
        path = "/sys/bus/pci/devices/%04x:%02x:%02x.0/local_cpulist" % (
            p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        cpus = set()
        for part in open(path).read().strip().split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        cpus &= os.sched_getaffinity(0)
        return cpus or None
    except Exception:
        return None


def _part(lst, c):
    """The entries of a per-rank list that communicator `c` hosts."""
    return None if lst is None else lst[c.first_rank:c.first_rank + c.num_ranks]


def run_e2e(comms, inp, wl, dev, mask, steps):
    """Rounds through the public API with every step's inputs copied in from
    pinned host memory and its outputs copied back, pipelined over three
    streams with two sets of device buffers: step i's host-to-device copy and
    step i-1's device-to-host copy overlap step i's kernels. Returns the
    mean wall time per step on the device (ms), after `steps` steps, and the
    bytes copied in each direction per step (the packed buffers' sizes)."""
    kinds = [k for k in ("hidden", "topk_ids", "topk_weights", "scale") if getattr(inp, k) is not None]
    # pinned buffers are placed on the memory node of the allocating CPU:
    # allocate them from the GPU's local CPUs
    local = gpu_local_cpus(dev)
    prev = os.sched_getaffinity(0)
    if local:
        os.sched_setaffinity(0, local)
    # every input of a step in one pinned buffer (one host-to-device copy per step)
    flat = [t for k in kinds for t in getattr(inp, k)]
    split = lambda views: {k: views[i * wl.ep_size:(i + 1) * wl.ep_size] for i, k in enumerate(kinds)}
    host_buf, host_views = _packed(flat, pin=True)
    for v, t in zip(host_views, flat):
        v.copy_(t)
    devsets = []
    for _ in range(2):
        buf, views = _packed(flat, device=dev)
        devsets.append((buf, split(views)))
    outs = [torch.empty(n, wl.hidden, dtype=torch.bfloat16) for n in inp.num_tokens]
    dev_out = [_packed(outs, device=dev) for _ in range(2)]
    host_out = [_packed(outs, pin=True) for _ in range(2)]
    for _, views in host_out:  # touch the output pages from the local CPUs too
        for v in views:
            v.zero_()
    if local:
        os.sched_setaffinity(0, prev)
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    for e in in_free + out_free:
        e.record(comp)

    def step(i):
        k = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(in_free[k])
            devsets[k][0].copy_(host_buf, non_blocking=True)
            in_ready[k].record(s_in)
        comp.wait_event(in_ready[k])
        comp.wait_event(out_free[k])
        v = devsets[k][1]
        for c in comms:
            c.dispatch(_part(v["hidden"], c), _part(v["topk_ids"], c), _part(v.get("topk_weights"), c),
                       hidden_states_scale=_part(v.get("scale"), c), runtime_max_tokens_per_rank=wl.runtime_max,
                       active_rank_mask=mask)
        in_free[k].record(comp)
        for c in comms:
            c.combine(output=_part(dev_out[k][1], c), active_rank_mask=mask)
        out_ready[k].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(out_ready[k])
            host_out[k][0].copy_(dev_out[k][0], non_blocking=True)
            out_free[k].record(s_out)

    for i in range(3):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    for i in range(steps):
        step(i)
    comp.wait_stream(s_in)
    comp.wait_stream(s_out)
    e1.record(comp)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / steps, host_buf.numel(), host_out[0][0].numel()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="dsv3_prefill",
                    choices=sorted(workloads.WORKLOADS) + sorted(workloads.GEOMETRIES))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample size, in seconds")
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="total oracle time of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2-flush", default="write+read", choices=["write", "write+read"],
                    help="how L2 is evicted between timed steps")
    ap.add_argument("--pdl", action=argparse.BooleanOptionalAction, default=False,
                    help="launch the kernels with programmatic dependent launch")
    ap.add_argument("--partitions", type=int, default=1,
                    help="run the group as this many partitions, each with its own workspace")
    ap.add_argument("--partition-streams", action="store_true",
                    help="launch each partition on a stream of its own (side by side)")
    ap.add_argument("--tokens-per-rank", type=int, default=None,
                    help="shrink the workload to this many tokens per rank (profiling runs only)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.tokens_per_rank is not None:
        wl = workloads.by_name(args.workload)
        m = args.tokens_per_rank
        counts = wl.counts
        if counts[0] == "uniform":
            counts = ("uniform", min(counts[1], m), min(counts[2], m))
        elif counts[0] == "fixed":
            counts = ("fixed",) + tuple(min(c, m) for c in counts[1:])
        workloads.WORKLOADS[args.workload] = wl.replace(
            name=f"{wl.name}_T{m}", capacity=m, runtime_max=None if wl.runtime_max is None else m,
            counts=counts)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus != world and rank == 0:
        print(f"bench.py: --gpus {args.gpus} but {world} process(es) were launched; measuring {world} "
              "(start N>1 with torch.distributed.run, one process per GPU)", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
