"""Whole-workload comparison with the oracle, one chunk of tokens at a time,
on a pool of host processes.

The receive layout is rank-major: token t of source rank s lands in row
s*T + t of every rank it is routed to, and that row depends on nothing but
the token's own hidden row, scales, ids and weights (page
"flashinfer.moe_ep.NVLinkOneSidedAlltoAll", class description). Combine's
output for the token likewise depends only on its own routed rows (page
"flashinfer.moe_ep.MoEEpCommunication", combine()). So tokens [t0, t0+Tm)
of every source rank form a small problem of their own, with
tokens_per_rank Tm: its row s*Tm + j stands for full row s*T + t0 + j. The
oracle solves each such chunk; a worker process compares the chunk's
oracle results with the GPU's rows of the same tokens, and together the
chunks cover every token of the workload.

The workers start with the ``spawn`` method (a process forked after CUDA was
initialised would hang) and use the oracle and the seeded input generator
only; the GPU results reach them as numpy arrays.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor
from dataclasses import dataclass
from typing import Iterator, List, Optional

import numpy as np

from ep_testutil import EO_SEED, INV

CHUNK_RECV_BYTES = 64 << 20  # oracle receive-row bytes per chunk


@dataclass
class Geometry:
    ep: int
    E: int
    K: int
    H: int
    T: int  # tokens_per_rank of the full problem
    row_bytes: int
    scale_cols: int
    combine_dtype: str
    mask_enabled: bool
    active_rank_mask: int


def chunk_tokens(g: Geometry, budget: int = CHUNK_RECV_BYTES) -> int:
    """Tokens per rank of one chunk: the oracle's receive rows of a chunk
    (ep ranks x ep*Tm rows x row_bytes) stay within ``budget`` bytes."""
    per = g.ep * g.ep * max(g.row_bytes, 1)
    return max(1, min(max(g.T, 1), budget // per))


def chunk_starts(counts, Tm: int) -> List[int]:
    """First token of every chunk; chunk t0 covers tokens [t0, t0+Tm) of each rank."""
    top = max(counts) if len(counts) else 0
    return list(range(0, top, Tm))


def chunk_counts(counts, t0: int, Tm: int) -> List[int]:
    return [int(min(max(n - t0, 0), Tm)) for n in counts]


def full_rows(g: Geometry, t0: int, Tm: int) -> np.ndarray:
    """int64 [ep*Tm]: the full-problem row that mini row s*Tm + j stands for."""
    s = np.repeat(np.arange(g.ep, dtype=np.int64), Tm)
    j = np.tile(np.arange(Tm, dtype=np.int64), g.ep)
    return s * g.T + t0 + j


def live_rows(g: Geometry, counts_m, Tm: int) -> np.ndarray:
    """bool [ep*Tm]: mini rows that hold a token (j < the rank's chunk count)."""
    return np.concatenate([np.arange(Tm) < m for m in counts_m]) if g.ep else np.zeros(0, bool)


def _bytes2d(a: np.ndarray) -> np.ndarray:
    """uint8 [rows, bytes per row] view of an array's raw bytes."""
    a = np.ascontiguousarray(a)
    if a.size == 0:
        return np.zeros((a.shape[0] if a.ndim else 0, 0), np.uint8)
    return a.view(np.uint8).reshape(a.shape[0], -1)


def chunk_inputs(inp, t0: int, Tm: int) -> dict:
    """The source rows of chunk t0 as numpy arrays (hidden rows as raw bytes)."""
    import torch
    counts_m = chunk_counts(inp.num_tokens, t0, Tm)

    def cut(lst, raw=False):
        if lst is None:
            return None
        out = []
        for x, m in zip(lst, counts_m):
            y = x[t0:t0 + m]
            if raw:
                if y.dtype in (torch.bfloat16, torch.float16):
                    y = y.view(torch.int16)
                elif y.dtype == torch.float8_e4m3fn:
                    y = y.view(torch.uint8)
                out.append(_bytes2d(y.contiguous().numpy()) if m else np.zeros((0, 0), np.uint8))
            else:
                out.append(y.contiguous().numpy())
        return out

    return dict(counts=counts_m, hidden=cut(inp.hidden, raw=True), ids=cut(inp.topk_ids),
                weights=cut(inp.topk_weights), scale=cut(inp.scale))


def make_jobs(g: Geometry, inp, ids_host, Tm: int, rows_of, out_of, has_scale: bool,
              has_weights: bool) -> Iterator[dict]:
    """One job per chunk: the chunk's inputs and the results under test for its
    tokens. ``ids_host[d]`` is rank d's whole receive id plane (numpy);
    ``rows_of(kind, d, rows)`` returns rank d's receive rows ``rows`` (int64
    full-problem rows) of kind "hidden" (raw bytes), "scale" or "weights";
    ``out_of(s, t0, m)`` returns the raw bits of rank s's outputs t0..t0+m-1.
    Only routed rows (id row not all invalid) are fetched."""
    for t0 in chunk_starts(inp.num_tokens, Tm):
        cm = chunk_counts(inp.num_tokens, t0, Tm)
        rows = full_rows(g, t0, Tm)[live_rows(g, cm, Tm)]
        job = dict(g=g, t0=t0, Tm=Tm, inputs=chunk_inputs(inp, t0, Tm), gpu_ids=[], gpu_hidden=[],
                   gpu_scale=[] if has_scale else None, gpu_weights=[] if has_weights else None)
        for d in range(g.ep):
            ids_d = ids_host[d][rows]
            job["gpu_ids"].append(ids_d)
            routed = rows[(ids_d != INV).any(axis=1)]
            job["gpu_hidden"].append(rows_of("hidden", d, routed))
            if has_scale:
                job["gpu_scale"].append(rows_of("scale", d, routed))
            if has_weights:
                job["gpu_weights"].append(rows_of("weights", d, routed))
        job["gpu_out"] = [out_of(s, t0, cm[s]) for s in range(g.ep)]
        yield job


def check_chunk(job: dict) -> Optional[str]:
    """Runs in a worker: the oracle's dispatch and combine of one chunk,
    compared bit for bit with the GPU's rows of the same tokens.

    job: geometry ``g``, ``t0``, ``Tm``, the chunk's inputs (``chunk_inputs``),
    and the GPU's results for the chunk's live tokens, in mini-row order:
    ``gpu_ids[d]`` int32 [live, K] (rank d's id rows), ``gpu_hidden[d]``
    uint8 [routed, row_bytes], ``gpu_scale[d]`` / ``gpu_weights[d]`` fp32
    [routed, *] or None (the rows whose GPU id row is not all invalid), and
    ``gpu_out[s]`` [m_s, H] raw bits. Returns None, or what differs.
    """
    import torch

    import oracle
    import workloads
    torch.set_num_threads(1)
    g: Geometry = job["g"]
    t0, Tm = job["t0"], job["Tm"]
    x = job["inputs"]
    counts_m = x["counts"]
    where = f"tokens [{t0}, {t0 + Tm}) of every rank"
    disp = oracle.dispatch(g.ep, g.E, g.K, Tm, counts_m, x["hidden"], x["ids"], scale=x["scale"],
                           topk_weights=x["weights"], mask_enabled=g.mask_enabled,
                           active_rank_mask=g.active_rank_mask, row_bytes=g.row_bytes,
                           scale_cols=g.scale_cols if x["scale"] is not None else None)
    live = live_rows(g, counts_m, Tm)
    for d in range(g.ep):
        want_ids = disp.recv_ids[d][live]
        if not np.array_equal(job["gpu_ids"][d], want_ids):
            return f"{where}: id rows of rank {d} differ"
        valid = (want_ids != INV).any(axis=1)
        pairs = [("hidden rows", job["gpu_hidden"][d], disp.recv_hidden[d])]
        if disp.recv_scale is not None:
            pairs.append(("scale rows", job["gpu_scale"][d], disp.recv_scale[d]))
        elif job["gpu_scale"] is not None:
            return f"{where}: the GPU returned scale rows the oracle has none of"
        if disp.recv_weights is not None:
            pairs.append(("weight rows", job["gpu_weights"][d], disp.recv_weights[d]))
        elif job["gpu_weights"] is not None:
            return f"{where}: the GPU returned weight rows the oracle has none of"
        for what, got, allrows in pairs:
            want = allrows[live][valid]
            if got.shape != want.shape or not np.array_equal(_bytes2d(got), _bytes2d(want)):
                return f"{where}: {what} of rank {d} differ"
    rows = torch.from_numpy(full_rows(g, t0, Tm))
    eo = []
    for d in range(g.ep):
        e = workloads.expert_output_rows(EO_SEED, d, rows, g.H, dtype=g.combine_dtype).contiguous()
        eo.append(e.view(torch.int32 if e.dtype == torch.float32 else torch.int16).numpy())
    out = oracle.combine_typed(g.ep, g.E, g.K, g.H, Tm, counts_m, x["ids"], eo, g.combine_dtype,
                               mask_enabled=g.mask_enabled, active_rank_mask=g.active_rank_mask)
    for s in range(g.ep):
        got, want = job["gpu_out"][s], out[s]
        if got.shape != want.shape or not np.array_equal(_bytes2d(got), _bytes2d(want)):
            bad = np.argwhere(_bytes2d(got) != _bytes2d(want)) if got.shape == want.shape else None
            first = "" if bad is None or not len(bad) else f" (first at token {t0 + int(bad[0][0])})"
            return f"{where}: combine output of rank {s} differs{first}"
    return None


def pool(workers: Optional[int] = None) -> ProcessPoolExecutor:
    """A spawn-started pool on the host cores this process may use."""
    n = workers or len(os.sched_getaffinity(0))
    return ProcessPoolExecutor(max_workers=max(1, min(n, 16)), mp_context=mp.get_context("spawn"))


def run_jobs(executor: ProcessPoolExecutor, jobs: Iterator[dict], in_flight: int) -> int:
    """Submits ``jobs`` with at most ``in_flight`` pending; raises AssertionError
    with the first difference found. Returns the number of jobs checked."""
    pending, done = [], 0
    for job in jobs:
        pending.append(executor.submit(check_chunk, job))
        while len(pending) >= in_flight:
            msg = pending.pop(0).result()
            done += 1
            if msg:
                raise AssertionError(msg)
    for f in pending:
        msg = f.result()
        done += 1
        if msg:
            raise AssertionError(msg)
    return done
