"""Randomised GPU parity: many small seeded geometries (ep_size, experts per
rank, top_k, hidden width, payload dtype, scale width, counts, tokens per rank,
masks, id laws, weights on/off, caller-owned or backend expert outputs), each
compared bit for bit with the oracle."""
import random

import pytest

import workloads
from ep_testutil import assert_round_equal, clamp_count, cut_inputs, gpu_round, oracle_round

pytestmark = pytest.mark.gpu

N_CASES = 40


def _case(seed):
    rng = random.Random(1000 + seed)
    ep = rng.choice([1, 2, 3, 4, 5, 8, 13, 16, 31, 33, 64])
    epr = rng.choice([1, 2, 3, 4, 8])
    E = ep * epr
    K = rng.randint(1, min(E, 12)) if rng.random() < 0.8 else rng.randint(1, 32)
    dtype = rng.choice(["bf16", "fp8_e4m3", "fp16", "fp32"])
    align = {"bf16": 8, "fp16": 8, "fp8_e4m3": 16, "fp32": 8}[dtype]
    hidden = align * rng.randint(1, 96)
    scales = rng.random() < 0.5
    scale_cols = None
    if scales and (hidden % 128 != 0 or rng.random() < 0.5):
        scale_cols = rng.randint(1, 20)
    cap = rng.randint(0, 12)
    rt = None if rng.random() < 0.5 else rng.randint(0, cap)
    T = cap if rt is None else rt
    counts = ("uniform", 0, T) if rng.random() < 0.7 else ("full",)
    ids = "uniform_distinct" if K <= E else "uniform_dups"
    ids = rng.choice([ids, "uniform_dups", "with_invalid"]) if K <= E else ids
    dropped = None
    if rng.random() < 0.4:
        dropped = tuple(r for r in range(ep) if rng.random() < 0.3)
    cdt = rng.choice(["bf16", "bf16", "fp16", "fp32"])
    return workloads.EpWorkload(
        name=f"fuzz{seed}", ep_size=ep, num_experts=E, top_k=K, hidden=hidden, dtype=dtype,
        combine_dtype=cdt,
        capacity=cap, runtime_max=rt, counts=counts, ids=ids, weights=rng.random() < 0.7,
        scales=scales, scale_cols_override=scale_cols, dropped_ranks=dropped, seed=seed), \
        rng.random() < 0.3


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_geometry(cuda_device, seed):
    wl, caller_eo = _case(seed)
    inp = workloads.make_inputs(wl)
    got = gpu_round(inp, cuda_device, caller_eo=caller_eo)
    disp, out = oracle_round(inp)
    assert_round_equal(inp, got, disp, out)


@pytest.mark.parametrize("seed", range(20))
def test_random_geometry_device_counts(cuda_device, seed):
    """The same geometries with device-side token counts drawn in [-2, rows + 2]:
    the round must equal the oracle's round of the inputs cut to the clamped
    counts."""
    wl, caller_eo = _case(seed)
    inp = workloads.make_inputs(wl)
    rng = random.Random(5000 + seed)
    dev = [rng.randint(-2, n + 2) for n in inp.num_tokens]
    got = gpu_round(inp, cuda_device, caller_eo=caller_eo, dev_counts=dev)
    cut = cut_inputs(inp, [clamp_count(c, n) for c, n in zip(dev, inp.num_tokens)])
    disp, out = oracle_round(cut)
    assert_round_equal(cut, got, disp, out)
