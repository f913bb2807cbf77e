"""The chunked whole-workload comparison that the full-size GPU parity test
uses (ep_chunked.py), checked on the CPU against the oracle run on the whole
problem at once.

The rank-major row rule (page "flashinfer.moe_ep.NVLinkOneSidedAlltoAll",
class description: token t of source rank s is row s*T + t of every rank it
reaches) is what lets tokens [t0, t0+Tm) of every rank be solved as a problem
of their own. Here the "results under test" are the whole-problem oracle's:
every chunk must agree with them, the chunks must reach every token, and a
single flipped byte in a routed row, a weight or an output must be reported.
"""
import numpy as np
import pytest
import torch

import ep_chunked
import oracle
import workloads
from ep_testutil import EO_SEED, out_bits

CASES = [
    # uneven counts with an empty rank, a masked rank and T below capacity
    workloads.EpWorkload(name="chunk_bf16_mask", ep_size=6, num_experts=12, top_k=3, hidden=64, dtype="bf16",
                         capacity=20, runtime_max=17, counts=("uniform", 0, 17), empty_ranks=(2,),
                         dropped_ranks=(4,), seed=3),
    # fp8 rows with two scale columns, every slot full
    workloads.EpWorkload(name="chunk_fp8", ep_size=5, num_experts=10, top_k=2, hidden=256, dtype="fp8_e4m3",
                         scales=True, capacity=13, runtime_max=None, counts=("full",), seed=4),
    # fp32 combine, duplicate ids
    workloads.EpWorkload(name="chunk_f32", ep_size=4, num_experts=8, top_k=4, hidden=32, dtype="bf16",
                         capacity=11, runtime_max=None, counts=("fixed", 11, 3, 0, 7), ids="uniform_dups",
                         combine_dtype="fp32", seed=5),
]


@pytest.fixture(scope="module")
def pool():
    ex = ep_chunked.pool(workers=2)
    try:
        yield ex
    finally:
        ex.shutdown(wait=True, cancel_futures=True)


def _whole(wl):
    inp = workloads.make_inputs(wl)
    T, ep, H = wl.tokens_per_rank, wl.ep_size, wl.hidden
    disp = oracle.dispatch(ep, wl.num_experts, wl.top_k, T, inp.num_tokens, inp.hidden, inp.topk_ids,
                           scale=inp.scale, topk_weights=inp.topk_weights, mask_enabled=wl.enable_rank_mask,
                           active_rank_mask=inp.active_rank_mask, row_bytes=H * wl.elem_bytes,
                           scale_cols=wl.scale_cols if wl.scales else None)
    rows = torch.arange(ep * T)
    eo = [out_bits(workloads.expert_output_rows(EO_SEED, d, rows, H, dtype=wl.combine_dtype)) for d in range(ep)]
    out = oracle.combine_typed(ep, wl.num_experts, wl.top_k, H, T, inp.num_tokens, inp.topk_ids, eo,
                               wl.combine_dtype, mask_enabled=wl.enable_rank_mask,
                               active_rank_mask=inp.active_rank_mask)
    g = ep_chunked.Geometry(ep=ep, E=wl.num_experts, K=wl.top_k, H=H, T=T, row_bytes=H * wl.elem_bytes,
                            scale_cols=wl.scale_cols, combine_dtype=wl.combine_dtype,
                            mask_enabled=wl.enable_rank_mask, active_rank_mask=inp.active_rank_mask)
    return inp, disp, out, g


def _jobs(inp, disp, out, g, Tm, flip=None):
    """Jobs whose results under test are the whole-problem oracle's; ``flip`` =
    (kind, rank, full row) changes one byte of that row in the copy handed over."""
    arrays = {"hidden": disp.recv_hidden, "scale": disp.recv_scale, "weights": disp.recv_weights}

    def rows_of(kind, d, rows):
        x = np.array(arrays[kind][d][rows])
        if flip and flip[0] == kind and flip[1] == d and flip[2] in rows:
            x.view(np.uint8).reshape(len(rows), -1)[list(rows).index(flip[2]), 0] ^= 1
        return x

    def out_of(s, t0, m):
        x = np.array(out[s][t0:t0 + m])
        if flip and flip[0] == "out" and flip[1] == s and t0 <= flip[2] < t0 + m:
            x.view(np.uint8).reshape(m, -1)[flip[2] - t0, 0] ^= 1
        return x

    return ep_chunked.make_jobs(g, inp, disp.recv_ids, Tm, rows_of, out_of, disp.recv_scale is not None,
                                disp.recv_weights is not None)


@pytest.mark.parametrize("wl", CASES, ids=[c.name for c in CASES])
@pytest.mark.parametrize("Tm", [1, 4, 64])
def test_chunks_agree_with_the_whole_problem(pool, wl, Tm):
    inp, disp, out, g = _whole(wl)
    Tm = min(Tm, g.T)
    n = ep_chunked.run_jobs(pool, _jobs(inp, disp, out, g, Tm), in_flight=4)
    assert n == len(ep_chunked.chunk_starts(inp.num_tokens, Tm)) == -(-max(inp.num_tokens) // Tm)


def _routed_row(disp, g, d, last=True):
    """A full row of rank d that holds a routed token (the last one, or the first)."""
    rows = np.flatnonzero((disp.recv_ids[d] != -1).any(axis=1))
    assert len(rows)
    return int(rows[-1] if last else rows[0])


@pytest.mark.parametrize("kind", ["hidden", "scale", "weights", "out"])
def test_a_flipped_byte_is_reported(pool, kind):
    wl = CASES[1] if kind == "scale" else CASES[0]
    inp, disp, out, g = _whole(wl)
    if kind == "out":
        s = max(range(g.ep), key=lambda r: inp.num_tokens[r])
        flip = ("out", s, inp.num_tokens[s] - 1)  # the last token of the fullest rank
        what = f"combine output of rank {s}"
    else:
        d = 1
        flip = (kind, d, _routed_row(disp, g, d))
        what = {"hidden": "hidden rows", "scale": "scale rows", "weights": "weight rows"}[kind] + f" of rank {d}"
    with pytest.raises(AssertionError, match=what):
        ep_chunked.run_jobs(pool, _jobs(inp, disp, out, g, 4, flip=flip), in_flight=4)


def test_chunk_size_stays_within_budget():
    g = ep_chunked.Geometry(ep=32, E=256, K=8, H=7168, T=1024, row_bytes=7168, scale_cols=56,
                            combine_dtype="bf16", mask_enabled=False, active_rank_mask=(1 << 32) - 1)
    Tm = ep_chunked.chunk_tokens(g)
    assert 1 <= Tm and g.ep * g.ep * Tm * g.row_bytes <= ep_chunked.CHUNK_RECV_BYTES
    assert ep_chunked.chunk_counts([5, 0, 12], 8, 4) == [0, 0, 4]
    assert ep_chunked.chunk_counts([5, 0, 12], 4, 4) == [1, 0, 4]
