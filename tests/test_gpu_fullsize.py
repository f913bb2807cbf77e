"""GPU parity at the workloads' full sizes, through the same EpComm/C-ABI
launch path the bench times: every token is compared with the oracle.

- The whole receive id plane of every rank is compared with the oracle's.
- Every token of every source rank is then compared bit for bit: its
  routed hidden, scale and weight rows in each rank it reaches, and its
  combine output. The oracle works through the tokens in chunks (tokens
  [t0, t0+Tm) of every rank as a problem of its own, see ep_chunked.py) on a
  pool of host processes; the chunks together cover the whole workload.
- Two workloads run again as partitioned groups (the ranks split into G
  blocks, each with a workspace and communicator of its own) and are
  compared the same way.
"""
import numpy as np
import pytest
import torch

import ep_chunked
import oracle
import workloads
from ep_testutil import fill_expert_outputs, out_bits, raw_bytes

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


# Combines whose output reaches 192 MiB take the library's 32-byte-access path;
# these cover it for every combine type (the prefill workload covers bf16 too).
LARGE = {
    f"large_{cdt}": workloads.EpWorkload(
        name=f"large_{cdt}", ep_size=4, num_experts=16, top_k=4, hidden=7168, dtype="bf16",
        capacity=5000 if cdt == "fp32" else 9400, runtime_max=None, counts=("full",),
        combine_dtype=cdt, dropped_ranks=(2,), seed=31)
    for cdt in ("bf16", "fp16", "fp32")
}
# One receive region (and one combine-input region) larger than 4 GiB: 64 KB fp32
# rows, 4 ranks x 16400 slots; only rank 3 sends, so its last slots lie more than
# 2^32 bytes into every region while the inputs stay at about 1 GB.
LARGE["region_over_4gib"] = workloads.EpWorkload(
    name="region_over_4gib", ep_size=4, num_experts=8, top_k=2, hidden=16384, dtype="fp32", capacity=16400,
    runtime_max=None, counts=("fixed", 0, 0, 0, 16400), combine_dtype="fp32", seed=33)


@pytest.fixture(scope="module")
def oracle_pool():
    ex = ep_chunked.pool()
    try:
        yield ex
    finally:
        ex.shutdown(wait=True, cancel_futures=True)


def _round(wl, inp, G, device):
    """dispatch + stand-in expert outputs + combine of the whole workload, with
    one communicator (G = 1) or G partitions (each with its own workspace);
    returns the communicators, every rank's receive views by global rank, the
    outputs by source rank, and tokens_per_rank."""
    from combine_topk_ids_dest_gb300 import EpComm, connect_partitions
    ep, E, K, H = wl.ep_size, wl.num_experts, wl.top_k, wl.hidden
    comms = [EpComm(ep, E, K, H, wl.capacity, dtype=wl.torch_dtype, enable_rank_mask=wl.enable_rank_mask,
                    device=device, combine_dtype=wl.combine_torch_dtype, num_partitions=G, partition=g)
             for g in range(G)]
    if G > 1:
        connect_partitions(comms)
    mask = inp.active_rank_mask if wl.enable_rank_mask else None
    part = lambda lst, c: None if lst is None else [x.to(device) for x in lst[c.first_rank:c.first_rank + c.num_ranks]]
    res = [c.dispatch(part(inp.hidden, c), part(inp.topk_ids, c), part(inp.topk_weights, c),
                      hidden_states_scale=part(inp.scale, c), runtime_max_tokens_per_rank=wl.runtime_max,
                      active_rank_mask=mask) for c in comms]
    T = res[0].tokens_per_rank
    for c in comms:
        fill_expert_outputs(c, T, device)
    out = [o for c in comms for o in c.combine(active_rank_mask=mask)]
    torch.cuda.synchronize(device)
    bufs = {"hidden": [x for r in res for x in r.hidden_states],
            "scale": None if res[0].hidden_states_scale is None else [x for r in res for x in r.hidden_states_scale],
            "weights": None if res[0].topk_weights is None else [x for r in res for x in r.topk_weights],
            "ids": [x for r in res for x in r.topk_ids]}
    return comms, bufs, out, T


@pytest.mark.parametrize("name,G", [("tiny", 1), ("mixtral_decode", 1), ("dsv3_decode", 1), ("dsv3_prefill", 1),
                                    ("qwen3_mask", 1), ("large_bf16", 1), ("large_fp16", 1), ("large_fp32", 1),
                                    ("region_over_4gib", 1), ("dsv3_prefill", 4), ("qwen3_mask", 2)])
def test_full_size_every_token(cuda_device, oracle_pool, name, G):
    """G > 1: the same workload as G partitions, each with its own workspace."""
    wl = workloads.WORKLOADS[name] if name in workloads.WORKLOADS else LARGE[name]
    inp = workloads.make_inputs(wl)
    ep, E, K, H = wl.ep_size, wl.num_experts, wl.top_k, wl.hidden
    comms, bufs, out, T = _round(wl, inp, G, cuda_device)
    try:
        # 1. the whole id plane
        want_ids = oracle.dispatch(ep, E, K, T, inp.num_tokens, inp.hidden, inp.topk_ids,
                                   mask_enabled=wl.enable_rank_mask,
                                   active_rank_mask=inp.active_rank_mask, payload=False).recv_ids
        ids_host = [bufs["ids"][d].cpu().numpy() for d in range(ep)]
        for d in range(ep):
            np.testing.assert_array_equal(ids_host[d], want_ids[d], err_msg=f"id plane of rank {d}")
        del want_ids

        # 2. every token, chunk by chunk, on the oracle pool
        g = ep_chunked.Geometry(ep=ep, E=E, K=K, H=H, T=T, row_bytes=H * wl.elem_bytes,
                                scale_cols=wl.scale_cols, combine_dtype=wl.combine_dtype,
                                mask_enabled=wl.enable_rank_mask, active_rank_mask=inp.active_rank_mask)
        Tm = ep_chunked.chunk_tokens(g)
        n_chunks = len(ep_chunked.chunk_starts(inp.num_tokens, Tm))

        def rows_of(kind, d, rows):
            x = bufs[kind][d].index_select(0, torch.from_numpy(rows).to(cuda_device)).cpu()
            return raw_bytes(x) if kind == "hidden" else x.numpy()

        def out_of(s, t0, m):
            return out_bits(out[s][t0:t0 + m].cpu())

        jobs = ep_chunked.make_jobs(g, inp, ids_host, Tm, rows_of, out_of, bufs["scale"] is not None,
                                    bufs["weights"] is not None)
        checked = ep_chunked.run_jobs(oracle_pool, jobs, in_flight=2 * oracle_pool._max_workers)
        assert checked == n_chunks
        assert n_chunks * Tm >= max(inp.num_tokens)  # the chunks reach every rank's last token
    finally:
        for c in comms:
            c.destroy()
