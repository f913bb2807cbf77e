"""GPU parity at the workloads' full sizes, through the same EpComm/C-ABI
launch path the bench times: every token is compared with the oracle.

- The whole receive id plane of every rank is compared with the oracle's.
- Every token of every source rank is then compared bit for bit: its
  routed hidden, scale and weight rows in each rank it reaches, and its
  combine output. The oracle works through the tokens in chunks (tokens
  [t0, t0+Tm) of every rank as a problem of its own, see ep_chunked.py) on a
  pool of host processes; the chunks together cover the whole workload.
"""
import numpy as np
import pytest
import torch

import ep_chunked
import oracle
import workloads
from ep_testutil import fill_expert_outputs, out_bits, raw_bytes, to_dev

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


@pytest.mark.parametrize("name", ["tiny", "mixtral_decode", "dsv3_decode", "dsv3_prefill", "qwen3_mask",
                                  "large_bf16", "large_fp16", "large_fp32", "region_over_4gib"])
def test_full_size_every_token(cuda_device, oracle_pool, name):
    from combine_topk_ids_dest_gb300 import EpComm
    wl = workloads.WORKLOADS[name] if name in workloads.WORKLOADS else LARGE[name]
    inp = workloads.make_inputs(wl)
    ep, E, K, H = wl.ep_size, wl.num_experts, wl.top_k, wl.hidden
    comm = EpComm(ep, E, K, H, wl.capacity, dtype=wl.torch_dtype, enable_rank_mask=wl.enable_rank_mask,
                  device=cuda_device, combine_dtype=wl.combine_torch_dtype)
    try:
        mask = inp.active_rank_mask if wl.enable_rank_mask else None
        res = comm.dispatch(to_dev(inp.hidden, cuda_device), to_dev(inp.topk_ids, cuda_device),
                            to_dev(inp.topk_weights, cuda_device),
                            hidden_states_scale=to_dev(inp.scale, cuda_device),
                            runtime_max_tokens_per_rank=wl.runtime_max, active_rank_mask=mask)
        T = res.tokens_per_rank
        fill_expert_outputs(comm, T, cuda_device)
        out = comm.combine(active_rank_mask=mask)
        torch.cuda.synchronize(cuda_device)

        # 1. the whole id plane
        want_ids = oracle.dispatch(ep, E, K, T, inp.num_tokens, inp.hidden, inp.topk_ids,
                                   mask_enabled=wl.enable_rank_mask,
                                   active_rank_mask=inp.active_rank_mask, payload=False).recv_ids
        ids_host = [res.topk_ids[d].cpu().numpy() for d in range(ep)]
        for d in range(ep):
            np.testing.assert_array_equal(ids_host[d], want_ids[d], err_msg=f"id plane of rank {d}")
        del want_ids

        # 2. every token, chunk by chunk, on the oracle pool
        g = ep_chunked.Geometry(ep=ep, E=E, K=K, H=H, T=T, row_bytes=H * wl.elem_bytes,
                                scale_cols=wl.scale_cols, combine_dtype=wl.combine_dtype,
                                mask_enabled=wl.enable_rank_mask, active_rank_mask=inp.active_rank_mask)
        Tm = ep_chunked.chunk_tokens(g)
        n_chunks = len(ep_chunked.chunk_starts(inp.num_tokens, Tm))
        bufs = {"hidden": res.hidden_states, "scale": res.hidden_states_scale, "weights": res.topk_weights}

        def rows_of(kind, d, rows):
            x = bufs[kind][d].index_select(0, torch.from_numpy(rows).to(cuda_device)).cpu()
            return raw_bytes(x) if kind == "hidden" else x.numpy()

        def out_of(s, t0, m):
            return out_bits(out[s][t0:t0 + m].cpu())

        jobs = ep_chunked.make_jobs(g, inp, ids_host, Tm, rows_of, out_of, res.hidden_states_scale is not None,
                                    res.topk_weights is not None)
        checked = ep_chunked.run_jobs(oracle_pool, jobs, in_flight=2 * oracle_pool._max_workers)
        assert checked == n_chunks
        assert n_chunks * Tm >= max(inp.num_tokens)  # the chunks reach every rank's last token
    finally:
        comm.destroy()
