"""GPU parity at the workloads' full sizes, through the same EpComm/C-ABI
launch path the bench times.

- The whole receive id plane of every rank is compared with the oracle's
  (cheap at any size).
- A sample of source tokens (every rank represented, first and last slots
  included) is rebuilt as a small problem for the oracle; its receive rows and
  combine outputs must equal the GPU's rows for the same tokens bit for bit.
- Property at any size: a token's output is exactly the ordered fp32 sum of
  the stand-in expert rows of the ranks the oracle routes it to.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from ep_testutil import EO_SEED, INV, fill_expert_outputs, out_bits, raw_bytes, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLE = 256


def _sample_slots(inp, rng):
    ep = inp.wl.ep_size
    picks = {s: set() for s in range(ep)}
    live = [(s, t) for s in range(ep) for t in (0, inp.num_tokens[s] - 1) if inp.num_tokens[s] > 0]
    for s, t in live:
        picks[s].add(t)
    total = inp.total_tokens
    for _ in range(min(SAMPLE, total)):
        g = int(rng.integers(0, total))
        for s in range(ep):  # global token index -> (s, t)
            if g < inp.num_tokens[s]:
                picks[s].add(g)
                break
            g -= inp.num_tokens[s]
    return {s: sorted(v) for s, v in picks.items()}


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


@pytest.mark.parametrize("name", ["mixtral_decode", "dsv3_decode", "dsv3_prefill", "qwen3_mask",
                                  "large_bf16", "large_fp16", "large_fp32", "region_over_4gib"])
def test_full_size_sampled(cuda_device, name):
    from combine_topk_ids_dest_gb300 import EpComm
    wl = workloads.WORKLOADS[name] if name in workloads.WORKLOADS else LARGE[name]
    inp = workloads.make_inputs(wl)
    ep, E, K, H = wl.ep_size, wl.num_experts, wl.top_k, wl.hidden
    dtype = wl.torch_dtype
    comm = EpComm(ep, E, K, H, wl.capacity, dtype=dtype, enable_rank_mask=wl.enable_rank_mask,
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
        for d in range(ep):
            np.testing.assert_array_equal(res.topk_ids[d].cpu().numpy(), want_ids[d],
                                          err_msg=f"id plane of rank {d}")

        # 2. sampled tokens as a small oracle problem
        picks = _sample_slots(inp, np.random.default_rng(5))
        Tm = max(1, max(len(v) for v in picks.values()))
        def sub(lst, s):  # rows of the sampled tokens (fp8 rows indexed as raw bytes)
            if lst is None:
                return None
            x = lst[s].view(torch.uint8) if lst[s].dtype == torch.float8_e4m3fn else lst[s]
            return x[torch.tensor(picks[s], dtype=torch.long)]
        m_hidden = [sub(inp.hidden, s) for s in range(ep)]
        m_ids = [sub(inp.topk_ids, s) for s in range(ep)]
        m_w = None if inp.topk_weights is None else [sub(inp.topk_weights, s) for s in range(ep)]
        m_sc = None if inp.scale is None else [sub(inp.scale, s) for s in range(ep)]
        m_counts = [len(picks[s]) for s in range(ep)]
        # mini row s*Tm+j stands for full row s*T+picks[s][j]
        full_rows = np.zeros(ep * Tm, np.int64)
        for s in range(ep):
            for j, t in enumerate(picks[s]):
                full_rows[s * Tm + j] = s * T + t
        disp = oracle.dispatch(ep, E, K, Tm, m_counts, m_hidden, m_ids, scale=m_sc, topk_weights=m_w,
                               mask_enabled=wl.enable_rank_mask, active_rank_mask=inp.active_rank_mask,
                               row_bytes=H * wl.elem_bytes, scale_cols=wl.scale_cols)
        rows_t = torch.from_numpy(full_rows)
        eo = [out_bits(workloads.expert_output_rows(EO_SEED, d, rows_t, H, dtype=wl.combine_dtype))
              for d in range(ep)]
        mout = oracle.combine_typed(ep, E, K, H, Tm, m_counts, m_ids, eo, wl.combine_dtype,
                                    mask_enabled=wl.enable_rank_mask,
                              active_rank_mask=inp.active_rank_mask)

        live = np.array([j < m_counts[s] for s in range(ep) for j in range(Tm)])
        idx = torch.from_numpy(full_rows[live]).to(cuda_device)
        for d in range(ep):
            want = disp.recv_ids[d][live]
            np.testing.assert_array_equal(res.topk_ids[d].index_select(0, idx).cpu().numpy(), want)
            valid = (want != INV).any(axis=1)
            got_h = raw_bytes(res.hidden_states[d].index_select(0, idx).cpu())
            np.testing.assert_array_equal(got_h[valid], disp.recv_hidden[d][live][valid])
            if m_sc is not None:
                got = res.hidden_states_scale[d].index_select(0, idx).cpu().numpy()
                np.testing.assert_array_equal(got[valid].view(np.uint32),
                                              disp.recv_scale[d][live][valid].view(np.uint32))
            if m_w is not None:
                got = res.topk_weights[d].index_select(0, idx).cpu().numpy()
                np.testing.assert_array_equal(got[valid].view(np.uint32),
                                              disp.recv_weights[d][live][valid].view(np.uint32))
        for s in range(ep):
            if not picks[s]:
                continue
            ts = torch.tensor(picks[s], dtype=torch.long, device=cuda_device)
            got = out_bits(out[s].index_select(0, ts).cpu())
            if got.dtype == np.uint32:
                mout[s] = mout[s].view(np.uint32)
            np.testing.assert_array_equal(got, mout[s], err_msg=f"combine output of rank {s}")
    finally:
        comm.destroy()
