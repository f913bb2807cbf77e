"""Device-side token counts (ep_dispatch_args.num_tokens_device): one captured
CUDA graph of dispatch + combine, replayed with different per-rank counts
written into a device array between replays.

After each replay the receive buffers and the combine outputs must equal the
oracle's dispatch and combine of the same inputs cut to those counts (each
count clamped to [0, the rank's maximum]); output rows at or past a rank's
count must be left as they were.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from combine_topk_ids_dest_gb300 import EpComm
from ep_testutil import EO_SEED, INV, bf16_bits, raw_bytes, to_dev

pytestmark = pytest.mark.gpu

# 8 ranks, per-rank maxima of 0..64 tokens, duplicate ids, rank 2 masked off.
MAXIMA = (64, 40, 64, 0, 64, 64, 12, 64)
WL = workloads.EpWorkload(name="devcounts", ep_size=8, num_experts=32, top_k=4, hidden=1024, dtype="bf16",
                          capacity=64, runtime_max=None, counts=("fixed",) + MAXIMA, ids="uniform_dups",
                          dropped_ranks=(2,), seed=81)
COUNT_SETS = [
    list(MAXIMA),                       # every rank at its maximum
    [10, 0, 63, 0, 1, 64, 12, 5],       # ragged, some empty
    [-3, 99, 0, 0, 64, 2, 13, 70],      # out of range: clamped to [0, maximum]
    [0] * 8,                            # nothing at all
]
SENTINEL = 0x7FC1


def _expected(inp, counts):
    """Oracle dispatch and combine of the inputs cut to `counts`."""
    T, ep, H = WL.capacity, WL.ep_size, WL.hidden
    hid = [h[:n] for h, n in zip(inp.hidden, counts)]
    ids = [x[:n] for x, n in zip(inp.topk_ids, counts)]
    w = [x[:n] for x, n in zip(inp.topk_weights, counts)]
    disp = oracle.dispatch(ep, WL.num_experts, WL.top_k, T, counts, hid, ids, topk_weights=w,
                           mask_enabled=True, active_rank_mask=inp.active_rank_mask, row_bytes=2 * H)
    rows = torch.arange(ep * T)
    eo = [bf16_bits(workloads.expert_output_rows(EO_SEED, d, rows, H)) for d in range(ep)]
    out = oracle.combine(ep, WL.num_experts, WL.top_k, H, T, counts, ids, eo, mask_enabled=True,
                         active_rank_mask=inp.active_rank_mask)
    return disp, out


def test_one_graph_serves_changing_device_counts(cuda_device):
    inp = workloads.make_inputs(WL)
    mask = inp.active_rank_mask
    comm = EpComm(WL.ep_size, WL.num_experts, WL.top_k, WL.hidden, WL.capacity, enable_rank_mask=True,
                  device=cuda_device)
    try:
        hid, ids, w = (to_dev(inp.hidden, cuda_device), to_dev(inp.topk_ids, cuda_device),
                       to_dev(inp.topk_weights, cuda_device))
        rows = torch.arange(WL.ep_size * WL.capacity, device=cuda_device)
        eo = [workloads.expert_output_rows(EO_SEED, d, rows, WL.hidden, device=cuda_device)
              for d in range(WL.ep_size)]
        outs = [torch.empty(n, WL.hidden, dtype=torch.bfloat16, device=cuda_device) for n in MAXIMA]
        dev_counts = torch.tensor(MAXIMA, dtype=torch.int32, device=cuda_device)

        def round_():
            res = comm.dispatch(hid, ids, w, active_rank_mask=mask, num_tokens_device=dev_counts)
            comm.combine(eo, output=outs, active_rank_mask=mask)
            return res

        side = torch.cuda.Stream(cuda_device)
        side.wait_stream(torch.cuda.current_stream(cuda_device))
        with torch.cuda.stream(side):
            round_()  # warm-up outside the capture
        torch.cuda.current_stream(cuda_device).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            res = round_()

        for counts in COUNT_SETS:
            live = [min(max(c, 0), m) for c, m in zip(counts, MAXIMA)]
            dev_counts.copy_(torch.tensor(counts, dtype=torch.int32))
            for o in outs:
                o.view(torch.int16).fill_(SENTINEL)
            g.replay()
            torch.cuda.synchronize(cuda_device)
            disp, out = _expected(inp, live)
            for d in range(WL.ep_size):
                got_ids = res.topk_ids[d].cpu().numpy()
                np.testing.assert_array_equal(got_ids, disp.recv_ids[d], err_msg=f"counts {counts}, rank {d}")
                valid = (disp.recv_ids[d] != INV).any(axis=1)
                np.testing.assert_array_equal(raw_bytes(res.hidden_states[d].cpu())[valid],
                                              disp.recv_hidden[d][valid])
                np.testing.assert_array_equal(res.topk_weights[d].cpu().numpy()[valid],
                                              disp.recv_weights[d][valid])
            for s in range(WL.ep_size):
                o = bf16_bits(outs[s].cpu())
                np.testing.assert_array_equal(o[:live[s]], out[s], err_msg=f"counts {counts}, rank {s}")
                assert (o[live[s]:] == SENTINEL).all(), f"counts {counts}: rank {s} wrote past its count"
    finally:
        torch.cuda.synchronize(cuda_device)
        comm.destroy()


def test_device_counts_equal_host_counts_eagerly(cuda_device):
    """Without a graph: dispatch with device counts over full-size tensors gives
    what dispatch with host counts over the cut tensors gives."""
    inp = workloads.make_inputs(WL)
    mask = inp.active_rank_mask
    counts = COUNT_SETS[1]
    comms = [EpComm(WL.ep_size, WL.num_experts, WL.top_k, WL.hidden, WL.capacity, enable_rank_mask=True,
                    device=cuda_device) for _ in range(2)]
    try:
        rows = torch.arange(WL.ep_size * WL.capacity, device=cuda_device)
        eo = [workloads.expert_output_rows(EO_SEED, d, rows, WL.hidden, device=cuda_device)
              for d in range(WL.ep_size)]
        a = comms[0].dispatch(to_dev(inp.hidden, cuda_device), to_dev(inp.topk_ids, cuda_device),
                              to_dev(inp.topk_weights, cuda_device), active_rank_mask=mask,
                              num_tokens_device=torch.tensor(counts, dtype=torch.int32, device=cuda_device))
        out_a = comms[0].combine(eo, active_rank_mask=mask)
        cut = lambda lst: [x[:n].to(cuda_device) for x, n in zip(lst, counts)]
        b = comms[1].dispatch(cut(inp.hidden), cut(inp.topk_ids), cut(inp.topk_weights), active_rank_mask=mask)
        out_b = comms[1].combine(eo, active_rank_mask=mask)
        for d in range(WL.ep_size):
            assert torch.equal(a.topk_ids[d], b.topk_ids[d])
            valid = (b.topk_ids[d] != INV).any(dim=1)
            assert torch.equal(a.hidden_states[d][valid].view(torch.int16), b.hidden_states[d][valid].view(torch.int16))
        for s, n in enumerate(counts):
            assert torch.equal(out_a[s][:n].view(torch.int16), out_b[s].view(torch.int16))
    finally:
        for c in comms:
            c.destroy()


def test_device_counts_argument_checks(cuda_device):
    comm = EpComm(2, 4, 2, 64, 8, device=cuda_device)
    try:
        hid = [torch.zeros(3, 64, dtype=torch.bfloat16, device=cuda_device)] * 2
        ids = [torch.zeros(3, 2, dtype=torch.int32, device=cuda_device)] * 2
        for bad in (torch.zeros(2, dtype=torch.int64, device=cuda_device),   # wrong dtype
                    torch.zeros(3, dtype=torch.int32, device=cuda_device),   # wrong length
                    torch.zeros(2, dtype=torch.int32)):                      # on the CPU
            with pytest.raises(ValueError):
                comm.dispatch(hid, ids, num_tokens_device=bad)
    finally:
        comm.destroy()
