"""The binding's stacked form: one [ep_size, M, ...] tensor per operand and a
list of per-rank counts, instead of ep_size per-rank tensors. It must give
exactly what the per-rank form gives (receive rows, ids, scales, weights and
combine outputs, bit for bit), never read the padding rows past a rank's
count, and leave stacked output rows past the counts untouched (the combine
returns the stacked output itself)."""
import pytest
import torch

import workloads
from combine_topk_ids_dest_gb300 import EpComm
from ep_testutil import EO_SEED, INV, to_dev

pytestmark = pytest.mark.gpu

WL = workloads.EpWorkload(name="stacked", ep_size=16, num_experts=64, top_k=8, hidden=512, dtype="fp8_e4m3",
                          scales=True, capacity=40, runtime_max=32, counts=("uniform", 0, 32),
                          empty_ranks=(5,), dropped_ranks=(3, 11), seed=91)
SENTINEL = 0x7FC1


def _stack(lst, M, fill):
    """[ep, M, cols] tensor whose rank s rows are lst[s] and whose padding rows hold `fill` bits."""
    ep, cols = len(lst), lst[0].shape[1]
    out = torch.empty(ep, M, cols, dtype=lst[0].dtype)
    raw = out.view(torch.uint8)  # byte views: fp8 tensors cannot be index-assigned on the CPU everywhere
    raw.fill_(fill)
    for s, x in enumerate(lst):
        if x.shape[0]:
            raw[s, :x.shape[0]] = x.contiguous().view(torch.uint8)
    return out


def test_stacked_form_equals_per_rank_form(cuda_device):
    inp = workloads.make_inputs(WL)
    mask = inp.active_rank_mask
    M = WL.tokens_per_rank
    comms = [EpComm(WL.ep_size, WL.num_experts, WL.top_k, WL.hidden, WL.capacity, dtype=WL.torch_dtype,
                    enable_rank_mask=True, device=cuda_device) for _ in range(2)]
    try:
        rows = torch.arange(WL.ep_size * M, device=cuda_device)
        eo = [workloads.expert_output_rows(EO_SEED, d, rows, WL.hidden, device=cuda_device)
              for d in range(WL.ep_size)]
        # padding rows past each count hold bytes that must never be read: id 0 (which would route
        # the row to rank 0) and non-zero payload
        hid = _stack(inp.hidden, M, 0x7E).to(cuda_device)
        ids = _stack(inp.topk_ids, M, 0x00).to(cuda_device)
        w = _stack(inp.topk_weights, M, 0x40).to(cuda_device)
        sc = _stack(inp.scale, M, 0x40).to(cuda_device)
        a = comms[0].dispatch(hid, ids, w, hidden_states_scale=sc, runtime_max_tokens_per_rank=WL.runtime_max,
                              active_rank_mask=mask, num_tokens=inp.num_tokens)
        out_a = comms[0].combine(torch.stack(eo), active_rank_mask=mask)
        b = comms[1].dispatch(to_dev(inp.hidden, cuda_device), to_dev(inp.topk_ids, cuda_device),
                              to_dev(inp.topk_weights, cuda_device), hidden_states_scale=to_dev(inp.scale, cuda_device),
                              runtime_max_tokens_per_rank=WL.runtime_max, active_rank_mask=mask)
        out_b = comms[1].combine(eo, active_rank_mask=mask)
        torch.cuda.synchronize(cuda_device)
        for d in range(WL.ep_size):
            ia, ib = a.topk_ids[d].cpu(), b.topk_ids[d].cpu()
            assert torch.equal(ia, ib), f"ids of rank {d}"
            valid = (ib != INV).any(dim=1)
            assert torch.equal(a.hidden_states[d].cpu().view(torch.uint8)[valid],
                               b.hidden_states[d].cpu().view(torch.uint8)[valid])
            assert torch.equal(a.hidden_states_scale[d].cpu()[valid].view(torch.int32),
                               b.hidden_states_scale[d].cpu()[valid].view(torch.int32))
            assert torch.equal(a.topk_weights[d].cpu()[valid].view(torch.int32),
                               b.topk_weights[d].cpu()[valid].view(torch.int32))
        assert isinstance(out_a, torch.Tensor) and out_a.shape == (WL.ep_size, max(inp.num_tokens), WL.hidden)
        for s, n in enumerate(inp.num_tokens):
            assert torch.equal(out_a[s, :n].cpu().view(torch.int16), out_b[s].cpu().view(torch.int16)), f"rank {s}"
    finally:
        for c in comms:
            c.destroy()


def test_stacked_output_rows_past_the_counts_are_untouched(cuda_device):
    inp = workloads.make_inputs(WL)
    mask = inp.active_rank_mask
    M = WL.tokens_per_rank
    comm = EpComm(WL.ep_size, WL.num_experts, WL.top_k, WL.hidden, WL.capacity, dtype=WL.torch_dtype,
                  enable_rank_mask=True, device=cuda_device)
    try:
        hid = _stack(inp.hidden, M, 0).to(cuda_device)
        ids = _stack(inp.topk_ids, M, 0xFF).to(cuda_device)
        w = _stack(inp.topk_weights, M, 0).to(cuda_device)
        sc = _stack(inp.scale, M, 0).to(cuda_device)
        comm.dispatch(hid, ids, w, hidden_states_scale=sc, runtime_max_tokens_per_rank=WL.runtime_max,
                      active_rank_mask=mask, num_tokens=inp.num_tokens)
        out = torch.full((WL.ep_size, M + 3, WL.hidden), SENTINEL, dtype=torch.int16,
                         device=cuda_device).view(torch.bfloat16)
        res = comm.combine(output=out, active_rank_mask=mask)
        torch.cuda.synchronize(cuda_device)
        assert res is out
        bits = out.view(torch.int16).cpu().numpy()
        for s, n in enumerate(inp.num_tokens):
            assert (bits[s, n:] == SENTINEL).all(), f"rank {s} wrote past its count"
    finally:
        comm.destroy()


def test_stacked_argument_checks(cuda_device):
    comm = EpComm(2, 4, 2, 64, 8, device=cuda_device)
    try:
        hid = torch.zeros(2, 5, 64, dtype=torch.bfloat16, device=cuda_device)
        ids = torch.zeros(2, 5, 2, dtype=torch.int32, device=cuda_device)
        bad = [
            dict(hidden_states=hid, topk_ids=ids[:, :4]),                         # ids rows differ
            dict(hidden_states=hid, topk_ids=ids.to(torch.int64)),                # ids dtype
            dict(hidden_states=hid[:1], topk_ids=ids[:1]),                        # not ep_size ranks
            dict(hidden_states=hid, topk_ids=ids, num_tokens=[5, 6]),             # count past the rows
            dict(hidden_states=hid, topk_ids=ids, num_tokens=[5]),                # one count missing
            dict(hidden_states=hid.transpose(0, 1).contiguous().transpose(0, 1), topk_ids=ids),  # not contiguous
            dict(hidden_states=list(hid), topk_ids=list(ids), num_tokens=[5, 5]),  # counts with lists
        ]
        for kw in bad:
            with pytest.raises(ValueError):
                comm.dispatch(**kw)
        comm.dispatch(hid, ids, num_tokens=[3, 5])
        with pytest.raises(ValueError):  # stacked output with too few rows
            comm.combine(output=torch.zeros(2, 4, 64, dtype=torch.bfloat16, device=cuda_device))
        out = comm.combine()
        assert out.shape == (2, 5, 64)
    finally:
        comm.destroy()


def test_stacked_form_with_device_counts(cuda_device):
    """Stacked operands with device-side counts: the same as per-rank tensors cut
    to those counts."""
    inp = workloads.make_inputs(WL)
    mask = inp.active_rank_mask
    M = WL.tokens_per_rank
    dev_counts = [min(n, 5) if s % 3 else n for s, n in enumerate(inp.num_tokens)]
    comms = [EpComm(WL.ep_size, WL.num_experts, WL.top_k, WL.hidden, WL.capacity, dtype=WL.torch_dtype,
                    enable_rank_mask=True, device=cuda_device) for _ in range(2)]
    try:
        rows = torch.arange(WL.ep_size * M, device=cuda_device)
        eo = torch.stack([workloads.expert_output_rows(EO_SEED, d, rows, WL.hidden, device=cuda_device)
                          for d in range(WL.ep_size)])
        a = comms[0].dispatch(_stack(inp.hidden, M, 0x7E).to(cuda_device), _stack(inp.topk_ids, M, 0).to(cuda_device),
                              _stack(inp.topk_weights, M, 0x40).to(cuda_device),
                              hidden_states_scale=_stack(inp.scale, M, 0x40).to(cuda_device),
                              runtime_max_tokens_per_rank=WL.runtime_max, active_rank_mask=mask,
                              num_tokens=inp.num_tokens,
                              num_tokens_device=torch.tensor(dev_counts, dtype=torch.int32, device=cuda_device))
        out_a = comms[0].combine(eo, active_rank_mask=mask)
        cut = lambda lst: [x[:n].contiguous().to(cuda_device) for x, n in zip(lst, dev_counts)]
        b = comms[1].dispatch(cut(inp.hidden), cut(inp.topk_ids), cut(inp.topk_weights),
                              hidden_states_scale=cut(inp.scale), runtime_max_tokens_per_rank=WL.runtime_max,
                              active_rank_mask=mask)
        out_b = comms[1].combine(eo, active_rank_mask=mask)
        torch.cuda.synchronize(cuda_device)
        for d in range(WL.ep_size):
            assert torch.equal(a.topk_ids[d], b.topk_ids[d]), f"ids of rank {d}"
            valid = (b.topk_ids[d] != INV).any(dim=1)
            assert torch.equal(a.hidden_states[d][valid].view(torch.uint8), b.hidden_states[d][valid].view(torch.uint8))
        for s, n in enumerate(dev_counts):
            assert torch.equal(out_a[s, :n].view(torch.int16), out_b[s].view(torch.int16)), f"rank {s}"
    finally:
        for c in comms:
            c.destroy()
