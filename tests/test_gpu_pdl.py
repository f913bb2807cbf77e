"""Programmatic dependent launch (EP_LAUNCH_PDL): the same results as
ordinary stream order, bit for bit against the oracle.

With the flag each kernel lets the next one of its stream be scheduled
early and waits (griddepcontrol.wait) for its predecessor before touching
global memory. The tests cover a combine right after its dispatch, device
token counts that the dispatch leaves for the combine, and rounds queued back
to back with no host synchronisation, where the next dispatch rewrites the
routing state and receive rows the previous combine reads.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from combine_topk_ids_dest_gb300 import EpComm
from ep_testutil import (EO_SEED, assert_round_equal, bf16_bits, clamp_count, cut_inputs, gpu_round,
                         oracle_round, raw_bytes, small, to_dev)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "mixtral_decode", "dsv3_decode", "dsv3_prefill", "qwen3_mask"])
def test_pdl_round_matches_oracle(cuda_device, name):
    wl = workloads.WORKLOADS[name]
    if name != "tiny":
        wl = small(wl, hidden=1024, tokens=40)
    inp = workloads.make_inputs(wl)
    got = gpu_round(inp, cuda_device, pdl=True)
    disp, out = oracle_round(inp)
    assert_round_equal(inp, got, disp, out)


def test_pdl_with_device_counts(cuda_device):
    wl = small(workloads.WORKLOADS["qwen3_mask"], hidden=512, tokens=32)
    inp = workloads.make_inputs(wl)
    counts = [(7 * s + 3) % 40 - 4 for s in range(wl.ep_size)]  # ragged, some negative, some above
    got = gpu_round(inp, cuda_device, dev_counts=counts, pdl=True)
    cut = cut_inputs(inp, [clamp_count(c, n) for c, n in zip(counts, inp.num_tokens)])
    disp, out = oracle_round(cut)
    for s in range(wl.ep_size):
        np.testing.assert_array_equal(got["out"][s], out[s], err_msg=f"combine output of rank {s}")
    for d in range(wl.ep_size):
        np.testing.assert_array_equal(got["recv_ids"][d], disp.recv_ids[d], err_msg=f"ids of rank {d}")


def test_pdl_rounds_back_to_back_without_host_sync(cuda_device):
    """Four rounds with different inputs queued on one stream; the host waits
    only at the end. Receive rows are copied out on the stream right after
    each dispatch, before the next round can overwrite them."""
    dev = cuda_device
    base = small(workloads.WORKLOADS["dsv3_prefill"], hidden=1024, tokens=24)
    wls = [base.replace(name=f"b2b{i}", seed=60 + i, counts=("uniform", 0, 24)) for i in range(4)]
    comm = EpComm(base.ep_size, base.num_experts, base.top_k, base.hidden, base.capacity,
                  dtype=base.torch_dtype, device=dev, pdl=True)
    try:
        rounds = []
        for i, wl in enumerate(wls):
            inp = workloads.make_inputs(wl)
            res = comm.dispatch(to_dev(inp.hidden, dev), to_dev(inp.topk_ids, dev), to_dev(inp.topk_weights, dev),
                                hidden_states_scale=to_dev(inp.scale, dev))
            T = res.tokens_per_rank
            ids_copy = [x.clone() for x in res.topk_ids]
            hid_copy = [x.clone() for x in res.hidden_states]
            rows = torch.arange(base.ep_size * T, device=dev)
            eo = [workloads.expert_output_rows(EO_SEED + i, d, rows, base.hidden, device=dev).contiguous()
                  for d in range(base.ep_size)]
            out = comm.combine(eo)
            rounds.append((inp, T, ids_copy, hid_copy, out))
        torch.cuda.synchronize(dev)
        for i, (inp, T, ids_copy, hid_copy, out) in enumerate(rounds):
            ep, E, K, H = base.ep_size, base.num_experts, base.top_k, base.hidden
            want = oracle.dispatch(ep, E, K, T, inp.num_tokens, inp.hidden, inp.topk_ids, scale=inp.scale,
                                   topk_weights=inp.topk_weights, row_bytes=H * base.elem_bytes,
                                   scale_cols=base.scale_cols)
            rows = torch.arange(ep * T)
            eo_host = [bf16_bits(workloads.expert_output_rows(EO_SEED + i, d, rows, H)) for d in range(ep)]
            want_out = oracle.combine(ep, E, K, H, T, inp.num_tokens, inp.topk_ids, eo_host)
            for d in range(ep):
                np.testing.assert_array_equal(ids_copy[d].cpu().numpy(), want.recv_ids[d],
                                              err_msg=f"round {i}: ids of rank {d}")
                valid = (want.recv_ids[d] != -1).any(axis=1)
                np.testing.assert_array_equal(raw_bytes(hid_copy[d].cpu())[valid], want.recv_hidden[d][valid],
                                              err_msg=f"round {i}: hidden rows of rank {d}")
            for s in range(ep):
                np.testing.assert_array_equal(bf16_bits(out[s].cpu()), want_out[s],
                                              err_msg=f"round {i}: combine output of rank {s}")
    finally:
        comm.destroy()
