"""Partitioned EP groups (ep_partition_describe / ep_partition_connect): the
ep_size ranks split into G contiguous blocks, each in a workspace and handle
of its own, the layout the pages' one-rank-per-GPU backends use
(NVLinkOneSidedAlltoAll, class description: rows move between the ranks'
buffers with one-sided stores and loads). Here the G workspaces are separate
allocations on one GPU.

Every partition dispatches its own ranks' tokens into every rank's receive
rows and combines its own tokens from every rank's combine input; the
results, put back together by rank, must equal the oracle's bit for bit
(receive id rows everywhere, routed hidden/scale/weight rows, every output).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from combine_topk_ids_dest_gb300 import EP_ERR_STATE, EpComm, connect_partitions
from combine_topk_ids_dest_gb300._lib import EpError
from ep_testutil import (EO_SEED, assert_round_equal, clamp_count, cut_inputs, out_bits, raw_bytes,
                         small, to_dev)

pytestmark = pytest.mark.gpu


def _make(wl, G, device, **kw):
    comms = [EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, dtype=wl.torch_dtype,
                    enable_rank_mask=wl.enable_rank_mask, device=device,
                    scale_cols=wl.scale_cols if wl.scales else None, combine_dtype=wl.combine_torch_dtype,
                    num_partitions=G, partition=g, **kw) for g in range(G)]
    connect_partitions(comms)
    return comms


def _part(lst, c):
    return None if lst is None else lst[c.first_rank:c.first_rank + c.num_ranks]


def _partitioned_round(inp, G, device, streams=False, dev_counts=None, eplb=None, comms=None):
    """One step of every partition: all dispatches, the stand-in expert outputs
    of every rank, all combines. With ``streams`` each partition runs on a
    stream of its own and events order the phases across partitions."""
    wl = inp.wl
    own = comms is None
    comms = comms or _make(wl, G, device)
    mask = inp.active_rank_mask if wl.enable_rank_mask else None
    hid, ids = to_dev(inp.hidden, device), to_dev(inp.topk_ids, device)
    wts, scl = to_dev(inp.topk_weights, device), to_dev(inp.scale, device)
    dc = None if dev_counts is None else torch.tensor(dev_counts, dtype=torch.int32, device=device)
    main = torch.cuda.current_stream(device)
    ss = [torch.cuda.Stream(device) for _ in comms] if streams else [main] * len(comms)
    start = torch.cuda.Event()
    start.record(main)
    res, done = [], []
    for c, s in zip(comms, ss):
        s.wait_event(start)
        with torch.cuda.stream(s):
            r = c.dispatch(_part(hid, c), _part(ids, c), _part(wts, c), hidden_states_scale=_part(scl, c),
                           runtime_max_tokens_per_rank=wl.runtime_max, active_rank_mask=mask,
                           num_tokens_device=None if dc is None else dc[c.first_rank:c.first_rank + c.num_ranks],
                           eplb_local_stats=_part(eplb, c))
            e = torch.cuda.Event()
            e.record(s)
            done.append(e)
        res.append(r)
    for e in done:  # every partition's dispatch is complete before any expert reads its rows
        main.wait_event(e)
    T = res[0].tokens_per_rank
    rows = torch.arange(wl.ep_size * T, device=device)
    for c in comms:
        for j, buf in enumerate(c.get_combine_input_buffer()):
            buf.copy_(workloads.expert_output_rows(EO_SEED, c.first_rank + j, rows, wl.hidden, device=device,
                                                   dtype=wl.combine_dtype))
    experts = torch.cuda.Event()
    experts.record(main)
    outs, done = [], []
    for c, s in zip(comms, ss):
        s.wait_event(experts)
        with torch.cuda.stream(s):
            outs.append(c.combine(active_rank_mask=mask))
            e = torch.cuda.Event()
            e.record(s)
            done.append(e)
    for e in done:
        main.wait_event(e)
    torch.cuda.synchronize(device)
    out = [o for part in outs for o in part]
    if dev_counts is not None:
        out = [o[:clamp_count(n, m)] for o, n, m in zip(out, dev_counts, inp.num_tokens)]
    got = dict(T=T,
               recv_ids=[x.cpu().numpy() for r in res for x in r.topk_ids],
               recv_hidden=[raw_bytes(x.cpu()) for r in res for x in r.hidden_states],
               recv_scale=None if res[0].hidden_states_scale is None else
               [x.cpu().numpy() for r in res for x in r.hidden_states_scale],
               recv_weights=None if res[0].topk_weights is None else
               [x.cpu().numpy() for r in res for x in r.topk_weights],
               out=[out_bits(o.cpu()) for o in out],
               eplb=[None if r.eplb_global_stats is None else r.eplb_global_stats.cpu() for r in res])
    if own:
        for c in comms:
            c.destroy()
    return got


def _oracle(inp):
    wl = inp.wl
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
    return disp, [o.view(np.uint32) if o.dtype == np.float32 else o for o in out]


CASES = {
    "qwen3_mask": small(workloads.WORKLOADS["qwen3_mask"], hidden=512, tokens=40),
    "dsv3_decode": small(workloads.WORKLOADS["dsv3_decode"], hidden=1024, tokens=6),
    "dsv3_prefill": small(workloads.WORKLOADS["dsv3_prefill"], hidden=7168, tokens=8),
    "mixtral_decode": small(workloads.WORKLOADS["mixtral_decode"], hidden=4096, tokens=24),
    "fp32_combine": workloads.EpWorkload(name="part_f32", ep_size=8, num_experts=32, top_k=4, hidden=256,
                                         dtype="fp16", capacity=20, runtime_max=17, counts=("uniform", 0, 17),
                                         ids="with_invalid", combine_dtype="fp32", dropped_ranks=(6,), seed=71),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("G", [2, 4])
def test_partitioned_round_matches_oracle(cuda_device, name, G):
    inp = workloads.make_inputs(CASES[name])
    got = _partitioned_round(inp, G, cuda_device)
    disp, out = _oracle(inp)
    assert_round_equal(inp, got, disp, out)


def test_one_partition_per_rank_on_separate_streams(cuda_device):
    wl = CASES["mixtral_decode"]  # ep = 8: eight partitions of one rank each
    inp = workloads.make_inputs(wl)
    got = _partitioned_round(inp, wl.ep_size, cuda_device, streams=True)
    disp, out = _oracle(inp)
    assert_round_equal(inp, got, disp, out)


def test_partitions_with_device_counts_and_eplb(cuda_device):
    wl = CASES["qwen3_mask"]
    inp = workloads.make_inputs(wl)
    counts = [(5 * s + 7) % 45 - 3 for s in range(wl.ep_size)]
    stats = [torch.arange(12, dtype=torch.int32, device=cuda_device) * 100 + s for s in range(wl.ep_size)]
    comms = _make(wl, 4, cuda_device, eplb_stats_max_bytes=64)
    try:
        got = _partitioned_round(inp, 4, cuda_device, dev_counts=counts, eplb=stats, comms=comms)
    finally:
        for c in comms:
            c.destroy()
    cut = cut_inputs(inp, [clamp_count(c, n) for c, n in zip(counts, inp.num_tokens)])
    disp, out = _oracle(cut)
    for s in range(wl.ep_size):
        np.testing.assert_array_equal(got["out"][s], out[s], err_msg=f"combine output of rank {s}")
    for d in range(wl.ep_size):
        np.testing.assert_array_equal(got["recv_ids"][d], disp.recv_ids[d], err_msg=f"ids of rank {d}")
    want = oracle.eplb_gather([x.cpu() for x in stats])
    for g, st in enumerate(got["eplb"]):  # every partition holds every rank's statistics
        np.testing.assert_array_equal(st.contiguous().view(torch.uint8).numpy().reshape(wl.ep_size, -1), want,
                                      err_msg=f"gathered statistics of partition {g}")


def test_unconnected_partition_refuses_to_dispatch(cuda_device):
    wl = CASES["qwen3_mask"]
    c = EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, device=cuda_device,
               num_partitions=2, partition=1)
    try:
        inp = workloads.make_inputs(wl)
        with pytest.raises(EpError) as e:
            c.dispatch(to_dev(inp.hidden[8:], cuda_device), to_dev(inp.topk_ids[8:], cuda_device))
        assert e.value.status == EP_ERR_STATE
        other = EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, device=cuda_device,
                       num_partitions=2, partition=0)
        try:
            with pytest.raises(EpError):  # descriptions out of order
                c.connect([c.partition_info(), other.partition_info()])
            connect_partitions([other, c])
        finally:
            other.destroy()
    finally:
        c.destroy()


def _divisors(n):
    return [g for g in range(1, n + 1) if n % g == 0]


@pytest.mark.parametrize("seed", range(12))
def test_random_partitioned_geometry(cuda_device, seed):
    """The randomised geometries of the fuzz test, each split into a random
    number of partitions (a divisor of ep_size), with PDL on half of them."""
    import random

    from test_gpu_fuzz import _case
    wl, _ = _case(seed)
    rng = random.Random(7000 + seed)
    G = rng.choice(_divisors(wl.ep_size))
    inp = workloads.make_inputs(wl)
    comms = _make(wl, G, cuda_device, pdl=rng.random() < 0.5)
    try:
        got = _partitioned_round(inp, G, cuda_device, streams=rng.random() < 0.5, comms=comms)
    finally:
        for c in comms:
            c.destroy()
    disp, out = _oracle(inp)
    assert_round_equal(inp, got, disp, out)


def test_connect_refuses_another_group(cuda_device):
    """A handle is connected only with descriptions of its own group: a valid
    group of another size, or one whose own entry is another workspace, is
    refused."""
    wl = CASES["qwen3_mask"]
    kw = dict(device=cuda_device)
    four = [EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, num_partitions=4, partition=g, **kw)
            for g in range(4)]
    two = [EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, num_partitions=2, partition=g, **kw)
           for g in range(2)]
    try:
        infos2 = [c.partition_info() for c in two]
        with pytest.raises(EpError, match="one of 4 partitions"):
            four[3].connect(infos2)
        swapped = [c.partition_info() for c in four]
        other = EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, num_partitions=4, partition=1,
                       **kw)
        try:
            swapped[1] = other.partition_info()
            with pytest.raises(EpError, match="not of this handle's workspace"):
                four[1].connect(swapped)
        finally:
            other.destroy()
        connect_partitions(four)
    finally:
        for c in four + two:
            c.destroy()
