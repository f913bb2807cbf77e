"""ep_combine_noalloc: the combine for callers that cannot allocate device memory.

Such callers (code inside an arena that owns all device memory, plug-ins of a
runtime that forbids their own allocations, code running during a stream
capture) have no ep_handle, whose workspace is an allocation; this entry point
keeps its only scratch in a fixed device array inside the library. The GPU
test calls it through the C ABI and checks its output bit for bit (the
tolerance of every combine test here) against ep_combine after ep_dispatch with
the same ids, mask and expert outputs, on two calls in a row whose routing
differs, so anything the first call leaves in the shared scratch would show in
the second.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from combine_topk_ids_dest_gb300 import EP_ERR_INVALID_ARG, EP_OK, EpComm, _lib
from combine_topk_ids_dest_gb300._lib import ptr_array
from ep_testutil import fill_expert_outputs, to_dev

ROUNDS = [
    # a wide round first: 16 ranks x 96 slots, two ranks masked off, one empty rank
    workloads.EpWorkload(name="noalloc_a", ep_size=16, num_experts=64, top_k=8, hidden=512,
                         dtype="bf16", capacity=96, runtime_max=96, counts=("uniform", 0, 96),
                         empty_ranks=(4,), dropped_ranks=(3, 9), seed=21),
    # then fewer slots, every rank active, duplicate ids
    workloads.EpWorkload(name="noalloc_b", ep_size=16, num_experts=64, top_k=8, hidden=512,
                         dtype="bf16", capacity=96, runtime_max=40, counts=("uniform", 1, 40),
                         ids="uniform_dups", dropped_ranks=(), seed=22),
]


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.gpu
def test_noalloc_combine_matches_combine_on_two_calls(cuda_device):
    L = _lib.load()
    wl0 = ROUNDS[0]
    comm = EpComm(wl0.ep_size, wl0.num_experts, wl0.top_k, wl0.hidden, wl0.capacity,
                  enable_rank_mask=True, device=cuda_device)
    try:
        for wl in ROUNDS:
            inp = workloads.make_inputs(wl)
            ids = to_dev(inp.topk_ids, cuda_device)
            mask = inp.active_rank_mask
            res = comm.dispatch(to_dev(inp.hidden, cuda_device), ids,
                                to_dev(inp.topk_weights, cuda_device),
                                runtime_max_tokens_per_rank=wl.runtime_max, active_rank_mask=mask)
            T = res.tokens_per_rank
            eo = fill_expert_outputs(comm, T, cuda_device, caller=True)
            want = comm.combine(eo, active_rank_mask=mask)

            got = [torch.full((n, wl.hidden), float("nan"), dtype=torch.bfloat16, device=cuda_device)
                   for n in inp.num_tokens]
            counts = (ctypes.c_int32 * wl.ep_size)(*inp.num_tokens)
            stream = torch.cuda.current_stream(cuda_device).cuda_stream
            st = L.ep_combine_noalloc(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, T, counts,
                                      ptr_array([x.data_ptr() for x in ids]), mask,
                                      ptr_array([e.data_ptr() for e in eo]),
                                      ptr_array([o.data_ptr() for o in got]),
                                      ctypes.c_void_p(stream))
            assert st == EP_OK, L.ep_last_error()
            torch.cuda.synchronize(cuda_device)
            for s in range(wl.ep_size):
                np.testing.assert_array_equal(_bits(got[s]), _bits(want[s]),
                                              err_msg=f"{wl.name}: output of rank {s}")
    finally:
        comm.destroy()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    L = _lib.load()
    ep, T = 64, _lib.EP_NOALLOC_MAX_SLOTS // 64 + 1
    counts = (ctypes.c_int32 * ep)(*([0] * ep))
    nulls = ptr_array([0] * ep)
    st = L.ep_combine_noalloc(ep, 64, 8, 256, T, counts, nulls, _lib.ALL_RANKS, nulls, nulls, None)
    assert st == EP_ERR_INVALID_ARG
    assert b"static scratch" in L.ep_last_error()


@pytest.mark.gpu
def test_python_wrapper_matches_combine(cuda_device):
    from combine_topk_ids_dest_gb300 import combine_noalloc
    wl = ROUNDS[0]
    inp = workloads.make_inputs(wl)
    comm = EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, enable_rank_mask=True,
                  device=cuda_device)
    try:
        ids = to_dev(inp.topk_ids, cuda_device)
        mask = inp.active_rank_mask
        res = comm.dispatch(to_dev(inp.hidden, cuda_device), ids, to_dev(inp.topk_weights, cuda_device),
                            runtime_max_tokens_per_rank=wl.runtime_max, active_rank_mask=mask)
        eo = fill_expert_outputs(comm, res.tokens_per_rank, cuda_device, caller=True)
        want = comm.combine(eo, active_rank_mask=mask)
        got = [torch.full((n, wl.hidden), float("nan"), dtype=torch.bfloat16, device=cuda_device)
               for n in inp.num_tokens]
        ret = combine_noalloc(wl.num_experts, wl.top_k, ids, eo, got, tokens_per_rank=res.tokens_per_rank,
                              active_rank_mask=mask)
        torch.cuda.synchronize(cuda_device)
        assert all(r is g for r, g in zip(ret, got))
        for s in range(wl.ep_size):
            np.testing.assert_array_equal(_bits(got[s]), _bits(want[s]), err_msg=f"output of rank {s}")
        with pytest.raises(ValueError):
            combine_noalloc(wl.num_experts, wl.top_k, ids, eo, got[:-1], tokens_per_rank=res.tokens_per_rank)
    finally:
        comm.destroy()
