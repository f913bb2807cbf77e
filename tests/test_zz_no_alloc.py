"""ep_combine_noalloc: the combine for callers that cannot allocate device memory.

Such callers (code inside an arena that owns all device memory after
start-up, plug-ins of a runtime that forbids allocations of their own) have no
ep_handle, whose workspace is an allocation; this entry point keeps its only
scratch in a fixed device array inside the library. The GPU test calls it
through the C ABI and checks its output bit for bit (the tolerance of every
combine test here) against ep_combine after ep_dispatch with the same ids,
mask and expert outputs, and against the oracle's combine of the same inputs,
on calls in a row whose routing differs, so anything one call leaves in the
shared scratch would show in the next. The third call's ids hold duplicates,
negative and out-of-range entries, which the entry point's own routing pass
must treat as the oracle does. After the first call (which looks up the
scratch array's address) the calls leave the device's free memory and
torch's allocation count unchanged.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from combine_topk_ids_dest_gb300 import EP_ERR_INVALID_ARG, EP_OK, EpComm, _lib
from combine_topk_ids_dest_gb300._lib import ptr_array
from ep_testutil import EO_SEED, bf16_bits, fill_expert_outputs, to_dev

ROUNDS = [
    # a wide round first: 16 ranks x 96 slots, two ranks masked off, one empty rank
    workloads.EpWorkload(name="noalloc_a", ep_size=16, num_experts=64, top_k=8, hidden=512,
                         dtype="bf16", capacity=96, runtime_max=96, counts=("uniform", 0, 96),
                         empty_ranks=(4,), dropped_ranks=(3, 9), seed=21),
    # then fewer slots, every rank active, duplicate ids
    workloads.EpWorkload(name="noalloc_b", ep_size=16, num_experts=64, top_k=8, hidden=512,
                         dtype="bf16", capacity=96, runtime_max=40, counts=("uniform", 1, 40),
                         ids="uniform_dups", dropped_ranks=(), seed=22),
    # ids with duplicates, -1, E and 2E+3 mixed in, one rank masked off
    workloads.EpWorkload(name="noalloc_c", ep_size=16, num_experts=64, top_k=8, hidden=512,
                         dtype="bf16", capacity=96, runtime_max=64, counts=("uniform", 0, 64),
                         ids="with_invalid", dropped_ranks=(7,), seed=23),
]


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _oracle_out(wl, inp, T):
    """The oracle's combine of the same ids and mask, over stand-in expert
    outputs drawn on the CPU from the same seeded generator."""
    rows = torch.arange(wl.ep_size * T)
    eo = [bf16_bits(workloads.expert_output_rows(EO_SEED, d, rows, wl.hidden)) for d in range(wl.ep_size)]
    return oracle.combine(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, T, inp.num_tokens, inp.topk_ids, eo,
                          mask_enabled=True, active_rank_mask=inp.active_rank_mask)


@pytest.mark.gpu
def test_noalloc_combine_matches_combine_and_oracle_on_calls_in_a_row(cuda_device):
    L = _lib.load()
    wl0 = ROUNDS[0]
    comm = EpComm(wl0.ep_size, wl0.num_experts, wl0.top_k, wl0.hidden, wl0.capacity,
                  enable_rank_mask=True, device=cuda_device)
    try:
        for i, wl in enumerate(ROUNDS):
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
            id_ptrs = ptr_array([x.data_ptr() for x in ids])
            eo_ptrs = ptr_array([e.data_ptr() for e in eo])
            out_ptrs = ptr_array([o.data_ptr() for o in got])
            torch.cuda.synchronize(cuda_device)
            alloc_before = torch.cuda.memory_allocated(cuda_device)
            free_before = torch.cuda.mem_get_info(cuda_device)[0]
            st = L.ep_combine_noalloc(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, T, counts, id_ptrs,
                                      mask, eo_ptrs, out_ptrs, ctypes.c_void_p(stream))
            assert st == EP_OK, L.ep_last_error()
            torch.cuda.synchronize(cuda_device)
            if i > 0:  # the first call may load the library's device code; later ones change nothing
                assert torch.cuda.memory_allocated(cuda_device) == alloc_before
                assert torch.cuda.mem_get_info(cuda_device)[0] == free_before
            want_oracle = _oracle_out(wl, inp, T)
            for s in range(wl.ep_size):
                np.testing.assert_array_equal(_bits(got[s]), _bits(want[s]),
                                              err_msg=f"{wl.name}: output of rank {s} vs ep_combine")
                np.testing.assert_array_equal(_bits(got[s]), want_oracle[s],
                                              err_msg=f"{wl.name}: output of rank {s} vs the oracle")
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
