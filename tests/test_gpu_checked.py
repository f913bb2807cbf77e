"""The checked build (EP_CHECKED=1, libep_gb300_checked.so): every global
access of the kernels is tested against the extent of its buffer; an access
outside is skipped and the call returns EP_ERR_DEVICE_CHECK.

test_gpu_suite_under_checked_build runs the parity, golden, eplb, fuzz,
graph, stream, device-count, stacked-form, full-size, programmatic-launch,
partitioned-group and no-alloc GPU tests in a child process that loads the
checked library. Every call there waits for its kernels and reads the check
record, so the suite passing shows that none of those runs touched memory
outside the buffers the C ABI gives each operand; the full-size workloads
include the 32-byte combine path that only combines of 192 MiB or more take.

The child also runs the two tests below, which show that the checks fire.
They use the checked build's test hook, which declares one access site's
buffers a row shorter than they are: the accesses to that last row are still
inside the real buffer (nothing unsafe is touched), but past the declared
end, so they must be reported, counted and skipped.
"""
import os
import re
import subprocess
import sys

import numpy as np
import pytest
import torch

import workloads
from combine_topk_ids_dest_gb300 import EpComm, _lib
from combine_topk_ids_dest_gb300._lib import EpError
from ep_testutil import expected_dests, fill_expert_outputs, to_dev

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITE = ["tests/test_gpu_parity.py", "tests/test_gpu_golden.py", "tests/test_gpu_eplb.py",
         "tests/test_gpu_fuzz.py", "tests/test_gpu_graph.py", "tests/test_gpu_streams.py",
         "tests/test_gpu_checked.py", "tests/test_gpu_device_counts.py", "tests/test_gpu_stacked.py",
         "tests/test_gpu_fullsize.py", "tests/test_gpu_pdl.py", "tests/test_gpu_partitions.py",
         "tests/test_zz_no_alloc.py"]

in_checked_child = pytest.mark.skipif(not _lib.checked(), reason="runs in the checked build's child process")

# 4 ranks, 16 slots each; rank 2 sends nothing, rank 3 fills all its slots.
WL = workloads.EpWorkload(name="checked_trim", ep_size=4, num_experts=16, top_k=4, hidden=512, dtype="bf16",
                          capacity=16, runtime_max=None, counts=("fixed", 16, 9, 0, 16), seed=41)
SENTINEL = 0x7FC1  # a bf16 NaN no combine produces here


@pytest.mark.gpu
@pytest.mark.skipif(_lib.checked(), reason="already the checked build")
def test_gpu_suite_under_checked_build(cuda_device):
    env = dict(os.environ, EP_GB300_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "gpu",
                        "-k", "not 1024-", *SUITE], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=1800)
    assert r.returncode == 0, r.stdout[-6000:] + r.stderr[-3000:]
    tail = r.stdout.strip().splitlines()[-1]
    # well over a hundred tests pass; the only one the child skips is this one
    passed = re.search(r"(\d+) passed", tail)
    assert passed and int(passed.group(1)) >= 100 and re.search(r"\b1 skipped\b", tail), tail


def _trim(site: str, nbytes: int):
    L = _lib.load()
    assert L.ep_checked_trim_extent(_lib.CHECK_SITES.index(site) if site else -1, nbytes) == _lib.EP_OK


def _round(comm, inp, device):
    return comm.dispatch(to_dev(inp.hidden, device), to_dev(inp.topk_ids, device),
                         to_dev(inp.topk_weights, device))


@pytest.mark.gpu
@in_checked_child
def test_trimmed_combine_output_is_reported_and_skipped(cuda_device):
    inp = workloads.make_inputs(WL)
    comm = EpComm(WL.ep_size, WL.num_experts, WL.top_k, WL.hidden, WL.capacity, device=cuda_device)
    try:
        res = _round(comm, inp, cuda_device)
        fill_expert_outputs(comm, res.tokens_per_rank, cuda_device)
        want = [x.cpu() for x in comm.combine()]

        _round(comm, inp, cuda_device)
        fill_expert_outputs(comm, res.tokens_per_rank, cuda_device)
        got = [torch.full((n, WL.hidden), SENTINEL, dtype=torch.int16, device=cuda_device).view(torch.bfloat16)
               for n in inp.num_tokens]
        row_bytes = WL.hidden * 2
        _trim("combine_out", row_bytes)
        try:
            with pytest.raises(EpError) as e:
                comm.combine(output=got)
        finally:
            _trim("", 0)
        assert e.value.status == _lib.EP_ERR_DEVICE_CHECK
        # each rank with tokens loses exactly its last row: 1024 bytes in 16-byte stores
        live = sum(1 for n in inp.num_tokens if n > 0)
        assert f"{live * row_bytes // 16} device accesses" in str(e.value), str(e.value)
        assert "combine: output row" in str(e.value)
        for s, n in enumerate(inp.num_tokens):
            g = got[s].cpu().view(torch.int16).numpy().view(np.uint16)
            w = want[s].view(torch.int16).numpy().view(np.uint16)
            if n == 0:
                continue
            np.testing.assert_array_equal(g[:n - 1], w[:n - 1], err_msg=f"rank {s}: rows inside the extent")
            assert (g[n - 1] == SENTINEL).all(), f"rank {s}: the skipped row was written"
        # the call's state change stands, and the next round is clean
        _round(comm, inp, cuda_device)
        fill_expert_outputs(comm, res.tokens_per_rank, cuda_device)
        again = comm.combine()
        for s in range(WL.ep_size):
            assert torch.equal(again[s].cpu().view(torch.int16), want[s].view(torch.int16))
    finally:
        comm.destroy()


@pytest.mark.gpu
@in_checked_child
def test_trimmed_receive_rows_are_reported_and_skipped(cuda_device):
    inp = workloads.make_inputs(WL)
    T = WL.capacity
    comm = EpComm(WL.ep_size, WL.num_experts, WL.top_k, WL.hidden, WL.capacity, device=cuda_device)
    try:
        row_bytes = WL.hidden * 2
        # clear every receive row, so a skipped store leaves zeros behind
        res = _round(comm, inp, cuda_device)
        for x in res.hidden_states:
            x.zero_()
        comm.combine()
        # the last slot of every receive region (source rank 3, token 15) lies
        # past the declared end; rank 3 has 16 tokens, so that token is live
        _trim("recv_hidden", row_bytes)
        try:
            with pytest.raises(EpError) as e:
                _round(comm, inp, cuda_device)
        finally:
            _trim("", 0)
        assert e.value.status == _lib.EP_ERR_DEVICE_CHECK
        dests = expected_dests(inp.topk_ids[3][T - 1].tolist(), WL.num_experts, WL.ep_size)
        # one 4 KB chunk per row, 32-byte stores (rows and sources are 32-byte aligned)
        assert f"{len(dests) * row_bytes // 32} device accesses" in str(e.value), str(e.value)
        assert "dispatch: receive hidden row" in str(e.value)
        src = inp.hidden[3].view(torch.int16)
        for d in range(WL.ep_size):
            h = res.hidden_states[d].cpu().view(torch.int16)
            if d in dests:
                assert (h[3 * T + T - 1] == 0).all(), f"rank {d}: the skipped row was written"
            for t in range(T - 1):
                if d in expected_dests(inp.topk_ids[3][t].tolist(), WL.num_experts, WL.ep_size):
                    assert torch.equal(h[3 * T + t], src[t]), f"rank {d}, token {t}"
        comm.combine()  # the dispatch's state change stood: it is pending
    finally:
        comm.destroy()
