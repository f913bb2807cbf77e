"""GPU parity: the CUDA library (through EpComm and the C ABI) against the
oracle, element by element, bit for bit.

Receive id rows are compared everywhere; hidden, scale and weight rows where
the oracle routes the token (elsewhere the method leaves them unspecified);
combine outputs everywhere. Workloads: the five EP configurations shrunk to
oracle-friendly sizes (same ep/E/K, id laws, masks, dtypes) plus edge cases.
"""
import numpy as np
import pytest
import torch

import workloads
from ep_testutil import assert_round_equal, gpu_round, oracle_round, small

pytestmark = pytest.mark.gpu


def _check(wl, device, **kw):
    inp = workloads.make_inputs(wl)
    got = gpu_round(inp, device, **kw)
    disp, out = oracle_round(inp, special=kw.get("special", False))
    assert_round_equal(inp, got, disp, out)
    return inp, got


def test_tiny_full_size(cuda_device):
    _check(workloads.WORKLOADS["tiny"], cuda_device)


@pytest.mark.parametrize("name", ["mixtral_decode", "dsv3_decode", "dsv3_prefill", "qwen3_mask"])
@pytest.mark.parametrize("hidden", [256, 1024])
def test_shrunk_workloads(cuda_device, name, hidden):
    # several 4 KB dispatch chunks per row at hidden=1024 fp8/bf16, a ragged
    # last chunk at 256 bf16 (512 B rows)
    _check(small(workloads.WORKLOADS[name], hidden=hidden, tokens=40), cuda_device)


@pytest.mark.parametrize("name", sorted(workloads.GEOMETRIES))
def test_shrunk_geometries(cuda_device, name):
    # the further bandwidth geometries (ep 8..64, top_k 4..32, bf16/fp8) at oracle-friendly sizes
    _check(small(workloads.GEOMETRIES[name], hidden=512, tokens=12), cuda_device)


def test_mixtral_full_hidden_small_tokens(cuda_device):
    _check(small(workloads.WORKLOADS["mixtral_decode"], hidden=4096, tokens=20), cuda_device)


def test_dsv3_full_hidden_small_tokens(cuda_device):
    _check(small(workloads.WORKLOADS["dsv3_prefill"], hidden=7168, tokens=6), cuda_device)


BASE = workloads.EpWorkload(name="edge", ep_size=4, num_experts=16, top_k=4, hidden=256, dtype="bf16",
                            capacity=12, runtime_max=None, counts=("uniform", 0, 12), seed=11)


@pytest.mark.parametrize("variant", [
    dict(ids="with_invalid"),                              # -1, E, 2E+3 ids mixed in
    dict(ids="uniform_dups"),                              # repeated ids in one token
    dict(top_k=1, num_experts=4),                          # K=1, one expert per rank
    dict(top_k=2),                                         # scalar id-plane path (K % 4 != 0)
    dict(top_k=3, ids="uniform_dups"),
    dict(top_k=32, num_experts=64),                        # largest top_k
    dict(ep_size=1, num_experts=8),                        # a single rank
    dict(ep_size=64, num_experts=64, top_k=8, capacity=3, counts=("uniform", 0, 3)),  # high mask word
    dict(ep_size=64, num_experts=128, top_k=8, capacity=3, counts=("uniform", 0, 3),
         dropped_ranks=(0, 31, 32, 63)),
    dict(runtime_max=7, counts=("uniform", 0, 7)),         # tokens_per_rank below capacity
    dict(runtime_max=0, counts=("fixed", 0, 0, 0, 0)),     # zero tokens per rank
    dict(counts=("fixed", 0, 0, 0, 0)),                    # all ranks empty, T = capacity
    dict(counts=("fixed", 12, 0, 12, 0)),
    dict(dropped_ranks=()),                                # masking on, every rank active
    dict(dropped_ranks=(0, 1, 2, 3)),                      # mask drops every rank
    dict(dropped_ranks=(1,)),
    dict(dropped_ranks=(0, 2, 3)),
    dict(weights=False),                                   # no weights
    dict(dtype="fp8_e4m3", hidden=256, scales=True),
    dict(dtype="fp8_e4m3", hidden=272, scales=False),      # fp8 row not a multiple of 128
    dict(dtype="bf16", hidden=384, scales=True),           # scales with a bf16 payload
    dict(dtype="fp16", scales=True),                       # fp16 payload, hidden/128 scales
    dict(dtype="fp32", hidden=264),                        # fp32 payload (1056-byte rows)
    dict(dtype="bf16", scales=True, scale_cols_override=7),  # odd scale width
    dict(dtype="fp8_e4m3", hidden=512, scales=True, scale_cols_override=16),  # 32-column groups
    dict(dtype="fp32", hidden=16384, capacity=3, counts=("uniform", 0, 3)),  # 64 KB rows: 16 chunks
    dict(ep_size=64, num_experts=128, top_k=32, capacity=2, counts=("full",)),  # widest fan-out
    dict(ep_size=64, num_experts=64, top_k=32, capacity=2, counts=("full",), ids="uniform_dups",
         dropped_ranks=tuple(range(0, 64, 3))),
    dict(combine_dtype="fp16"),                            # fp16 expert outputs and results
    dict(combine_dtype="fp32", hidden=264),                # fp32 combine, 1056-byte rows
    dict(combine_dtype="fp32", dtype="fp8_e4m3", hidden=512, scales=True, dropped_ranks=(1,)),
    dict(combine_dtype="fp16", hidden=4104, capacity=4, counts=("uniform", 0, 4)),  # ragged blocks
    dict(hidden=8),                                        # one 16-byte vector per row
    dict(hidden=264),                                      # combine: 33 vectors, ragged block
])
def test_edge_cases(cuda_device, variant):
    _check(BASE.replace(**variant), cuda_device)


@pytest.mark.parametrize("cdt", ["bf16", "fp16", "fp32"])
def test_subnormal_and_zero_expert_outputs(cuda_device, cdt):
    _check(BASE.replace(hidden=512, combine_dtype=cdt), cuda_device, special=True)


def test_caller_owned_expert_outputs(cuda_device):
    _check(BASE.replace(hidden=512, dropped_ranks=(2,)), cuda_device, caller_eo=True)


def test_rounds_reuse_handle_with_changing_T(cuda_device):
    """One handle, several rounds with different tokens_per_rank, masks and
    counts: every round matches the oracle (no state leaks between rounds)."""
    from combine_topk_ids_dest_gb300 import EpComm
    wl0 = BASE.replace(capacity=16, dropped_ranks=(3,))
    comm = EpComm(wl0.ep_size, wl0.num_experts, wl0.top_k, wl0.hidden, wl0.capacity,
                  enable_rank_mask=True, device=cuda_device)
    try:
        for i, (rt, drop) in enumerate([(16, (3,)), (5, ()), (9, (0, 1)), (16, (3,)), (1, (2,))]):
            wl = wl0.replace(runtime_max=rt, counts=("uniform", 0, rt), dropped_ranks=drop, seed=100 + i)
            inp = workloads.make_inputs(wl)
            got = gpu_round(inp, cuda_device, comm=comm)
            disp, out = oracle_round(inp)
            assert_round_equal(inp, got, disp, out)
    finally:
        comm.destroy()


def test_packed_fp4_payload_with_byte_scales(cuda_device):
    """A quantised payload of any byte-aligned format travels as opaque bytes
    (MoEEpCommunication.dispatch: hidden_states "unquantized or quantized",
    [local_num_tokens, *]): here packed 4-bit values (two per byte, 7168 values
    = 3584 bytes per row, passed as an 8-bit payload) with one 8-bit scale per
    16 values (448 bytes per row, passed as 112 fp32 words). Scale bytes stay
    below 0x7F, so no 32-bit word is a NaN. Receive rows must equal the
    source bytes exactly, and the ids and weights the oracle's."""
    import torch

    import oracle
    from combine_topk_ids_dest_gb300 import EpComm
    from ep_testutil import INV, raw_bytes, to_dev
    values, group = 7168, 16
    row_bytes, scale_bytes = values // 2, values // group
    wl = workloads.EpWorkload(name="fp4_bytes", ep_size=8, num_experts=64, top_k=8, hidden=row_bytes,
                              dtype="fp8_e4m3", capacity=24, runtime_max=None, counts=("uniform", 0, 24),
                              dropped_ranks=(6,), seed=81)
    inp = workloads.make_inputs(wl)
    g = torch.Generator().manual_seed(82)
    rows = [torch.randint(0, 256, (n, row_bytes), generator=g, dtype=torch.uint8) for n in inp.num_tokens]
    scales = [torch.randint(0, 0x7F, (n, scale_bytes), generator=g, dtype=torch.uint8) for n in inp.num_tokens]
    hid = [r.view(torch.float8_e4m3fn) for r in rows]
    scl = [s.view(torch.float32) for s in scales]  # [n, 112] words of 4 scale bytes
    comm = EpComm(wl.ep_size, wl.num_experts, wl.top_k, row_bytes, wl.capacity, dtype=torch.float8_e4m3fn,
                  enable_rank_mask=True, device=cuda_device, scale_cols=scale_bytes // 4)
    try:
        mask = inp.active_rank_mask
        res = comm.dispatch(to_dev(hid, cuda_device), to_dev(inp.topk_ids, cuda_device),
                            to_dev(inp.topk_weights, cuda_device), hidden_states_scale=to_dev(scl, cuda_device),
                            active_rank_mask=mask)
        T = res.tokens_per_rank
        want = oracle.dispatch(wl.ep_size, wl.num_experts, wl.top_k, T, inp.num_tokens, rows, inp.topk_ids,
                               scale=[s.view(torch.float32) for s in scales], topk_weights=inp.topk_weights,
                               mask_enabled=True, active_rank_mask=mask, row_bytes=row_bytes,
                               scale_cols=scale_bytes // 4)
        rows_id = torch.arange(wl.ep_size * T, device=cuda_device)
        for d, buf in enumerate(comm.get_combine_input_buffer()):
            buf.copy_(workloads.expert_output_rows(5, d, rows_id, row_bytes, device=cuda_device))
        comm.combine(active_rank_mask=mask)
        torch.cuda.synchronize(cuda_device)
        for d in range(wl.ep_size):
            np.testing.assert_array_equal(res.topk_ids[d].cpu().numpy(), want.recv_ids[d])
            valid = (want.recv_ids[d] != INV).any(axis=1)
            np.testing.assert_array_equal(raw_bytes(res.hidden_states[d].cpu())[valid], want.recv_hidden[d][valid])
            np.testing.assert_array_equal(res.hidden_states_scale[d].cpu().numpy()[valid].view(np.uint32),
                                          want.recv_scale[d][valid].view(np.uint32))
            np.testing.assert_array_equal(res.topk_weights[d].cpu().numpy()[valid].view(np.uint32),
                                          want.recv_weights[d][valid].view(np.uint32))
    finally:
        comm.destroy()
