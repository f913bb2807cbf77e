"""The hand-worked examples of tests/golden/ through the CUDA library."""
import json
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits_tensor(v, rows, H, device):
    return torch.full((rows, H), int(v, 16) - (0x10000 if int(v, 16) >= 0x8000 else 0),
                      dtype=torch.int16, device=device).view(torch.bfloat16)


@pytest.mark.parametrize("masked", [False, True])
def test_worked_example_on_gpu(cuda_device, masked):
    from combine_topk_ids_dest_gb300 import EpComm
    g = _load("worked_example.json")
    c = g["config"]
    ep, E, K, T = c["ep_size"], c["num_experts"], c["top_k"], c["tokens_per_rank"]
    H = 8  # one 16-byte bf16 vector per row
    comm = EpComm(ep, E, K, H, T, enable_rank_mask=True, device=cuda_device)
    try:
        ids = [torch.tensor(r, dtype=torch.int32, device=cuda_device).view(-1, K) for r in g["topk_ids"]]
        hid = [torch.randn(x.shape[0], H, device=cuda_device).to(torch.bfloat16) for x in ids]
        mask = comm.active_rank_mask([0] if masked else [0, 1])
        res = comm.dispatch(hid, ids, active_rank_mask=mask)
        exp = g["expected_recv_ids_mask_rank0_only" if masked else "expected_recv_ids"]
        for d in range(ep):
            assert res.topk_ids[d].cpu().tolist() == exp[f"dest{d}"]
        comm.combine(active_rank_mask=mask)
        for case in g["combine_cases"]:
            if ("mask" in case) != masked:
                continue
            s, t = case["token"]
            res = comm.dispatch(hid, ids, active_rank_mask=mask)
            bufs = comm.get_combine_input_buffer()
            for d, key in ((0, "eo_dest0"), (1, "eo_dest1")):
                bufs[d].copy_(_bits_tensor("0x7FC1", ep * T, H, cuda_device))  # NaN elsewhere
                bufs[d][s * T + t] = _bits_tensor(case[key], 1, H, cuda_device)[0]
            out = comm.combine(active_rank_mask=mask)
            got = out[s][t].view(torch.int16).cpu().numpy().view(np.uint16)
            assert (got == int(case["expected"], 16)).all(), case["what"]
    finally:
        comm.destroy()


def test_combine_rounding_on_gpu(cuda_device):
    from combine_topk_ids_dest_gb300 import EpComm
    g = _load("combine_rounding.json")
    c = g["config"]
    ep, E, K, T = c["ep_size"], c["num_experts"], c["top_k"], c["tokens_per_rank"]
    H = 8
    comm = EpComm(ep, E, K, H, T, device=cuda_device)
    try:
        ids = [torch.tensor([g["topk_ids"]], dtype=torch.int32, device=cuda_device)] + \
              [torch.zeros(0, K, dtype=torch.int32, device=cuda_device)] * (ep - 1)
        hid = [torch.zeros(x.shape[0], H, dtype=torch.bfloat16, device=cuda_device) for x in ids]
        for case in g["cases"]:
            comm.dispatch(hid, ids)
            eo = [_bits_tensor(v, ep * T, H, cuda_device) for v in case["eo"]]
            out = comm.combine(eo)
            got = out[0][0].view(torch.int16).cpu().numpy().view(np.uint16)
            assert (got == int(case["expected"], 16)).all(), case["what"]
    finally:
        comm.destroy()


@pytest.mark.parametrize("cdt", ["fp16", "fp32"])
def test_combine_rounding_f16_f32_on_gpu(cuda_device, cdt):
    from combine_topk_ids_dest_gb300 import EpComm
    g = _load("combine_rounding_f16_f32.json")
    c = g["config"]
    ep, E, K, T = c["ep_size"], c["num_experts"], c["top_k"], c["tokens_per_rank"]
    H = 8
    tdt, idt = (torch.float16, torch.int16) if cdt == "fp16" else (torch.float32, torch.int32)
    comm = EpComm(ep, E, K, H, T, device=cuda_device, combine_dtype=tdt)
    try:
        ids = [torch.tensor([g["topk_ids"]], dtype=torch.int32, device=cuda_device)] + \
              [torch.zeros(0, K, dtype=torch.int32, device=cuda_device)] * (ep - 1)
        hid = [torch.zeros(x.shape[0], H, dtype=torch.bfloat16, device=cuda_device) for x in ids]
        for case in (x for x in g["cases"] if x["dtype"] == cdt):
            comm.dispatch(hid, ids)
            eo = []
            for v in case["eo"]:
                b = int(v, 16)
                width = 16 if cdt == "fp16" else 32
                if b >= 1 << (width - 1):
                    b -= 1 << width
                eo.append(torch.full((ep * T, H), b, dtype=idt, device=cuda_device).view(tdt))
            out = comm.combine(eo)
            got = out[0][0].view(idt).cpu().numpy().view(np.uint16 if cdt == "fp16" else np.uint32)
            assert (got == int(case["expected"], 16)).all(), case["what"]
    finally:
        comm.destroy()
