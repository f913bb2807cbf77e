"""Static shapes and CUDA graphs (MoEEpCommunication.dispatch: without
runtime_max_tokens_per_rank the shapes stay at capacity, which is what graph
capture needs).

One dispatch and one combine are captured into a single CUDA graph over
fixed, capacity-sized buffers; each replay after writing new inputs into those
buffers must equal the oracle on the new inputs. Padding tokens inside the
static shapes are rows whose ids are all invalid: they route nowhere and
combine to +0.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from combine_topk_ids_dest_gb300 import EpComm
from ep_testutil import EO_SEED, INV, bf16_bits, raw_bytes

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pdl", [False, True], ids=["stream_order", "pdl"])
def test_captured_round_replays_with_new_inputs(cuda_device, pdl):
    ep, E, K, H, C = 8, 64, 6, 512, 24
    dev = cuda_device
    comm = EpComm(ep, E, K, H, C, dtype=torch.float8_e4m3fn, enable_rank_mask=True, device=dev, pdl=pdl)
    try:
        hid = [torch.zeros(C, H, dtype=torch.float8_e4m3fn, device=dev) for _ in range(ep)]
        scl = [torch.ones(C, H // 128, device=dev) for _ in range(ep)]
        ids = [torch.full((C, K), INV, dtype=torch.int32, device=dev) for _ in range(ep)]
        wts = [torch.zeros(C, K, device=dev) for _ in range(ep)]
        eo = [torch.zeros(ep * C, H, dtype=torch.bfloat16, device=dev) for _ in range(ep)]
        out = [torch.empty(C, H, dtype=torch.bfloat16, device=dev) for _ in range(ep)]
        mask = comm.active_rank_mask([r for r in range(ep) if r != 5])
        state = {}

        def round_():
            state["res"] = comm.dispatch(hid, ids, wts, hidden_states_scale=scl, active_rank_mask=mask)
            comm.combine(eo, output=out, active_rank_mask=mask)

        round_()  # eager once (first-use set-up happens outside the capture)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            round_()
        res = state["res"]

        for it in range(3):
            wl = workloads.EpWorkload(name="graph", ep_size=ep, num_experts=E, top_k=K, hidden=H,
                                      dtype="fp8_e4m3", scales=True, capacity=C, runtime_max=None,
                                      counts=("uniform", 0, C), dropped_ranks=(5,), seed=40 + it)
            inp = workloads.make_inputs(wl)
            # pad every rank to C tokens: padding rows carry only invalid ids
            full_ids = []
            for s in range(ep):
                n = inp.num_tokens[s]
                pad_ids = torch.full((C, K), INV, dtype=torch.int32)
                pad_ids[:n] = inp.topk_ids[s]
                full_ids.append(pad_ids)
                hid[s][:n].copy_(inp.hidden[s].to(dev))
                scl[s][:n].copy_(inp.scale[s].to(dev))
                wts[s][:n].copy_(inp.topk_weights[s].to(dev))
                ids[s].copy_(pad_ids.to(dev))
            rows = torch.arange(ep * C)
            eo_host = [workloads.expert_output_rows(EO_SEED + it, d, rows, H) for d in range(ep)]
            for d in range(ep):
                eo[d].copy_(eo_host[d].to(dev))
            g.replay()
            torch.cuda.synchronize(dev)

            full_hidden = [torch.cat([inp.hidden[s].view(torch.uint8),
                                      torch.zeros(C - inp.num_tokens[s], H, dtype=torch.uint8)])
                           for s in range(ep)]
            want = oracle.dispatch(ep, E, K, C, [C] * ep, full_hidden, full_ids, mask_enabled=True,
                                   active_rank_mask=int(mask.item()), payload=True, row_bytes=H)
            want_out = oracle.combine(ep, E, K, H, C, [C] * ep, full_ids, [bf16_bits(x) for x in eo_host],
                                      mask_enabled=True, active_rank_mask=int(mask.item()))
            for d in range(ep):
                np.testing.assert_array_equal(res.topk_ids[d].cpu().numpy(), want.recv_ids[d])
                valid = (want.recv_ids[d] != INV).any(axis=1)
                np.testing.assert_array_equal(raw_bytes(res.hidden_states[d].cpu())[valid],
                                              want.recv_hidden[d][valid])
            for s in range(ep):
                got = bf16_bits(out[s].cpu())
                np.testing.assert_array_equal(got, want_out[s])
                assert (got[inp.num_tokens[s]:] == 0).all()  # padding tokens combine to +0
    finally:
        comm.destroy()
