"""Independent handles on independent streams: two communicators with
different geometries run dispatch and combine concurrently on two non-default
streams; each must match the oracle (no shared state on the main path). Also
the binding's argument checks for tensors of the wrong kind."""
import numpy as np
import pytest
import torch

import workloads
from combine_topk_ids_dest_gb300 import EpComm
from ep_testutil import EO_SEED, INV, bf16_bits, oracle_round, raw_bytes, to_dev

pytestmark = pytest.mark.gpu


def test_two_handles_on_two_streams(cuda_device):
    wls = [workloads.EpWorkload(name="sa", ep_size=8, num_experts=32, top_k=4, hidden=1024, dtype="bf16",
                                capacity=64, runtime_max=None, counts=("uniform", 0, 64), seed=71),
           workloads.EpWorkload(name="sb", ep_size=16, num_experts=64, top_k=8, hidden=512,
                                dtype="fp8_e4m3", scales=True, capacity=48, runtime_max=40,
                                counts=("uniform", 0, 40), dropped_ranks=(2, 7), seed=72)]
    inps = [workloads.make_inputs(wl) for wl in wls]
    comms = [EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, dtype=wl.torch_dtype,
                    enable_rank_mask=wl.enable_rank_mask, device=cuda_device) for wl in wls]
    streams = [torch.cuda.Stream(cuda_device) for _ in wls]
    try:
        dev_in = [(to_dev(i.hidden, cuda_device), to_dev(i.topk_ids, cuda_device),
                   to_dev(i.topk_weights, cuda_device), to_dev(i.scale, cuda_device)) for i in inps]
        eos = []
        for wl in wls:
            rows = torch.arange(wl.ep_size * wl.tokens_per_rank)
            eos.append([workloads.expert_output_rows(EO_SEED, d, rows, wl.hidden).to(cuda_device)
                        for d in range(wl.ep_size)])
        torch.cuda.synchronize(cuda_device)
        results, outs = [], []
        for _ in range(3):  # interleave the two handles' calls on their streams
            results, outs = [None, None], [None, None]
            for i, (wl, inp, comm, st) in enumerate(zip(wls, inps, comms, streams)):
                with torch.cuda.stream(st):
                    h, ids, w, sc = dev_in[i]
                    mask = inp.active_rank_mask if wl.enable_rank_mask else None
                    results[i] = comm.dispatch(h, ids, w, hidden_states_scale=sc,
                                               runtime_max_tokens_per_rank=wl.runtime_max,
                                               active_rank_mask=mask)
            for i, (wl, inp, comm, st) in enumerate(zip(wls, inps, comms, streams)):
                with torch.cuda.stream(st):
                    mask = inp.active_rank_mask if wl.enable_rank_mask else None
                    outs[i] = comm.combine(eos[i], active_rank_mask=mask)
        torch.cuda.synchronize(cuda_device)
        for i, inp in enumerate(inps):
            disp, out = oracle_round(inp)
            res = results[i]
            for d in range(inp.wl.ep_size):
                np.testing.assert_array_equal(res.topk_ids[d].cpu().numpy(), disp.recv_ids[d])
                valid = (disp.recv_ids[d] != INV).any(axis=1)
                np.testing.assert_array_equal(raw_bytes(res.hidden_states[d].cpu())[valid],
                                              disp.recv_hidden[d][valid])
            for s in range(inp.wl.ep_size):
                np.testing.assert_array_equal(bf16_bits(outs[i][s].cpu()), out[s])
    finally:
        for c in comms:
            c.destroy()


def test_handles_used_from_two_host_threads(cuda_device):
    """Two host threads, each with its own handle and stream, run rounds at the
    same time (ctypes calls release the interpreter lock, so the library's
    host code runs concurrently); each thread's last round matches the oracle."""
    import threading
    wls = [workloads.EpWorkload(name="ta", ep_size=4, num_experts=16, top_k=2, hidden=2048, dtype="bf16",
                                capacity=96, runtime_max=None, counts=("uniform", 0, 96), seed=73),
           workloads.EpWorkload(name="tb", ep_size=32, num_experts=128, top_k=8, hidden=256, dtype="bf16",
                                capacity=24, runtime_max=None, counts=("uniform", 0, 24),
                                dropped_ranks=(5,), seed=74)]
    inps = [workloads.make_inputs(wl) for wl in wls]
    got, errors = [None, None], []

    def worker(i):
        try:
            wl, inp = wls[i], inps[i]
            comm = EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity,
                          enable_rank_mask=wl.enable_rank_mask, device=cuda_device)
            st = torch.cuda.Stream(cuda_device)
            try:
                with torch.cuda.stream(st):
                    h, ids, w = (to_dev(inp.hidden, cuda_device), to_dev(inp.topk_ids, cuda_device),
                                 to_dev(inp.topk_weights, cuda_device))
                    rows = torch.arange(wl.ep_size * wl.tokens_per_rank)
                    eo = [workloads.expert_output_rows(EO_SEED, d, rows, wl.hidden).to(cuda_device)
                          for d in range(wl.ep_size)]
                    mask = inp.active_rank_mask if wl.enable_rank_mask else None
                    for _ in range(5):
                        res = comm.dispatch(h, ids, w, active_rank_mask=mask)
                        out = comm.combine(eo, active_rank_mask=mask)
                    ids_out = [x.cpu() for x in res.topk_ids]
                    got[i] = (ids_out, [x.cpu() for x in out])
                st.synchronize()
            finally:
                comm.destroy()
        except Exception as e:  # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    assert not errors, errors
    for i, inp in enumerate(inps):
        disp, out = oracle_round(inp)
        ids_out, outs = got[i]
        for d in range(inp.wl.ep_size):
            np.testing.assert_array_equal(ids_out[d].numpy(), disp.recv_ids[d])
        for s in range(inp.wl.ep_size):
            np.testing.assert_array_equal(bf16_bits(outs[s]), out[s])


def test_hidden_rows_of_any_trailing_shape(cuda_device):
    """hidden_states[s] as [n, 4, H/4] (the pages' [local_num_tokens, *]) gives
    exactly what [n, H] gives; a wrong element count per row is refused."""
    wl = workloads.EpWorkload(name="shape", ep_size=4, num_experts=8, top_k=2, hidden=256, dtype="bf16",
                              capacity=16, runtime_max=None, counts=("uniform", 0, 16), seed=76)
    inp = workloads.make_inputs(wl)
    comms = [EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, device=cuda_device)
             for _ in range(2)]
    try:
        h2 = to_dev(inp.hidden, cuda_device)
        h3 = [x.view(x.shape[0], 4, wl.hidden // 4) for x in h2]
        ids = to_dev(inp.topk_ids, cuda_device)
        a = comms[0].dispatch(h3, ids)
        b = comms[1].dispatch(h2, ids)
        torch.cuda.synchronize(cuda_device)
        for d in range(wl.ep_size):
            assert torch.equal(a.topk_ids[d], b.topk_ids[d])
            valid = (b.topk_ids[d] != INV).any(dim=1)
            assert torch.equal(a.hidden_states[d][valid].view(torch.int16), b.hidden_states[d][valid].view(torch.int16))
        for c in comms:
            c.combine()
        bad = [x.view(x.shape[0], 4, wl.hidden // 4)[:, :3] for x in h2]  # 3/4 of each row
        with pytest.raises(ValueError):
            comms[0].dispatch(bad, ids)
    finally:
        for c in comms:
            c.destroy()


def test_binding_rejects_wrong_tensors(cuda_device):
    comm = EpComm(2, 4, 2, 64, 8, device=cuda_device)
    try:
        ids = [torch.zeros(3, 2, dtype=torch.int32, device=cuda_device)] * 2
        good = [torch.zeros(3, 64, dtype=torch.bfloat16, device=cuda_device)] * 2
        bad_cases = [
            [torch.zeros(3, 64, dtype=torch.float16, device=cuda_device)] * 2,  # wrong dtype
            [torch.zeros(3, 64, dtype=torch.bfloat16)] * 2,                     # on the CPU
            [torch.zeros(64, 3, dtype=torch.bfloat16, device=cuda_device).t()] * 2,  # not contiguous
            [torch.zeros(3, 32, dtype=torch.bfloat16, device=cuda_device)] * 2,  # wrong width
            good[:1],                                                          # one rank missing
        ]
        for hid in bad_cases:
            with pytest.raises(ValueError):
                comm.dispatch(hid, ids)
        with pytest.raises(ValueError):
            comm.dispatch(good, [torch.zeros(3, 2, dtype=torch.int64, device=cuda_device)] * 2)
        comm.dispatch(good, ids)  # the handle is still usable
        with pytest.raises(ValueError):
            comm.combine([torch.zeros(16, 64, dtype=torch.float32, device=cuda_device)] * 2)
        comm.combine()
    finally:
        comm.destroy()
