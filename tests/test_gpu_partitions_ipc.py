"""A partitioned group with one process per partition, all on one GPU.

Each process creates its partition and connects with the others over a gloo
group: either with EpComm.connect_across_processes (workspaces shared as CUDA
IPC handles inside the gathered objects) or by hand, handing its workspace to
the others as a CUDA tensor through torch.multiprocessing queues (the memory
is mapped into each receiving process) and then gather_partition_infos with
the peers' workspaces at the addresses mapped here. Each process then dispatches its own ranks' tokens
straight into the other processes' receive buffers, writes its ranks' stand-in
expert outputs, and combines its own tokens from every process's buffers.
The phases are ordered on the host (stream synchronisation, then a gloo
barrier); no kernel waits on another. Every process compares what it holds
with the oracle, bit for bit.
"""
import os
import socket
import traceback
from datetime import timedelta

import pytest
import torch

pytestmark = pytest.mark.gpu

WL = dict(name="ipc", ep_size=8, num_experts=32, top_k=4, hidden=1024, dtype="fp8_e4m3", scales=True,
          capacity=24, runtime_max=20, counts=("uniform", 0, 20), dropped_ranks=(5,), seed=91)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _child(rank, world, port, queues, results, by_hand):
    import numpy as np
    import torch.distributed as dist

    import oracle
    import workloads
    from combine_topk_ids_dest_gb300 import EpComm, gather_partition_infos
    from ep_testutil import EO_SEED, bf16_bits, raw_bytes
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=timedelta(seconds=120))
    comm = None
    try:
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        wl = workloads.EpWorkload(**WL)
        inp = workloads.make_inputs(wl)
        comm = EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, dtype=wl.torch_dtype,
                      enable_rank_mask=True, device=dev, num_partitions=world, partition=rank)
        if by_hand:
            for h in range(world):  # this partition's workspace, mapped into every other process
                if h != rank:
                    queues[h].put((rank, comm._ws))
            peers = dict(queues[rank].get(timeout=120) for _ in range(world - 1))
            infos = gather_partition_infos(comm.partition_info(),
                                           addresses={h: t.data_ptr() for h, t in peers.items()})
            comm.connect(infos)
        else:
            comm.connect_across_processes()
        lo, hi = comm.first_rank, comm.first_rank + comm.num_ranks
        mask = inp.active_rank_mask
        res = comm.dispatch([x.to(dev) for x in inp.hidden[lo:hi]], [x.to(dev) for x in inp.topk_ids[lo:hi]],
                            [x.to(dev) for x in inp.topk_weights[lo:hi]],
                            hidden_states_scale=[x.to(dev) for x in inp.scale[lo:hi]],
                            runtime_max_tokens_per_rank=wl.runtime_max, active_rank_mask=mask)
        torch.cuda.synchronize(dev)
        dist.barrier()  # every process's dispatch has landed in every receive buffer
        T = res.tokens_per_rank
        rows = torch.arange(wl.ep_size * T, device=dev)
        for j, buf in enumerate(comm.get_combine_input_buffer()):
            buf.copy_(workloads.expert_output_rows(EO_SEED, lo + j, rows, wl.hidden, device=dev))
        torch.cuda.synchronize(dev)
        dist.barrier()  # every rank's expert outputs are written
        out = comm.combine(active_rank_mask=mask)
        torch.cuda.synchronize(dev)

        want = oracle.dispatch(wl.ep_size, wl.num_experts, wl.top_k, T, inp.num_tokens, inp.hidden, inp.topk_ids,
                               scale=inp.scale, topk_weights=inp.topk_weights, mask_enabled=True,
                               active_rank_mask=mask, row_bytes=wl.hidden, scale_cols=wl.scale_cols)
        rows_h = torch.arange(wl.ep_size * T)
        eo = [bf16_bits(workloads.expert_output_rows(EO_SEED, d, rows_h, wl.hidden)) for d in range(wl.ep_size)]
        want_out = oracle.combine(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, T, inp.num_tokens,
                                  inp.topk_ids, eo, mask_enabled=True, active_rank_mask=mask)
        for j in range(comm.num_ranks):
            d = lo + j
            np.testing.assert_array_equal(res.topk_ids[j].cpu().numpy(), want.recv_ids[d], err_msg=f"ids of rank {d}")
            valid = (want.recv_ids[d] != -1).any(axis=1)
            np.testing.assert_array_equal(raw_bytes(res.hidden_states[j].cpu())[valid], want.recv_hidden[d][valid],
                                          err_msg=f"hidden rows of rank {d}")
            np.testing.assert_array_equal(res.hidden_states_scale[j].cpu().numpy()[valid],
                                          want.recv_scale[d][valid], err_msg=f"scale rows of rank {d}")
            np.testing.assert_array_equal(bf16_bits(out[j].cpu()), want_out[d], err_msg=f"combine output of rank {d}")
        results.put((rank, "ok", int(valid.sum())))
    except Exception:
        results.put((rank, "error", traceback.format_exc()[-3000:]))
    finally:
        try:
            dist.barrier()  # peers stop using this process's workspace before it is freed
        except Exception:
            pass
        if comm is not None:
            comm.destroy()
        dist.destroy_process_group()


@pytest.mark.parametrize("world,by_hand", [(2, True), (4, True), (2, False), (4, False)])
def test_one_process_per_partition(cuda_device, world, by_hand):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    queues = [ctx.Queue() for _ in range(world)]
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_child, args=(r, world, port, queues, results, by_hand)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        got = sorted(results.get(timeout=300) for _ in range(world))
    finally:
        for p in procs:
            p.join(timeout=120)
            if p.is_alive():
                p.kill()
                p.join()
    for rank, kind, detail in got:
        assert kind == "ok", f"process {rank}:\n{detail}"
    assert all(p.exitcode == 0 for p in procs)
