"""Host-side rules of partitioned EP groups, on the CPU (no GPU needed):
ep_partition_describe gives each partition its ranks and the layout of its
workspace, and ep_partition_check accepts a set of descriptions only when
they form one group. Two gloo ranks then bring their descriptions together
the way one process per partition would (gather_partition_infos), and both
learn of a partition whose configuration differs."""
import ctypes
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from combine_topk_ids_dest_gb300 import EP_ERR_INVALID_ARG, EP_OK, _lib

BASE = dict(ep_size=16, num_experts=128, top_k=8, hidden=4096, max_tokens_per_rank=64, dtype=0,
            enable_rank_mask=1, scale_cols=-1, eplb_stats_max_bytes=64, combine_dtype=0, launch_flags=0,
            num_partitions=4, partition=0)
SPACING = 1 << 40  # fake, non-overlapping workspace addresses


def _cfg(**kw):
    d = dict(BASE)
    d.update(kw)
    return _lib.EpConfigC(*[d[f] for f, _ in _lib.EpConfigC._fields_])


def _size(cfg):
    n = ctypes.c_size_t(0)
    assert _lib.load().ep_workspace_size_ex(ctypes.byref(cfg), ctypes.byref(n)) == EP_OK
    return n.value


def _describe(p, **kw):
    cfg = _cfg(partition=p, **kw)
    info = _lib.EpPartitionInfoC()
    st = _lib.load().ep_partition_describe(ctypes.byref(cfg), ctypes.c_void_p(SPACING * (p + 1)), _size(cfg),
                                           ctypes.byref(info))
    assert st == EP_OK, _lib.load().ep_last_error()
    return info


def _check(infos):
    arr = (_lib.EpPartitionInfoC * len(infos))(*infos)
    L = _lib.load()
    return L.ep_partition_check(arr, len(infos)), L.ep_last_error().decode()


def test_describe_gives_each_partition_its_ranks():
    for p in range(4):
        x = _describe(p)
        assert (x.first_rank, x.num_ranks) == (4 * p, 4)
    whole = _size(_cfg(num_partitions=1))
    part = _size(_cfg())
    # a partition holds a quarter of the rank regions and routing state; the
    # gathered eplb statistics ([ep][bytes]) are whole in every partition
    assert part < whole // 3


def test_a_whole_group_passes():
    assert _check([_describe(p) for p in range(4)])[0] == EP_OK
    one = _lib.EpPartitionInfoC()
    cfg = _cfg(num_partitions=1)
    assert _lib.load().ep_partition_describe(ctypes.byref(cfg), ctypes.c_void_p(SPACING), _size(cfg),
                                             ctypes.byref(one)) == EP_OK
    assert (one.first_rank, one.num_ranks) == (0, 16)
    assert _check([one])[0] == EP_OK
    # launch flags are a local choice of each partition
    assert _check([_describe(p, launch_flags=p % 2) for p in range(4)])[0] == EP_OK


@pytest.mark.parametrize("mutate,msg", [
    (lambda xs: xs[:3], "3 descriptions for a group of 4"),
    (lambda xs: [xs[1], xs[0], xs[2], xs[3]], "description 0 is of partition 1"),
    (lambda xs: xs[:2] + [_describe(2, hidden=2048)] + xs[3:], "partition 2 has another hidden"),
    (lambda xs: xs[:3] + [_describe(3, enable_rank_mask=0)], "another enable_rank_mask"),
    (lambda xs: xs[:1] + [_describe(1, max_tokens_per_rank=32)] + xs[2:], "another max_tokens_per_rank"),
])
def test_a_broken_group_is_refused(mutate, msg):
    st, err = _check(mutate([_describe(p) for p in range(4)]))
    assert st == EP_ERR_INVALID_ARG and msg in err, err


def test_layout_size_alignment_and_overlap_are_checked():
    xs = [_describe(p) for p in range(4)]
    xs[2].off_combine_in += 256
    assert "layout differs" in _check(xs)[1]
    xs = [_describe(p) for p in range(4)]
    xs[1].workspace_bytes -= 1
    assert "workspace has" in _check(xs)[1]
    xs = [_describe(p) for p in range(4)]
    xs[3].workspace = SPACING * 4 + 16
    assert "not 256-byte aligned" in _check(xs)[1]
    xs = [_describe(p) for p in range(4)]
    xs[3].workspace = xs[2].workspace + 256
    assert "overlap" in _check(xs)[1]


def test_partitions_must_divide_the_group():
    n = ctypes.c_size_t(0)
    L = _lib.load()
    assert L.ep_workspace_size_ex(ctypes.byref(_cfg(num_partitions=3)), ctypes.byref(n)) == EP_ERR_INVALID_ARG
    assert L.ep_workspace_size_ex(ctypes.byref(_cfg(partition=4)), ctypes.byref(n)) == EP_ERR_INVALID_ARG


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, hidden_of_rank1, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from combine_topk_ids_dest_gb300 import EpError, gather_partition_infos
        kw = dict(num_partitions=world)
        if rank == 1:
            kw["hidden"] = hidden_of_rank1
        mine = _describe(rank, **kw)
        try:
            infos = gather_partition_infos(mine)
            q.put((rank, "ok", [(x.config.partition, x.first_rank, x.num_ranks, x.workspace) for x in infos]))
        except EpError as e:
            q.put((rank, "error", str(e)))
    finally:
        dist.destroy_process_group()


def _run_two(hidden_of_rank1):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, hidden_of_rank1, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


def test_two_gloo_ranks_gather_their_partitions():
    res = _run_two(hidden_of_rank1=BASE["hidden"])
    for rank, kind, infos in res:
        assert kind == "ok"
        assert infos == [(0, 0, 8, SPACING), (1, 8, 8, 2 * SPACING)]  # both see the same group, in order


def test_two_gloo_ranks_both_refuse_a_mismatched_partition():
    res = _run_two(hidden_of_rank1=2048)
    for rank, kind, msg in res:
        assert kind == "error" and "another hidden" in msg, msg
