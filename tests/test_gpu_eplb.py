"""eplb_local_stats all-gather through the C ABI (MoEEpCommunication.dispatch,
parameter eplb_local_stats): the gathered buffer equals the oracle's, in the
same dispatch launch, for several element types and with zero-token steps;
misuse is rejected before launch."""
import numpy as np
import pytest
import torch

import oracle
from combine_topk_ids_dest_gb300 import EP_ERR_INVALID_ARG, EpComm, EpError

pytestmark = pytest.mark.gpu

EP, E, K, H, C = 8, 32, 4, 256, 16


def _inputs(dev, counts, seed=0):
    g = torch.Generator().manual_seed(seed)
    hid = [torch.randn(n, H, generator=g).to(torch.bfloat16).to(dev) for n in counts]
    ids = [torch.randint(0, E, (n, K), generator=g, dtype=torch.int32).to(dev) for n in counts]
    return hid, ids


@pytest.mark.parametrize("dtype,shape", [(torch.int32, (E // EP,)), (torch.int64, (E,)),
                                         (torch.float32, (2, E // EP))])
@pytest.mark.parametrize("counts", [(16, 3, 0, 9, 16, 1, 0, 5), (0,) * EP])
def test_eplb_gather_matches_oracle(cuda_device, dtype, shape, counts):
    comm = EpComm(EP, E, K, H, C, device=cuda_device, eplb_stats_max_bytes=1024)
    try:
        g = torch.Generator().manual_seed(3)
        local = [(torch.randint(0, 1 << 20, shape, generator=g)).to(dtype) for _ in range(EP)]
        hid, ids = _inputs(cuda_device, counts)
        res = comm.dispatch(hid, ids, eplb_local_stats=[x.to(cuda_device) for x in local])
        comm.combine()
        torch.cuda.synchronize(cuda_device)
        assert res.eplb_global_stats.shape == (EP,) + shape and res.eplb_global_stats.dtype == dtype
        got = res.eplb_global_stats.cpu().contiguous().view(torch.uint8).numpy().reshape(EP, -1)
        np.testing.assert_array_equal(got, oracle.eplb_gather(local))
    finally:
        comm.destroy()


def test_eplb_misuse_is_rejected(cuda_device):
    hid, ids = _inputs(cuda_device, (4,) * EP)
    stats = [torch.zeros(E, dtype=torch.int32, device=cuda_device) for _ in range(EP)]
    plain = EpComm(EP, E, K, H, C, device=cuda_device)
    small = EpComm(EP, E, K, H, C, device=cuda_device, eplb_stats_max_bytes=64)
    try:
        with pytest.raises(EpError) as ei:  # no capacity reserved
            plain.dispatch(hid, ids, eplb_local_stats=stats)
        assert ei.value.status == EP_ERR_INVALID_ARG
        with pytest.raises(EpError) as ei:  # 128 bytes per rank > 64
            small.dispatch(hid, ids, eplb_local_stats=stats)
        assert ei.value.status == EP_ERR_INVALID_ARG
        with pytest.raises(ValueError):  # every rank passes statistics
            small.dispatch(hid, ids, eplb_local_stats=[s[:16] for s in stats[:-1]] + [None])
        with pytest.raises(ValueError):  # same shape on every rank
            small.dispatch(hid, ids, eplb_local_stats=[s[:16] for s in stats[:-1]] + [stats[-1][:8]])
        res = small.dispatch(hid, ids, eplb_local_stats=[s[:16] for s in stats])  # 64 bytes fits
        assert res.eplb_global_stats.shape == (EP, 16)
        small.combine()
    finally:
        plain.destroy()
        small.destroy()
