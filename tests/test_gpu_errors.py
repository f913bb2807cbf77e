"""Host-side contract checks that need a live handle: state machine, masks,
sizes and the all-or-none rules. Every failing call returns a status before
anything is launched, and the handle stays usable afterwards."""
import ctypes

import numpy as np
import pytest
import torch

import combine_topk_ids_dest_gb300 as ep
from combine_topk_ids_dest_gb300 import EpComm, EpError, _lib
from combine_topk_ids_dest_gb300._lib import ptr_array

pytestmark = pytest.mark.gpu

EP, E, K, H, C = 4, 8, 2, 256, 8


def _inputs(dev, counts=(8, 3, 0, 5), weights=True):
    g = torch.Generator().manual_seed(1)
    hid = [torch.randn(n, H, generator=g).to(torch.bfloat16).to(dev) for n in counts]
    ids = [torch.randint(0, E, (n, K), generator=g, dtype=torch.int32).to(dev) for n in counts]
    w = [torch.rand(n, K, generator=g).to(dev) for n in counts] if weights else None
    return hid, ids, w


def _status(fn, *a, **kw):
    with pytest.raises(EpError) as ei:
        fn(*a, **kw)
    return ei.value.status


@pytest.fixture
def comm(cuda_device):
    c = EpComm(EP, E, K, H, C, enable_rank_mask=True, device=cuda_device)
    yield c
    c.destroy()


def test_state_machine(comm, cuda_device):
    hid, ids, w = _inputs(cuda_device)
    assert _status(comm.combine) == ep.EP_ERR_STATE
    assert _status(comm.get_combine_input_buffer) == ep.EP_ERR_STATE
    comm.dispatch(hid, ids, w)
    assert _status(comm.dispatch, hid, ids, w) == ep.EP_ERR_STATE  # two dispatches in a row
    assert len(comm.get_combine_input_buffer()) == EP
    comm.combine()
    assert _status(comm.combine) == ep.EP_ERR_STATE  # two combines in a row
    comm.dispatch(hid, ids, w)  # usable again
    comm.combine()


def test_mask_rules(comm, cuda_device):
    hid, ids, w = _inputs(cuda_device)
    assert _status(comm.dispatch, hid, ids, w, active_rank_mask=1 << EP) == ep.EP_ERR_INVALID_ARG
    comm.dispatch(hid, ids, w, active_rank_mask=comm.active_rank_mask([0, 2]))
    assert _status(comm.combine, active_rank_mask=comm.active_rank_mask([0])) == ep.EP_ERR_INVALID_ARG
    assert _status(comm.combine) == ep.EP_ERR_INVALID_ARG  # no mask = all ranks != {0,2}
    comm.combine(active_rank_mask=comm.active_rank_mask([0, 2]))


def test_mask_needs_enable_rank_mask(cuda_device):
    c = EpComm(EP, E, K, H, C, enable_rank_mask=False, device=cuda_device)
    try:
        hid, ids, w = _inputs(cuda_device)
        assert _status(c.dispatch, hid, ids, w, active_rank_mask=0b0111) == ep.EP_ERR_INVALID_ARG
        c.dispatch(hid, ids, w, active_rank_mask=0b1111)  # the full set is "no mask"
        c.combine()
    finally:
        c.destroy()


def test_size_rules(comm, cuda_device):
    hid, ids, w = _inputs(cuda_device)
    assert _status(comm.dispatch, hid, ids, w, runtime_max_tokens_per_rank=C + 1) == ep.EP_ERR_INVALID_ARG
    assert _status(comm.dispatch, hid, ids, w, runtime_max_tokens_per_rank=4) == ep.EP_ERR_INVALID_ARG
    with pytest.raises(ValueError):  # scales need hidden % 128 == 0 and fp32 [n, H/128]
        comm.dispatch(hid, ids, w, hidden_states_scale=[torch.ones(x.shape[0], 1, device=cuda_device)
                                                        for x in hid])
    comm.dispatch(hid, ids, w, runtime_max_tokens_per_rank=8)
    comm.combine()


def test_weights_all_or_none(comm, cuda_device):
    hid, ids, w = _inputs(cuda_device)
    w_some = list(w)
    w_some[1] = None
    with pytest.raises(ValueError):
        comm.dispatch(hid, ids, w_some)
    # the same rule in the C ABI: a NULL entry for a rank with tokens
    L = _lib.load()
    counts = (ctypes.c_int32 * EP)(*[x.shape[0] for x in hid])
    res = _lib.EpDispatchResultC()
    wp = [x.data_ptr() for x in w]
    wp[1] = 0
    st = L.ep_dispatch(comm._h, ptr_array([x.data_ptr() for x in hid]), None,
                       ptr_array([x.data_ptr() for x in ids]), ptr_array(wp), counts, -1,
                       ep.ALL_RANKS, None, ctypes.byref(res))
    assert st == ep.EP_ERR_INVALID_ARG
    assert b"all or none" in L.ep_last_error()
    # an empty rank may pass a NULL pointer (an empty [0, K] tensor)
    wp = [x.data_ptr() for x in w]
    wp[2] = 0
    st = L.ep_dispatch(comm._h, ptr_array([x.data_ptr() for x in hid]), None,
                       ptr_array([x.data_ptr() for x in ids]), ptr_array(wp), counts, -1,
                       ep.ALL_RANKS, None, ctypes.byref(res))
    assert st == ep.EP_OK
    assert res.recv_topk_weights
    comm._counts = [x.shape[0] for x in hid]
    comm.combine()


def test_misaligned_pointers_rejected(comm, cuda_device):
    hid, ids, w = _inputs(cuda_device)
    L = _lib.load()
    counts = (ctypes.c_int32 * EP)(*[x.shape[0] for x in hid])
    res = _lib.EpDispatchResultC()
    hp = [x.data_ptr() for x in hid]
    hp[0] += 2
    st = L.ep_dispatch(comm._h, ptr_array(hp), None, ptr_array([x.data_ptr() for x in ids]), None,
                       counts, -1, ep.ALL_RANKS, None, ctypes.byref(res))
    assert st == ep.EP_ERR_INVALID_ARG
    comm.dispatch(hid, ids, w)
    out = [torch.empty(x.shape[0], H, dtype=torch.bfloat16, device=cuda_device) for x in hid]
    op = [o.data_ptr() for o in out]
    op[0] += 2
    st = L.ep_combine(comm._h, None, ptr_array(op), ep.ALL_RANKS, None)
    assert st == ep.EP_ERR_INVALID_ARG
    comm.combine(output=out)


def test_destroy_is_idempotent(cuda_device):
    c = EpComm(EP, E, K, H, C, device=cuda_device)
    c.destroy()
    c.destroy()
    assert _status(c.dispatch, *_inputs(cuda_device)) == ep.EP_ERR_STATE


def test_self_allocating_create_and_plain_abi_round(cuda_device):
    """ep_create (cudaMalloc'd workspace) and the raw C ABI round trip."""
    L = _lib.load()
    h = ctypes.c_void_p()
    assert L.ep_create(2, 4, 2, 16, 3, ep.EP_DTYPE_BF16, 0, ctypes.byref(h)) == ep.EP_OK
    try:
        hid = [torch.arange(32, dtype=torch.float32, device=cuda_device).view(2, 16).to(torch.bfloat16),
               torch.ones(1, 16, dtype=torch.bfloat16, device=cuda_device)]
        ids = [torch.tensor([[0, 1], [1, 3]], dtype=torch.int32, device=cuda_device),
               torch.tensor([[2, 3]], dtype=torch.int32, device=cuda_device)]
        counts = (ctypes.c_int32 * 2)(2, 1)
        res = _lib.EpDispatchResultC()
        assert L.ep_dispatch(h, ptr_array([x.data_ptr() for x in hid]), None,
                             ptr_array([x.data_ptr() for x in ids]), None, counts, -1, ep.ALL_RANKS,
                             None, ctypes.byref(res)) == ep.EP_OK
        assert res.tokens_per_rank == 3 and not res.recv_topk_weights and not res.recv_scale
        out = [torch.empty(2, 16, dtype=torch.bfloat16, device=cuda_device),
               torch.empty(1, 16, dtype=torch.bfloat16, device=cuda_device)]
        for d in range(2):
            p = ctypes.c_void_p()
            assert L.ep_get_combine_input_buffer(h, d, ctypes.byref(p)) == ep.EP_OK
        assert L.ep_combine(h, None, ptr_array([o.data_ptr() for o in out]), ep.ALL_RANKS, None) == ep.EP_OK
        torch.cuda.synchronize()
    finally:
        assert L.ep_destroy(h) == ep.EP_OK
