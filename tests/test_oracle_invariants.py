"""Pins of the oracle by invariants that the pages fix, checked with code
independent of the oracle (CPU only):

- every valid routed row equals its source row byte for byte, and carries the
  token's id, scale and weight rows unchanged;
- every padding or unrouted row carries top_k x invalid_expert_id and its other
  payload rows are left alone;
- the number of valid rows equals the number of (token, rank) routes;
- with identity experts, combine(dispatch(x)) is x times the sum of the
  weights of the token's unmasked experts, within two bf16 roundings; exactly
  x when the weights are dyadic.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from ep_testutil import INV, bf16_bits, expected_dests, raw_bytes, small

CASES = ["tiny"] + [k for k in workloads.WORKLOADS if k != "tiny"]


def _wl(name):
    wl = workloads.WORKLOADS[name]
    return wl if name == "tiny" else small(wl)


def _run_dispatch(inp, payload=True):
    wl = inp.wl
    return oracle.dispatch(wl.ep_size, wl.num_experts, wl.top_k, wl.tokens_per_rank,
                           inp.num_tokens, inp.hidden, inp.topk_ids, scale=inp.scale,
                           topk_weights=inp.topk_weights, mask_enabled=wl.enable_rank_mask,
                           active_rank_mask=inp.active_rank_mask, payload=payload)


@pytest.mark.parametrize("name", CASES + ["with_invalid", "dups", "one_scale_column", "three_scale_columns_fp8",
                                  "mask_on_high_ranks"])
def test_dispatch_rows(name):
    if name == "mask_on_high_ranks":  # the mask is 64 bits: ranks 32..63 are masked like the others
        wl = small(workloads.WORKLOADS["dsv3_decode"]).replace(dropped_ranks=(0, 31, 32, 40, 63))
    elif name == "one_scale_column":  # scale rows of width 1 travel like any other
        wl = small(workloads.WORKLOADS["qwen3_mask"]).replace(scales=True, scale_cols_override=1)
    elif name == "three_scale_columns_fp8":
        wl = small(workloads.WORKLOADS["dsv3_decode"]).replace(scale_cols_override=3, ep_size=8, num_experts=16)
    elif name == "with_invalid":
        wl = small(workloads.WORKLOADS["qwen3_mask"]).replace(ids="with_invalid")
    elif name == "dups":
        wl = small(workloads.WORKLOADS["dsv3_decode"]).replace(ids="uniform_dups", ep_size=8,
                                                              num_experts=16)
    else:
        wl = _wl(name)
    inp = workloads.make_inputs(wl)
    out = _run_dispatch(inp)
    ep, T, K, E = wl.ep_size, wl.tokens_per_rank, wl.top_k, wl.num_experts
    n_valid, n_routes = 0, 0
    for s in range(ep):
        hb = raw_bytes(inp.hidden[s]) if inp.num_tokens[s] else None
        for t in range(inp.num_tokens[s]):
            n_routes += len(expected_dests(inp.topk_ids[s][t].tolist(), E, ep,
                                           wl.enable_rank_mask, inp.active_rank_mask))
        for d in range(ep):
            for t in range(T):
                r = s * T + t
                ids_row = out.recv_ids[d][r]
                dests = set()
                if t < inp.num_tokens[s]:
                    dests = expected_dests(inp.topk_ids[s][t].tolist(), E, ep,
                                           wl.enable_rank_mask, inp.active_rank_mask)
                if d in dests:
                    n_valid += 1
                    assert ids_row.tolist() == inp.topk_ids[s][t].tolist()
                    np.testing.assert_array_equal(out.recv_hidden[d][r], hb[t])
                    if inp.scale is not None:
                        np.testing.assert_array_equal(out.recv_scale[d][r].view(np.uint32),
                                                      inp.scale[s][t].numpy().view(np.uint32))
                    if inp.topk_weights is not None:
                        np.testing.assert_array_equal(out.recv_weights[d][r].view(np.uint32),
                                                      inp.topk_weights[s][t].numpy().view(np.uint32))
                else:
                    assert ids_row.tolist() == [INV] * K
                    assert (out.recv_hidden[d][r] == oracle.SENTINEL_BYTE).all()
                    if out.recv_weights is not None:
                        assert (out.recv_weights[d][r].view(np.uint32) == oracle.SENTINEL_F32_BITS).all()
    assert n_valid == n_routes


def _x_f64(inp, s):
    """Token values of source rank s as float64, the way the expert sees them."""
    h = inp.hidden[s]
    if h.dtype == torch.bfloat16:
        return h.to(torch.float64).numpy()
    x = h.to(torch.float32).to(torch.float64).numpy()
    sc = inp.scale[s].to(torch.float64).numpy()
    return x * np.repeat(sc, workloads.SCALE_GROUP, axis=1)


@pytest.mark.parametrize("name", CASES)
def test_identity_expert_roundtrip(name):
    wl = _wl(name)
    inp = workloads.make_inputs(wl)
    out = _run_dispatch(inp)
    ep, T, K, E, H = wl.ep_size, wl.tokens_per_rank, wl.top_k, wl.num_experts, wl.hidden
    eo = oracle.identity_expert(ep, E, K, H, wl.elem_bytes, T, out)
    comb = oracle.combine(ep, E, K, H, T, inp.num_tokens, inp.topk_ids, eo,
                          mask_enabled=wl.enable_rank_mask, active_rank_mask=inp.active_rank_mask)
    epr = E // ep
    for s in range(ep):
        n = inp.num_tokens[s]
        if n == 0:
            assert comb[s].shape == (0, H)
            continue
        x = _x_f64(inp, s)
        got = torch.from_numpy(comb[s].view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
        w = inp.topk_weights[s].to(torch.float64).numpy()
        ids = inp.topk_ids[s].numpy()
        W = np.zeros(n)
        for t in range(n):
            for k in range(K):
                e = int(ids[t, k])
                if 0 <= e < E and (not wl.enable_rank_mask or (inp.active_rank_mask >> (e // epr)) & 1):
                    W[t] += w[t, k]
        want = x * W[:, None]
        # two bf16 roundings (per rank, then the sum): relative 2^-7, plus fp32 slack
        bound = np.abs(want) * (2.0 ** -7) * 1.01 + (K + 1) * 2.0 ** -133
        assert (np.abs(got - want) <= bound).all()


@pytest.mark.parametrize("ep,E,mask", [(2, 4, None), (4, 8, None), (4, 8, (1,)), (3, 3, (0, 2))])
def test_identity_roundtrip_exact_with_dyadic_weights(ep, E, mask):
    wl = workloads.EpWorkload(name="dyadic", ep_size=ep, num_experts=E, top_k=2, hidden=64,
                              dtype="bf16", capacity=8, runtime_max=None, counts=("uniform", 0, 8),
                              dropped_ranks=mask, seed=3)
    inp = workloads.make_inputs(wl)
    inp.topk_weights = [torch.full((n, 2), 0.5) for n in inp.num_tokens]
    out = _run_dispatch(inp)
    eo = oracle.identity_expert(ep, E, 2, 64, 2, wl.tokens_per_rank, out)
    comb = oracle.combine(ep, E, 2, 64, wl.tokens_per_rank, inp.num_tokens, inp.topk_ids, eo,
                          mask_enabled=wl.enable_rank_mask, active_rank_mask=inp.active_rank_mask)
    for s in range(ep):
        x = bf16_bits(inp.hidden[s]) if inp.num_tokens[s] else np.zeros((0, 64), np.uint16)
        for t in range(inp.num_tokens[s]):
            kept = [e for e in inp.topk_ids[s][t].tolist()
                    if not wl.enable_rank_mask or (inp.active_rank_mask >> (e // (E // ep))) & 1]
            if len(kept) == 2:
                np.testing.assert_array_equal(comb[s][t], x[t])
            elif len(kept) == 1:  # x * 0.5 is exact in bf16 for these magnitudes
                half = (torch.from_numpy(x[t].view(np.int16)).view(torch.bfloat16) * 0.5)
                np.testing.assert_array_equal(comb[s][t], bf16_bits(half.view(1, -1))[0])
            else:
                assert (comb[s][t] == 0).all()
