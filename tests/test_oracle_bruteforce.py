"""Brute-force pin of the oracle's routing (CPU only).

For small EP groups, every top-k id tuple over [-1, E] (in-range, negative and
too-large ids, duplicates) is dispatched under every rank mask. The id plane
is compared with the set rule written independently in Python, and combine is
run on expert outputs equal to 2^d on rank d, so its (exact) result names the
set of ranks it summed.
"""
import itertools

import numpy as np
import pytest

import oracle
from ep_testutil import INV, expected_dests


@pytest.mark.parametrize("ep,epr,K", [(1, 1, 1), (1, 2, 2), (2, 1, 2), (2, 2, 3), (3, 1, 2),
                                      (3, 2, 2), (3, 1, 3)])
def test_bruteforce_routing(ep, epr, K):
    E = ep * epr
    tuples = list(itertools.product(range(-1, E + 1), repeat=K))
    n = len(tuples)
    T = (n + ep - 1) // ep + 1  # at least one padding slot per source rank
    counts = [len(tuples[s::ep]) for s in range(ep)]
    ids = [np.array(tuples[s::ep], np.int32).reshape(-1, K) for s in range(ep)]
    hidden = [np.zeros((c, 16), np.uint8) for c in counts]
    H = 1
    two_pow = [np.full((ep * T, H), oracle.f32_to_bf16(2.0 ** d), np.uint16) for d in range(ep)]
    for mask in range(1 << ep):
        for enabled in ((False, True) if mask == (1 << ep) - 1 else (True,)):
            out = oracle.dispatch(ep, E, K, T, counts, hidden, ids, mask_enabled=enabled,
                                  active_rank_mask=mask, payload=False)
            comb = oracle.combine(ep, E, K, H, T, counts, ids, two_pow, mask_enabled=enabled,
                                  active_rank_mask=mask)
            for s in range(ep):
                for t in range(T):
                    dests = set()
                    if t < counts[s]:
                        dests = expected_dests(ids[s][t].tolist(), E, ep, enabled, mask)
                        assert oracle.bf16_to_f32(int(comb[s][t, 0])) == float(sum(2 ** d for d in dests))
                    for d in range(ep):
                        row = out.recv_ids[d][s * T + t].tolist()
                        assert row == (ids[s][t].tolist() if d in dests else [INV] * K)
