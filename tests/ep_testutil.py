"""Helpers shared by the tests: independent restatements of the routing rule
(Python sets, not the oracle's loops) and shrunk variants of the workloads."""
import numpy as np
import torch

INV = -1


def expected_dests(ids_row, num_experts, ep_size, mask_enabled=False, active=None):
    """Set of ranks a token goes to: owners of its in-range expert ids, kept
    only if active when masking is on (experts split contiguously)."""
    epr = num_experts // ep_size
    dests = {int(e) // epr for e in ids_row if 0 <= int(e) < num_experts}
    if mask_enabled:
        dests = {d for d in dests if (active >> d) & 1}
    return dests


def raw_bytes(t):
    """uint8 numpy [n, row_bytes] of a bf16 / fp8 / any CPU tensor."""
    t = t.detach().contiguous()
    n = t.shape[0]
    return t.view(torch.uint8).numpy().reshape(n, -1)


def bf16_bits(t):
    return t.detach().contiguous().view(torch.int16).numpy().view(np.uint16)


def small(wl, hidden=256, tokens=None):
    """The same EP geometry, id law and dtypes as ``wl`` with a short hidden
    row and few tokens per rank, so the oracle runs in well under a second."""
    cap = tokens if tokens is not None else min(wl.capacity, 24)
    rt = None if wl.runtime_max is None else min(wl.runtime_max, cap)
    counts = wl.counts
    if counts[0] == "uniform":
        counts = ("uniform", min(counts[1], rt or cap), rt or cap)
    elif counts[0] == "fixed":
        counts = ("fixed",) + tuple(min(c, rt or cap) for c in counts[1:])
    return wl.replace(name=wl.name + "_small", hidden=hidden, capacity=cap, runtime_max=rt,
                      counts=counts)
