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
    if n == 0:
        return np.zeros((0, t[0:0].view(-1).element_size() * (t.shape[1] if t.dim() > 1 else 1)), np.uint8)
    return t.view(torch.uint8).numpy().reshape(n, -1)


def bf16_bits(t):
    return t.detach().contiguous().view(torch.int16).numpy().view(np.uint16)


def out_bits(t):
    """Raw bits of a bf16/fp16 (uint16) or fp32 (uint32) CPU tensor."""
    t = t.detach().contiguous()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


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


# ---------------------------------------------------------------------------
# GPU round trip through the library, and the matching oracle computation
# ---------------------------------------------------------------------------
EO_SEED = 7


def to_dev(lst, device):
    return None if lst is None else [x.to(device) for x in lst]


_CDT = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}


def fill_expert_outputs(comm, T, device, seed=EO_SEED, special=False, caller=False):
    """Writes the stand-in expert outputs of every rank: into the backend
    combine-input buffers of the communicator's ranks (all of them, or its
    partition's), or (caller=True) into fresh tensors of every rank it returns."""
    import workloads
    ep, H = comm.ep_size, comm.hidden
    rows = torch.arange(ep * T, device=device)
    outs = []
    for d in (range(ep) if caller else range(comm.first_rank, comm.first_rank + comm.num_ranks)):
        eo = workloads.expert_output_rows(seed, d, rows, H, device=device, special=special,
                                          dtype=_CDT[comm.combine_dtype])
        if caller:
            outs.append(eo.contiguous())
        else:
            comm.get_combine_input_buffer(rank=d).copy_(eo)
    return outs if caller else None


def gpu_round(inp, device, special=False, caller_eo=False, comm=None, keep=False, dev_counts=None, pdl=False):
    """dispatch + (stand-in expert) + combine of ``inp`` through EpComm.
    Returns host copies of the receive buffers and outputs. ``dev_counts``
    (a list of ints) is passed as device-side token counts; the outputs are
    then cut to the counts clamped to [0, the rank's rows]. ``pdl``: a
    communicator created here launches with programmatic dependent launch."""
    from combine_topk_ids_dest_gb300 import EpComm
    wl = inp.wl
    own = comm is None
    if own:
        comm = EpComm(wl.ep_size, wl.num_experts, wl.top_k, wl.hidden, wl.capacity, dtype=wl.torch_dtype,
                      enable_rank_mask=wl.enable_rank_mask, device=device,
                      scale_cols=wl.scale_cols if wl.scales else None,
                      combine_dtype=wl.combine_torch_dtype, pdl=pdl)
    mask = inp.active_rank_mask if wl.enable_rank_mask else None
    res = comm.dispatch(to_dev(inp.hidden, device), to_dev(inp.topk_ids, device),
                        to_dev(inp.topk_weights, device),
                        hidden_states_scale=to_dev(inp.scale, device),
                        runtime_max_tokens_per_rank=wl.runtime_max, active_rank_mask=mask,
                        num_tokens_device=None if dev_counts is None else
                        torch.tensor(dev_counts, dtype=torch.int32, device=device))
    T = res.tokens_per_rank
    eo = fill_expert_outputs(comm, T, device, special=special, caller=caller_eo)
    out = comm.combine(eo, active_rank_mask=mask)
    if dev_counts is not None:
        out = [o[:clamp_count(c, n)] for o, c, n in zip(out, dev_counts, inp.num_tokens)]
    torch.cuda.synchronize(device)
    host = dict(
        T=T,
        recv_ids=[x.cpu().numpy() for x in res.topk_ids],
        recv_hidden=[raw_bytes(x.cpu()) for x in res.hidden_states],
        recv_scale=None if res.hidden_states_scale is None else
        [x.cpu().numpy() for x in res.hidden_states_scale],
        recv_weights=None if res.topk_weights is None else [x.cpu().numpy() for x in res.topk_weights],
        out=[out_bits(o.cpu()) for o in out],
    )
    if own and not keep:
        comm.destroy()
    if keep:
        host["comm"] = comm
    return host


def oracle_round(inp, special=False):
    """The oracle's dispatch and combine of ``inp`` with the same stand-in
    expert outputs (generated on the CPU)."""
    import oracle
    import workloads
    wl = inp.wl
    T, ep, H = wl.tokens_per_rank, wl.ep_size, wl.hidden
    disp = oracle.dispatch(ep, wl.num_experts, wl.top_k, T, inp.num_tokens, inp.hidden, inp.topk_ids,
                           scale=inp.scale, topk_weights=inp.topk_weights,
                           mask_enabled=wl.enable_rank_mask, active_rank_mask=inp.active_rank_mask,
                           row_bytes=H * wl.elem_bytes, scale_cols=wl.scale_cols)
    rows = torch.arange(ep * T)
    eo = [out_bits(workloads.expert_output_rows(EO_SEED, d, rows, H, special=special,
                                                dtype=wl.combine_dtype)) for d in range(ep)]
    if wl.combine_dtype == "bf16":
        out = oracle.combine(ep, wl.num_experts, wl.top_k, H, T, inp.num_tokens, inp.topk_ids, eo,
                             mask_enabled=wl.enable_rank_mask, active_rank_mask=inp.active_rank_mask)
    else:
        out = oracle.combine_typed(ep, wl.num_experts, wl.top_k, H, T, inp.num_tokens, inp.topk_ids, eo,
                                   wl.combine_dtype, mask_enabled=wl.enable_rank_mask,
                                   active_rank_mask=inp.active_rank_mask)
        out = [o.view(np.uint32) if o.dtype == np.float32 else o for o in out]
    return disp, out


def assert_round_equal(inp, got, disp, out):
    """Bit-exact comparison: every id row; hidden/scale/weight rows where the
    oracle's id row is valid (the others are unspecified); every output."""
    wl = inp.wl
    for d in range(wl.ep_size):
        np.testing.assert_array_equal(got["recv_ids"][d], disp.recv_ids[d], err_msg=f"ids of rank {d}")
        valid = (disp.recv_ids[d] != INV).any(axis=1)  # a routed row holds an id owned by d
        np.testing.assert_array_equal(got["recv_hidden"][d][valid], disp.recv_hidden[d][valid],
                                      err_msg=f"hidden rows of rank {d}")
        if disp.recv_scale is not None:
            np.testing.assert_array_equal(got["recv_scale"][d][valid].view(np.uint32),
                                          disp.recv_scale[d][valid].view(np.uint32))
        else:
            assert got["recv_scale"] is None
        if disp.recv_weights is not None:
            np.testing.assert_array_equal(got["recv_weights"][d][valid].view(np.uint32),
                                          disp.recv_weights[d][valid].view(np.uint32))
        else:
            assert got["recv_weights"] is None
    for s in range(wl.ep_size):
        np.testing.assert_array_equal(got["out"][s], out[s], err_msg=f"combine output of rank {s}")


def clamp_count(c, n):
    """A device-side token count as the kernels use it: clamped to [0, n]."""
    return min(max(int(c), 0), int(n))


def cut_inputs(inp, counts):
    """``inp`` with every rank's tensors cut to its first ``counts[s]`` rows."""
    import dataclasses
    cut = lambda lst: None if lst is None else [x[:n] for x, n in zip(lst, counts)]
    return dataclasses.replace(inp, num_tokens=list(counts), hidden=cut(inp.hidden), scale=cut(inp.scale),
                               topk_ids=cut(inp.topk_ids), topk_weights=cut(inp.topk_weights))
