"""Special values through the combine: expert outputs holding +inf, -inf, NaN
and the largest finite values, so that the sums meet inf + inf, inf - inf,
NaN + x and overflow, in all three combine types. Where the oracle's result
is not a NaN the GPU's must match it bit for bit; where it is a NaN the GPU's
must be a NaN too (the two sides may encode NaN differently: any NaN is
accepted, as the combine's reading states)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from combine_topk_ids_dest_gb300 import EpComm
from ep_testutil import to_dev

pytestmark = pytest.mark.gpu

WL = workloads.EpWorkload(name="special", ep_size=4, num_experts=8, top_k=3, hidden=64, dtype="bf16",
                          capacity=8, runtime_max=None, counts=("fixed", 8, 5, 0, 8), ids="uniform_dups", seed=95)

# per combine type: +inf, -inf, NaN, largest finite, minus it, 1.0 (raw bits)
SPECIAL = {
    "bf16": (np.uint16, [0x7F80, 0xFF80, 0x7FC1, 0x7F7F, 0xFF7F, 0x3F80]),
    "fp16": (np.uint16, [0x7C00, 0xFC00, 0x7E01, 0x7BFF, 0xFBFF, 0x3C00]),
    "fp32": (np.uint32, [0x7F800000, 0xFF800000, 0x7FC00001, 0x7F7FFFFF, 0xFF7FFFFF, 0x3F800000]),
}
TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def _is_nan(bits, cdt):
    if cdt == "fp32":
        return ((bits & 0x7F800000) == 0x7F800000) & ((bits & 0x007FFFFF) != 0)
    if cdt == "fp16":
        return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x03FF) != 0)
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)


@pytest.mark.parametrize("cdt", ["bf16", "fp16", "fp32"])
def test_special_values_in_combine(cuda_device, cdt):
    npt, vals = SPECIAL[cdt]
    inp = workloads.make_inputs(WL)
    ep, T, H = WL.ep_size, WL.capacity, WL.hidden
    rng = np.random.default_rng(7)
    # each element picks one of the special values (1.0 twice as often), independently per rank
    pick = rng.choice(len(vals) + 1, size=(ep, ep * T, H))
    table = np.array(vals + [vals[-1]], dtype=npt)
    eo_bits = [table[pick[d]] for d in range(ep)]
    comm = EpComm(ep, WL.num_experts, WL.top_k, H, T, device=cuda_device, combine_dtype=TORCH[cdt])
    try:
        comm.dispatch(to_dev(inp.hidden, cuda_device), to_dev(inp.topk_ids, cuda_device),
                      to_dev(inp.topk_weights, cuda_device))
        view = torch.int32 if cdt == "fp32" else torch.int16
        signed = np.int32 if cdt == "fp32" else np.int16
        eo = [torch.from_numpy(b.view(signed).copy()).to(cuda_device).view(TORCH[cdt]) for b in eo_bits]
        out = comm.combine(eo)
        torch.cuda.synchronize(cuda_device)
        got = [o.cpu().view(view).numpy().view(npt) for o in out]
    finally:
        comm.destroy()
    want = oracle.combine_typed(ep, WL.num_experts, WL.top_k, H, T, inp.num_tokens, inp.topk_ids, eo_bits, cdt)
    want = [np.asarray(w).view(npt) for w in want]
    n_nan = n_inf = 0
    for s in range(ep):
        w, g = want[s], got[s]
        nan = _is_nan(w, cdt)
        np.testing.assert_array_equal(_is_nan(g, cdt), nan, err_msg=f"{cdt}: NaN positions of rank {s}")
        np.testing.assert_array_equal(g[~nan], w[~nan], err_msg=f"{cdt}: non-NaN results of rank {s}")
        n_nan += int(nan.sum())
        inf_bits = vals[0]
        n_inf += int(((w & ~npt(1 << (8 * np.dtype(npt).itemsize - 1))) == inf_bits).sum())
    assert n_nan > 0 and n_inf > 0  # the case really exercised both
