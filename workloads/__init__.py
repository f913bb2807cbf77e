"""Seeded synthetic inputs for rank-major MoE expert-parallel dispatch/combine.

This module is shared by the tests, the bench and the smoke check. It draws
inputs only: token counts, top-k expert ids, routing weights, hidden rows
(bf16, or fp8 e4m3 with per-128-column fp32 group scales) and the stand-in
expert outputs that combine consumes. It holds none of the dispatch/combine
arithmetic, and neither the oracle nor the CUDA library imports it.

Shapes follow the dispatch/combine contract of FlashInfer's
``MoEEpCommunication`` (page "flashinfer.moe_ep.MoEEpCommunication", methods
``dispatch`` and ``combine``): per source rank, ``hidden_states
[local_num_tokens, hidden]``, ``topk_ids [local_num_tokens, top_k]``,
``topk_weights [local_num_tokens, top_k]`` and ``hidden_states_scale
[local_num_tokens, hidden/128]``.

Draw order per workload (one ``torch.Generator`` seeded with ``seed``):
counts, expert permutation (Zipf id laws only), ids, weight logits, hidden.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

FP8_MAX = 448.0  # largest finite e4m3fn magnitude (OCP FP8 format)
SCALE_GROUP = 128  # columns per fp32 scale, as in DeepSeek-V3 style block quantisation


@dataclass(frozen=True)
class EpWorkload:
    """One dispatch/combine workload: EP geometry plus the input recipe."""

    name: str
    ep_size: int
    num_experts: int
    top_k: int
    hidden: int
    dtype: str  # "bf16", "fp8_e4m3", "fp16" or "fp32"
    capacity: int  # max_tokens_per_rank
    runtime_max: Optional[int]  # runtime_max_tokens_per_rank (None = capacity)
    counts: tuple = ("fixed",)  # ("fixed", c0, c1, ...), ("uniform", lo, hi), ("full",)
    empty_ranks: tuple = ()  # ranks forced to 0 tokens after the count draw
    ids: str = "uniform_distinct"  # "uniform_distinct" | "zipf" | "uniform_dups" | "with_invalid"
    zipf_s: float = 1.1
    weights: bool = True
    scales: bool = False
    dropped_ranks: Optional[tuple] = None  # ranks left out of active_rank_mask
    seed: int = 0
    scale_cols_override: Optional[int] = None  # scale columns when not hidden/128
    combine_dtype: str = "bf16"  # expert outputs / combine results: "bf16", "fp16" or "fp32"

    @property
    def tokens_per_rank(self) -> int:
        return self.capacity if self.runtime_max is None else self.runtime_max

    @property
    def enable_rank_mask(self) -> bool:
        return self.dropped_ranks is not None

    @property
    def elem_bytes(self) -> int:
        return {"bf16": 2, "fp16": 2, "fp8_e4m3": 1, "fp32": 4}[self.dtype]

    @property
    def torch_dtype(self):
        return {"bf16": torch.bfloat16, "fp16": torch.float16, "fp8_e4m3": torch.float8_e4m3fn,
                "fp32": torch.float32}[self.dtype]

    @property
    def combine_torch_dtype(self):
        return {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[self.combine_dtype]

    @property
    def scale_cols(self) -> int:
        if not self.scales:
            return 0
        if self.scale_cols_override is not None:
            return self.scale_cols_override
        return self.hidden // SCALE_GROUP

    def active_ranks(self) -> list:
        drop = set(self.dropped_ranks or ())
        return [r for r in range(self.ep_size) if r not in drop]

    def replace(self, **kw) -> "EpWorkload":
        return dataclasses.replace(self, **kw)


# The five workloads: sizes, dtypes and id laws of the EP configurations the
# method is meant for (Mixtral-8x7B, DeepSeek-V3, Qwen3-MoE shapes).
WORKLOADS = {
    "tiny": EpWorkload(
        name="tiny", ep_size=2, num_experts=8, top_k=2, hidden=256, dtype="bf16",
        capacity=16, runtime_max=None, counts=("fixed", 16, 11)),
    "mixtral_decode": EpWorkload(
        name="mixtral_decode", ep_size=8, num_experts=8, top_k=2, hidden=4096, dtype="bf16",
        capacity=256, runtime_max=256, counts=("uniform", 128, 256)),
    "dsv3_decode": EpWorkload(
        name="dsv3_decode", ep_size=64, num_experts=256, top_k=8, hidden=7168,
        dtype="fp8_e4m3", scales=True, capacity=128, runtime_max=None, counts=("full",)),
    "dsv3_prefill": EpWorkload(
        name="dsv3_prefill", ep_size=32, num_experts=256, top_k=8, hidden=7168,
        dtype="fp8_e4m3", scales=True, capacity=1024, runtime_max=1024, counts=("full",),
        ids="zipf", zipf_s=1.1),
    "qwen3_mask": EpWorkload(
        name="qwen3_mask", ep_size=16, num_experts=128, top_k=8, hidden=4096, dtype="bf16",
        capacity=2048, runtime_max=1536, counts=("uniform", 0, 1536), empty_ranks=(5,),
        dropped_ranks=(3, 11)),
}


# Further EP geometries, for the bandwidth across ep_size, top_k, payload type
# and row width (bench.py --workload <name>); they are not among the five
# configurations above. Every rank sends a full capacity of tokens.
GEOMETRIES = {
    name: EpWorkload(name=name, runtime_max=None, counts=("full",), **kw)
    for name, kw in {
        "geom_ep8_fp8": dict(ep_size=8, num_experts=64, top_k=8, hidden=7168, dtype="fp8_e4m3", scales=True,
                             capacity=2048),
        "geom_ep16_fp8": dict(ep_size=16, num_experts=128, top_k=8, hidden=7168, dtype="fp8_e4m3", scales=True,
                              capacity=1024),
        "geom_ep64_fp8": dict(ep_size=64, num_experts=256, top_k=8, hidden=7168, dtype="fp8_e4m3", scales=True,
                              capacity=512),
        "geom_ep32_bf16_k4": dict(ep_size=32, num_experts=256, top_k=4, hidden=7168, dtype="bf16", capacity=512),
        "geom_ep32_bf16_k16": dict(ep_size=32, num_experts=256, top_k=16, hidden=4096, dtype="bf16", capacity=512),
        "geom_ep64_bf16_k32": dict(ep_size=64, num_experts=64, top_k=32, hidden=2048, dtype="bf16", capacity=128,
                                   ids="uniform_dups"),
    }.items()
}


def by_name(name: str) -> EpWorkload:
    """One of the five workloads, or one of the further geometries."""
    return WORKLOADS[name] if name in WORKLOADS else GEOMETRIES[name]


@dataclass
class EpInputs:
    """Per-source-rank host tensors of one workload (all on the CPU)."""

    wl: EpWorkload
    num_tokens: list  # [ep] python ints
    hidden: list  # [ep] bf16 [n,H] or float8_e4m3fn [n,H]
    scale: Optional[list]  # [ep] fp32 [n,G] or None
    topk_ids: list  # [ep] int32 [n,K]
    topk_weights: Optional[list]  # [ep] fp32 [n,K] or None
    active_rank_mask: int  # uint64 bit set (all ones over ep when masking is off)
    expert_perm: Optional[torch.Tensor] = None

    @property
    def total_tokens(self) -> int:
        return int(sum(self.num_tokens))


def rank_bits(ranks: Sequence[int]) -> int:
    """uint64 bit set with bit r set for every r in ``ranks``."""
    m = 0
    for r in ranks:
        m |= 1 << int(r)
    return m


def _draw_counts(wl: EpWorkload, g: torch.Generator) -> list:
    kind = wl.counts[0]
    if kind == "fixed":
        counts = [int(c) for c in wl.counts[1:]]
        assert len(counts) == wl.ep_size
    elif kind == "full":
        counts = [wl.tokens_per_rank] * wl.ep_size
    elif kind == "uniform":
        lo, hi = int(wl.counts[1]), int(wl.counts[2])
        counts = torch.randint(lo, hi + 1, (wl.ep_size,), generator=g).tolist()
    else:
        raise ValueError(kind)
    for r in wl.empty_ranks:
        counts[r] = 0
    return counts


def _draw_ids(wl: EpWorkload, n: int, g: torch.Generator, perm: Optional[torch.Tensor]):
    E, K = wl.num_experts, wl.top_k
    if n == 0:
        return torch.empty(0, K, dtype=torch.int32)
    if wl.ids in ("uniform_distinct", "with_invalid"):
        ids = torch.multinomial(torch.ones(n, E), K, replacement=False, generator=g)
        if wl.ids == "with_invalid":
            # Out-of-range and negative ids mixed in: about one entry in four.
            junk = torch.randint(0, 4, (n, K), generator=g)
            bad = torch.randint(0, 3, (n, K), generator=g)
            repl = torch.where(bad == 0, torch.full_like(ids, -1),
                               torch.where(bad == 1, torch.full_like(ids, E), torch.full_like(ids, 2 * E + 3)))
            ids = torch.where(junk == 0, repl, ids)
    elif wl.ids == "uniform_dups":
        ids = torch.randint(0, E, (n, K), generator=g)
    elif wl.ids == "zipf":
        assert perm is not None
        p = torch.empty(E, dtype=torch.float64)
        # Expert perm[i] gets popularity (i+1)^-s.
        p[perm] = (torch.arange(E, dtype=torch.float64) + 1.0) ** (-wl.zipf_s)
        ids = torch.multinomial(p.expand(n, E), K, replacement=False, generator=g)
    else:
        raise ValueError(wl.ids)
    return ids.to(torch.int32).contiguous()


def quantize_fp8_groups(x: torch.Tensor):
    """Block-quantise fp32 rows to e4m3fn with one fp32 scale per 128 columns.

    scale = amax/448 per group (1 when the group is all zero); the stored
    value is x/scale clamped to +-448 and rounded by torch's e4m3fn cast.
    """
    n, H = x.shape
    G = H // SCALE_GROUP
    xg = x.view(n, G, SCALE_GROUP)
    amax = xg.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    q = (xg / scale.unsqueeze(-1)).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return q.view(n, H).contiguous(), scale.to(torch.float32).contiguous()


def make_inputs(wl: EpWorkload) -> EpInputs:
    """Draw the seeded inputs of ``wl`` on the CPU."""
    g = torch.Generator().manual_seed(wl.seed)
    counts = _draw_counts(wl, g)
    perm = torch.randperm(wl.num_experts, generator=g) if wl.ids == "zipf" else None
    ids = [_draw_ids(wl, n, g, perm) for n in counts]
    weights = None
    if wl.weights:
        weights = [torch.softmax(torch.randn(n, wl.top_k, generator=g), dim=-1).to(torch.float32).contiguous()
                   for n in counts]
    hidden, scale = [], ([] if wl.scales else None)
    for n in counts:
        x = torch.randn(n, wl.hidden, generator=g)
        if wl.dtype in ("bf16", "fp16", "fp32"):
            hidden.append(x.to(wl.torch_dtype).contiguous())
            if wl.scales:
                scale.append(torch.rand(n, wl.scale_cols, generator=g).to(torch.float32) + 0.5)
        elif wl.scales and wl.scale_cols_override is not None:  # fp8 rows with a custom scale width
            hidden.append(x.clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn).contiguous())
            scale.append(torch.rand(n, wl.scale_cols, generator=g).to(torch.float32) + 0.5)
        elif wl.scales:
            q, s = quantize_fp8_groups(x)
            hidden.append(q)
            scale.append(s)
        else:  # fp8 rows without scales: N(0,1) values cast directly
            hidden.append(x.clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn).contiguous())
    if wl.enable_rank_mask:
        mask = rank_bits(wl.active_ranks())
    else:
        mask = rank_bits(range(wl.ep_size))
    return EpInputs(wl=wl, num_tokens=counts, hidden=hidden, scale=scale, topk_ids=ids,
                    topk_weights=weights, active_rank_mask=mask, expert_perm=perm)


# ---------------------------------------------------------------------------
# Stand-in expert outputs for combine: a counter-based generator written with
# integer tensor ops only, so the CPU and any CUDA device produce the same bits.
# ---------------------------------------------------------------------------
_M32 = 0xFFFFFFFF


def _mix32(x: torch.Tensor) -> torch.Tensor:
    # Multiply-xorshift finaliser on 32-bit values held in int64; both
    # multipliers are below 2^31 so no int64 product overflows.
    x = x ^ (x >> 16)
    x = (x * 0x7FEB352D) & _M32
    x = x ^ (x >> 15)
    x = (x * 0x045D9F3B) & _M32
    x = x ^ (x >> 16)
    return x


def expert_output_rows(seed: int, dest: int, rows: torch.Tensor, hidden: int,
                       device=None, special: bool = False, dtype: str = "bf16") -> torch.Tensor:
    """[len(rows), hidden] stand-in expert output rows of rank ``dest``, as
    bf16 (default), fp16 or fp32.

    Element (dest, row, h) is a pure function of its coordinates: sign and
    mantissa bits from 32-bit hashes, exponent within 2^-7 .. 2^8 (bf16/fp32:
    biased 120..134; fp16: biased 8..22). With ``special`` the exponent range
    also covers zeros, subnormals and tiny normals (biased exponent 0..3), to
    exercise the fp32 accumulation without flush-to-zero.
    """
    if dtype != "bf16":
        return _expert_output_rows_wide(seed, dest, rows, hidden, device, special, dtype)
    device = rows.device if device is None else device
    r = rows.to(device=device, dtype=torch.int64).view(-1, 1)
    h = torch.arange(hidden, device=device, dtype=torch.int64).view(1, -1)
    key = (seed * 0x9E37 + dest * 0x3C6EF372 + r * 0x1B873593 + h * 0x27D4EB2F) & _M32
    x = _mix32(key)
    y = _mix32(x ^ 0x5BD1E995)
    sign = (x >> 31) & 1
    mant = (x >> 8) & 0x7F
    if special:
        ex = y % 19
        ex = torch.where(ex < 4, ex, ex + 116)  # 0..3 or 120..134
    else:
        ex = 120 + (y % 15)
    bits = (sign << 15) | (ex << 7) | mant
    bits = torch.where(bits >= 0x8000, bits - 0x10000, bits)  # reinterpret as int16
    return bits.to(torch.int16).view(torch.bfloat16)


def _expert_output_rows_wide(seed, dest, rows, hidden, device, special, dtype):
    device = rows.device if device is None else device
    r = rows.to(device=device, dtype=torch.int64).view(-1, 1)
    h = torch.arange(hidden, device=device, dtype=torch.int64).view(1, -1)
    key = (seed * 0x9E37 + dest * 0x3C6EF372 + r * 0x1B873593 + h * 0x27D4EB2F) & _M32
    x = _mix32(key)
    y = _mix32(x ^ 0x5BD1E995)
    z = _mix32(y ^ 0x68E31DA4)
    sign = (x >> 31) & 1
    if dtype == "fp16":
        mant = (x >> 8) & 0x3FF
        ex = y % 19 if special else 8 + (y % 15)
        if special:
            ex = torch.where(ex < 4, ex, ex + 4)  # 0..3 or 8..22
        bits = (sign << 15) | (ex << 10) | mant
        bits = torch.where(bits >= 0x8000, bits - 0x10000, bits)
        return bits.to(torch.int16).view(torch.float16)
    if dtype == "fp32":
        mant = (((x >> 8) & 0x7F) << 16) | (z & 0xFFFF)
        ex = y % 19 if special else 120 + (y % 15)
        if special:
            ex = torch.where(ex < 4, ex, ex + 116)
        bits = (sign << 31) | (ex << 23) | mant
        bits = torch.where(bits >= (1 << 31), bits - (1 << 32), bits)
        return bits.to(torch.int32).view(torch.float32)
    raise ValueError(dtype)
