"""CPU oracle of rank-major MoE expert-parallel dispatch/combine.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` import this package. The product library
(``combine_topk_ids_dest_gb300``) never imports it, and it imports nothing of
the product.

The arithmetic lives in ``ep_oracle.c`` (plain loops, see its header for the
passages of the FlashInfer ``moe_ep`` pages it follows and the readings taken
where they are silent). This module compiles it with gcc on first use and
marshals numpy / torch CPU arrays to it through ctypes.

Every function here is pinned by ``tests/test_oracle_*.py`` against values
that do not come from the oracle itself: the hand-worked example under
``tests/golden/``, closed forms, library format conversions and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np

INVALID_EXPERT_ID = -1
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libep_oracle.so")
_lock = threading.Lock()
_lib = None

# Payload sentinels for rows the method leaves unspecified.
SENTINEL_BYTE = 0xA5
SENTINEL_F32_BITS = 0x7FA5A5A5  # a NaN payload nobody writes by accident


def build(force: bool = False) -> str:
    """Compile ep_oracle.c into oracle/_build/libep_oracle.so (gcc, no fast-math).

    EP_ORACLE_LIB in the environment names another build to load instead; the
    mutation test uses it to run the pins against copies of the oracle with
    planted mistakes."""
    override = os.environ.get("EP_ORACLE_LIB")
    if override:
        return override
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC])
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, u64 = ctypes.c_int, ctypes.c_uint64
            L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f32.restype = ctypes.c_float
            L.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
            L.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
            L.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_to_f32.restype = ctypes.c_float
            L.oracle_routed_to.argtypes = [P, i32, i32, i32, i32, i32, u64]
            L.oracle_routed_to.restype = i32
            L.oracle_dispatch.argtypes = [i32, i32, i32, i32, i32, i32, i32, u64, P,
                                          P, P, P, P, P, P, P, P]
            L.oracle_dispatch.restype = i32
            L.oracle_combine.argtypes = [i32, i32, i32, i32, i32, i32, u64, P, P, P, P]
            L.oracle_combine.restype = i32
            L.oracle_identity_expert.argtypes = [i32, i32, i32, i32, i32, i32, i32,
                                                 P, P, P, P, P]
            L.oracle_identity_expert.restype = i32
            L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_f16_to_f32.restype = ctypes.c_float
            L.oracle_f32_to_f16_rne.argtypes = [ctypes.c_float]
            L.oracle_f32_to_f16_rne.restype = ctypes.c_uint16
            L.oracle_combine_typed.argtypes = [i32, i32, i32, i32, i32, i32, u64, P, P, i32, P, P]
            L.oracle_combine_typed.restype = i32
            L.oracle_eplb_gather.argtypes = [i32, i32, P, P]
            L.oracle_eplb_gather.restype = i32
            _lib = L
    return _lib


# ---- marshalling helpers ---------------------------------------------------

def _np(x, dtype=None):
    """numpy view of a numpy array or torch CPU tensor (bf16/fp8 as raw bits)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        import torch
        t = x.detach().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        elif t.dtype == torch.float8_e4m3fn:
            t = t.view(torch.uint8)
        x = t.numpy()
    a = np.ascontiguousarray(x)
    if dtype is not None:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def _ptrs(arrays: Optional[Sequence]):
    """(ctypes array of data pointers, keep-alive list) for a per-rank list."""
    if arrays is None:
        return None, []
    keep = list(arrays)
    arr = (ctypes.c_void_p * len(keep))(*[(a.ctypes.data if a is not None and a.size else None)
                                          for a in keep])
    return arr, keep


def _voidp(arr):
    return ctypes.cast(arr, ctypes.c_void_p) if arr is not None else None


# ---- scalar format functions -----------------------------------------------

def bf16_to_f32(bits: int) -> float:
    return float(lib().oracle_bf16_to_f32(int(bits) & 0xFFFF))


def f32_to_bf16(x: float) -> int:
    return int(lib().oracle_f32_to_bf16_rne(float(np.float32(x))))


def f32_bits_to_bf16(bits: int) -> int:
    """f32_to_bf16 for an exact binary32 bit pattern (NaNs and -0 included)."""
    f = np.array([bits], dtype=np.uint32).view(np.float32)[0]
    return int(lib().oracle_f32_to_bf16_rne(ctypes.c_float(f)))


def f16_to_f32(bits: int) -> float:
    return float(lib().oracle_f16_to_f32(int(bits) & 0xFFFF))


def f32_bits_to_f16(bits: int) -> int:
    """binary32 bit pattern -> binary16 bits, round to nearest even."""
    f = np.array([bits], dtype=np.uint32).view(np.float32)[0]
    return int(lib().oracle_f32_to_f16_rne(ctypes.c_float(f)))


def e4m3_to_f32(code: int) -> float:
    return float(lib().oracle_e4m3_to_f32(int(code) & 0xFF))


def routed_to(ids_row: Sequence[int], num_experts: int, ep_size: int, d: int,
              mask_enabled: bool = False, active_rank_mask: int = (1 << 64) - 1) -> bool:
    a = np.ascontiguousarray(np.asarray(ids_row, dtype=np.int32))
    return bool(lib().oracle_routed_to(a.ctypes.data, len(a), num_experts, ep_size, d,
                                       int(bool(mask_enabled)), active_rank_mask & ((1 << 64) - 1)))


# ---- dispatch / combine ----------------------------------------------------

@dataclass
class OracleDispatch:
    tokens_per_rank: int
    recv_hidden: Optional[List[np.ndarray]]  # [ep] uint8 [ep*T, row_bytes]
    recv_scale: Optional[List[np.ndarray]]  # [ep] float32 [ep*T, G]
    recv_ids: List[np.ndarray]  # [ep] int32 [ep*T, K]
    recv_weights: Optional[List[np.ndarray]]  # [ep] float32 [ep*T, K]


def dispatch(ep_size: int, num_experts: int, top_k: int, tokens_per_rank: int,
             num_tokens: Sequence[int], hidden: Sequence, topk_ids: Sequence, *,
             scale: Optional[Sequence] = None, topk_weights: Optional[Sequence] = None,
             mask_enabled: bool = False, active_rank_mask: int = (1 << 64) - 1,
             payload: bool = True, row_bytes: Optional[int] = None,
             scale_cols: Optional[int] = None) -> OracleDispatch:
    """Receive buffers of every rank after one dispatch (see ep_oracle.c).

    ``hidden[s]`` is [n_s, H] bf16/fp8 (raw bytes are copied); ``scale[s]``
    [n_s, G] fp32; ``topk_ids[s]`` [n_s, K] int32; ``topk_weights[s]`` [n_s, K]
    fp32. Rows the method leaves unspecified keep the sentinel fill. With
    ``payload=False`` only the id planes are produced. ``row_bytes`` (hidden
    row bytes) and ``scale_cols`` are taken from the data when omitted; pass
    them when every rank is empty.
    """
    ep, T, K = ep_size, tokens_per_rank, top_k
    counts = np.ascontiguousarray(np.asarray(num_tokens, dtype=np.int32))
    hid = [_np(h) for h in hidden]
    hid = [h.view(np.uint8).reshape(h.shape[0], -1) if h.size else h.reshape(0, 0).view(np.uint8)
           for h in hid]
    if row_bytes is None:  # from the data; pass it when every rank is empty
        row_bytes = max((h.shape[1] for h in hid if h.size), default=0)
    ids = [_np(i, np.int32) for i in topk_ids]
    sc = [_np(x, np.float32) for x in scale] if scale is not None else None
    G = 0
    if sc is not None:
        G = scale_cols if scale_cols is not None else max((x.shape[1] for x in sc if x.size), default=0)
    w = [_np(x, np.float32) for x in topk_weights] if topk_weights is not None else None

    rows = ep * T
    recv_ids = [np.empty((rows, K), np.int32) for _ in range(ep)]
    for a in recv_ids:
        a.fill(0x5A5A5A5A)
    recv_hidden = recv_scale = recv_weights = None
    if payload:
        recv_hidden = [np.full((rows, row_bytes), SENTINEL_BYTE, np.uint8) for _ in range(ep)]
        if sc is not None:
            recv_scale = [np.full((rows, G), SENTINEL_F32_BITS, np.uint32).view(np.float32)
                          for _ in range(ep)]
        if w is not None:
            recv_weights = [np.full((rows, K), SENTINEL_F32_BITS, np.uint32).view(np.float32)
                            for _ in range(ep)]
    p_hid, k1 = _ptrs(hid)
    p_sc, k2 = _ptrs(sc)
    p_ids, k3 = _ptrs(ids)
    p_w, k4 = _ptrs(w)
    p_rh, k5 = _ptrs(recv_hidden)
    p_rs, k6 = _ptrs(recv_scale)
    p_ri, k7 = _ptrs(recv_ids)
    p_rw, k8 = _ptrs(recv_weights)
    rc = lib().oracle_dispatch(ep, num_experts, K, row_bytes, G, T, int(bool(mask_enabled)),
                               active_rank_mask & ((1 << 64) - 1), counts.ctypes.data,
                               _voidp(p_hid), _voidp(p_sc), _voidp(p_ids), _voidp(p_w),
                               _voidp(p_rh), _voidp(p_rs), _voidp(p_ri), _voidp(p_rw))
    if rc != 0:
        raise ValueError("oracle_dispatch: inconsistent sizes")
    return OracleDispatch(T, recv_hidden, recv_scale, recv_ids, recv_weights)


def combine(ep_size: int, num_experts: int, top_k: int, hidden: int, tokens_per_rank: int,
            num_tokens: Sequence[int], topk_ids: Sequence, expert_output: Sequence, *,
            mask_enabled: bool = False, active_rank_mask: int = (1 << 64) - 1) -> List[np.ndarray]:
    """Per source rank, uint16 (bf16 bits) [n_s, hidden] combine output.

    ``expert_output[d]`` is the bf16 [ep*T, hidden] combine input of rank d.
    """
    ep = ep_size
    counts = np.ascontiguousarray(np.asarray(num_tokens, dtype=np.int32))
    ids = [_np(i, np.int32) for i in topk_ids]
    eo = [_np(e, np.uint16) for e in expert_output]
    out = [np.zeros((int(n), hidden), np.uint16) for n in counts]
    p_ids, k1 = _ptrs(ids)
    p_eo, k2 = _ptrs(eo)
    p_out, k3 = _ptrs(out)
    rc = lib().oracle_combine(ep, num_experts, top_k, hidden, tokens_per_rank,
                              int(bool(mask_enabled)), active_rank_mask & ((1 << 64) - 1),
                              counts.ctypes.data, _voidp(p_ids), _voidp(p_eo), _voidp(p_out))
    if rc != 0:
        raise ValueError("oracle_combine: inconsistent sizes")
    return out


def identity_expert(ep_size: int, num_experts: int, top_k: int, hidden: int, elem_bytes: int,
                    tokens_per_rank: int, disp: OracleDispatch) -> List[np.ndarray]:
    """bf16 bits [ep*T, hidden] per rank: received rows times their owned weights."""
    ep, rows = ep_size, ep_size * tokens_per_rank
    G = disp.recv_scale[0].shape[1] if disp.recv_scale is not None else 0
    eo = [np.zeros((rows, hidden), np.uint16) for _ in range(ep)]
    p_rh, k1 = _ptrs(disp.recv_hidden)
    p_rs, k2 = _ptrs(disp.recv_scale)
    p_ri, k3 = _ptrs(disp.recv_ids)
    p_rw, k4 = _ptrs(disp.recv_weights)
    p_eo, k5 = _ptrs(eo)
    rc = lib().oracle_identity_expert(ep, num_experts, top_k, hidden, elem_bytes,
                                      G if elem_bytes == 1 else 0, tokens_per_rank,
                                      _voidp(p_rh), _voidp(p_rs), _voidp(p_ri), _voidp(p_rw),
                                      _voidp(p_eo))
    if rc != 0:
        raise ValueError("oracle_identity_expert: inconsistent sizes")
    return eo


def eplb_gather(local: Sequence) -> np.ndarray:
    """uint8 [ep, bytes]: row r = rank r's statistics bytes (see ep_oracle.c)."""
    arrs = [np.ascontiguousarray(_np(x)).view(np.uint8).reshape(-1) for x in local]
    nbytes = arrs[0].size
    out = np.zeros((len(arrs), nbytes), np.uint8)
    p_loc, k = _ptrs(arrs)
    if lib().oracle_eplb_gather(len(arrs), nbytes, _voidp(p_loc), out.ctypes.data) != 0:
        raise ValueError("oracle_eplb_gather: inconsistent sizes")
    return out


COMBINE_DTYPES = {"bf16": (0, np.uint16), "fp16": (2, np.uint16), "fp32": (3, np.float32)}


def combine_typed(ep_size: int, num_experts: int, top_k: int, hidden: int, tokens_per_rank: int,
                  num_tokens: Sequence[int], topk_ids: Sequence, expert_output: Sequence, dtype: str, *,
                  mask_enabled: bool = False, active_rank_mask: int = (1 << 64) - 1) -> List[np.ndarray]:
    """combine() with expert outputs and results stored as ``dtype`` ("bf16",
    "fp16" or "fp32"); returns raw bits (uint16) or float32 arrays [n_s, hidden]."""
    code, npt = COMBINE_DTYPES[dtype]
    counts = np.ascontiguousarray(np.asarray(num_tokens, dtype=np.int32))
    ids = [_np(i, np.int32) for i in topk_ids]
    eo = [np.ascontiguousarray(_np(e)).view(npt) for e in expert_output]
    out = [np.zeros((int(n), hidden), npt) for n in counts]
    p_ids, k1 = _ptrs(ids)
    p_eo, k2 = _ptrs(eo)
    p_out, k3 = _ptrs(out)
    rc = lib().oracle_combine_typed(ep_size, num_experts, top_k, hidden, tokens_per_rank,
                                    int(bool(mask_enabled)), active_rank_mask & ((1 << 64) - 1),
                                    counts.ctypes.data, _voidp(p_ids), code, _voidp(p_eo), _voidp(p_out))
    if rc != 0:
        raise ValueError("oracle_combine_typed: inconsistent sizes")
    return out
