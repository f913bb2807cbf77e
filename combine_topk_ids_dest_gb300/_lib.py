"""ctypes declarations of the C ABI in include/ep.h (libep_gb300.so).

Loading fails loudly: there is no fallback implementation of any operation.
With EP_GB300_CHECKED=1 in the environment the checked build
(libep_gb300_checked.so: every kernel access tested against its buffer,
EP_ERR_DEVICE_CHECK on a violation) is loaded instead.
"""
from __future__ import annotations

import ctypes
import os
import threading


EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_STATE = 2
EP_ERR_CUDA = 3
EP_ERR_OOM = 4
EP_ERR_UNSUPPORTED = 5
EP_ERR_DEVICE_CHECK = 6
STATUS_NAMES = {0: "EP_OK", 1: "EP_ERR_INVALID_ARG", 2: "EP_ERR_STATE", 3: "EP_ERR_CUDA",
                4: "EP_ERR_OOM", 5: "EP_ERR_UNSUPPORTED", 6: "EP_ERR_DEVICE_CHECK"}

# Access sites of the checked build (enum CheckSite in csrc/ep_internal.h).
CHECK_SITES = ("src_hidden", "src_ids", "src_scale", "src_weights", "recv_hidden", "recv_ids",
               "recv_scale", "recv_weights", "route_write", "eplb_src", "eplb_dst", "route_read",
               "combine_in", "combine_out", "noalloc_ids", "noalloc_route", "dev_counts", "live_counts")

EP_DTYPE_BF16 = 0
EP_DTYPE_FP8_E4M3 = 1
EP_DTYPE_FP16 = 2
EP_DTYPE_FP32 = 3
EP_SCALE_COLS_DEFAULT = -1
EP_LAUNCH_PDL = 1
EP_INVALID_EXPERT_ID = -1
EP_MAX_EP_SIZE = 64
EP_MAX_TOP_K = 32
EP_SCALE_GROUP = 128
ALL_RANKS = (1 << 64) - 1  # "no mask": every rank active

# Every symbol include/ep.h declares.
EXPORTS = ("ep_is_supported", "ep_workspace_size", "ep_create", "ep_create_with_workspace",
           "ep_dispatch", "ep_get_combine_input_buffer", "ep_combine", "ep_destroy",
           "ep_rank_mask", "ep_last_error", "ep_combine_noalloc", "ep_workspace_size_ex",
           "ep_create_ex", "ep_dispatch_ex", "ep_binary_version", "ep_partition_describe",
           "ep_partition_check", "ep_partition_connect", "ep_partition_info_of")
EP_NOALLOC_MAX_SLOTS = 65536


class EpDispatchResultC(ctypes.Structure):
    _fields_ = [("tokens_per_rank", ctypes.c_int),
                ("ep_size", ctypes.c_int),
                ("first_rank", ctypes.c_int),
                ("num_ranks", ctypes.c_int),
                ("recv_hidden", ctypes.POINTER(ctypes.c_void_p)),
                ("recv_scale", ctypes.POINTER(ctypes.c_void_p)),
                ("recv_topk_ids", ctypes.POINTER(ctypes.c_void_p)),
                ("recv_topk_weights", ctypes.POINTER(ctypes.c_void_p)),
                ("eplb_global_stats", ctypes.c_void_p),
                ("eplb_stats_bytes", ctypes.c_int)]


class EpConfigC(ctypes.Structure):
    _fields_ = [("ep_size", ctypes.c_int), ("num_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("hidden", ctypes.c_int), ("max_tokens_per_rank", ctypes.c_int), ("dtype", ctypes.c_int),
                ("enable_rank_mask", ctypes.c_int), ("scale_cols", ctypes.c_int),
                ("eplb_stats_max_bytes", ctypes.c_int), ("combine_dtype", ctypes.c_int),
                ("launch_flags", ctypes.c_int), ("num_partitions", ctypes.c_int), ("partition", ctypes.c_int)]


class EpPartitionInfoC(ctypes.Structure):
    """ep_partition_info: one partition of a partitioned EP group as its peers see it."""
    _fields_ = [("config", EpConfigC), ("first_rank", ctypes.c_int), ("num_ranks", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)] + \
        [(f, ctypes.c_size_t) for f in ("off_recv_hidden", "off_recv_scale", "off_recv_ids", "off_recv_weights",
                                         "off_combine_in", "off_eplb", "stride_recv_hidden", "stride_recv_scale",
                                         "stride_recv_ids", "stride_recv_weights", "stride_combine_in")]


class EpDispatchArgsC(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_void_p), ("hidden_scale", ctypes.c_void_p),
                ("topk_ids", ctypes.c_void_p), ("topk_weights", ctypes.c_void_p),
                ("num_tokens", ctypes.c_void_p), ("runtime_max_tokens_per_rank", ctypes.c_int),
                ("active_rank_mask", ctypes.c_uint64), ("eplb_local_stats", ctypes.c_void_p),
                ("eplb_stats_bytes", ctypes.c_int), ("num_tokens_device", ctypes.c_void_p)]


class EpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def checked() -> bool:
    """True when this process uses the checked build (EP_GB300_CHECKED=1)."""
    return os.environ.get("EP_GB300_CHECKED", "0") == "1"


def lib_path() -> str:
    from . import build as _build
    return _build.LIB_CHECKED if checked() else _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libep_gb300.so, or libep_gb300_checked.so under EP_GB300_CHECKED=1
    (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import build as _build
        path = lib_path()
        if build_if_missing:
            path = _build.build(checked=checked())
        if not os.path.exists(path):
            raise ImportError(f"CUDA library {path} is missing; run "
                              "`python -m combine_topk_ids_dest_gb300.build`")
        L = ctypes.CDLL(path)
        P, i32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
        PP = ctypes.POINTER(ctypes.c_void_p)
        L.ep_is_supported.argtypes = []
        L.ep_is_supported.restype = i32
        L.ep_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
        L.ep_workspace_size.restype = i32
        L.ep_create.argtypes = [i32, i32, i32, i32, i32, i32, i32, PP]
        L.ep_create.restype = i32
        L.ep_create_with_workspace.argtypes = [i32, i32, i32, i32, i32, i32, i32, P, sz, PP]
        L.ep_create_with_workspace.restype = i32
        L.ep_dispatch.argtypes = [P, P, P, P, P, P, i32, u64, P, ctypes.POINTER(EpDispatchResultC)]
        L.ep_dispatch.restype = i32
        L.ep_get_combine_input_buffer.argtypes = [P, i32, PP]
        L.ep_get_combine_input_buffer.restype = i32
        L.ep_combine.argtypes = [P, P, P, u64, P]
        L.ep_combine.restype = i32
        L.ep_destroy.argtypes = [P]
        L.ep_destroy.restype = i32
        L.ep_rank_mask.argtypes = [ctypes.POINTER(ctypes.c_int), i32]
        L.ep_rank_mask.restype = u64
        L.ep_workspace_size_ex.argtypes = [ctypes.POINTER(EpConfigC), ctypes.POINTER(sz)]
        L.ep_workspace_size_ex.restype = i32
        L.ep_create_ex.argtypes = [ctypes.POINTER(EpConfigC), P, sz, PP]
        L.ep_create_ex.restype = i32
        L.ep_dispatch_ex.argtypes = [P, ctypes.POINTER(EpDispatchArgsC), P,
                                     ctypes.POINTER(EpDispatchResultC)]
        L.ep_dispatch_ex.restype = i32
        L.ep_combine_noalloc.argtypes = [i32, i32, i32, i32, i32, P, P, u64, P, P, P]
        L.ep_combine_noalloc.restype = i32
        L.ep_binary_version.argtypes = [ctypes.POINTER(i32)]
        L.ep_binary_version.restype = i32
        L.ep_partition_describe.argtypes = [ctypes.POINTER(EpConfigC), P, sz, ctypes.POINTER(EpPartitionInfoC)]
        L.ep_partition_describe.restype = i32
        L.ep_partition_info_of.argtypes = [P, ctypes.POINTER(EpPartitionInfoC)]
        L.ep_partition_info_of.restype = i32
        L.ep_partition_check.argtypes = [ctypes.POINTER(EpPartitionInfoC), i32]
        L.ep_partition_check.restype = i32
        L.ep_partition_connect.argtypes = [P, ctypes.POINTER(EpPartitionInfoC), i32]
        L.ep_partition_connect.restype = i32
        L.ep_last_error.argtypes = []
        L.ep_last_error.restype = ctypes.c_char_p
        if checked():
            L.ep_checked_trim_extent.argtypes = [i32, ctypes.c_longlong]
            L.ep_checked_trim_extent.restype = i32
        _lib = L
        return L


def check(status: int) -> None:
    if status != EP_OK:
        msg = load().ep_last_error()
        raise EpError(status, msg.decode() if msg else "")


def ptr_array(ptrs) -> ctypes.Array:
    """Host array of device pointers (None/0 entries become NULL)."""
    return (ctypes.c_void_p * len(ptrs))(*[(int(p) if p else None) for p in ptrs])
