"""PyTorch binding of the C ABI (include/ep.h): argument marshalling only.

Mirrors FlashInfer's ``MoEEpCommunication`` / ``NVLinkOneSidedAlltoAll``
interface (pages "flashinfer.moe_ep.MoEEpCommunication" and
"flashinfer.moe_ep.NVLinkOneSidedAlltoAll": ``is_platform_supported``,
``dispatch``, ``combine``, ``get_combine_input_buffer``, ``active_rank_mask``,
``destroy``) for an EP group whose ``ep_size`` ranks are virtual ranks on one
GPU. Every per-rank argument is a list with one tensor per rank; every
result is a list with one tensor per rank (per rank of the communicator's
partition, for a partitioned group). All work runs in the CUDA library
on torch's current stream; torch supplies device memory and streams only.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import _lib
from ._lib import ALL_RANKS, EpError, check

_DTYPES = {torch.bfloat16: _lib.EP_DTYPE_BF16, torch.float8_e4m3fn: _lib.EP_DTYPE_FP8_E4M3,
           torch.float16: _lib.EP_DTYPE_FP16, torch.float32: _lib.EP_DTYPE_FP32}
_COMBINE_DTYPES = (torch.bfloat16, torch.float16, torch.float32)


@dataclass
class EpDispatchResult:
    """Receive buffers of every rank after one dispatch (MoEEpDispatchResult).

    ``hidden_states[d]`` is rank d's ``[ep_size*tokens_per_rank, hidden]``
    receive buffer; row ``s*tokens_per_rank + t`` is token t of source rank s.
    Rows of tokens not routed to d, and padding rows, carry ``topk_ids`` of
    all -1; only their id rows are defined. The tensors view the handle's
    workspace: valid until destroy(), overwritten by the next dispatch().
    """

    tokens_per_rank: int
    hidden_states: List[torch.Tensor]
    hidden_states_scale: Optional[List[torch.Tensor]]
    topk_ids: List[torch.Tensor]
    topk_weights: Optional[List[torch.Tensor]]
    # every rank's eplb_local_stats stacked, [ep_size, *stats shape]; one
    # tensor shared by all virtual ranks (treat as read-only), or None
    eplb_global_stats: Optional[torch.Tensor] = None


# The pages name dispatch()'s result type MoEEpDispatchResult.
MoEEpDispatchResult = EpDispatchResult


def _mask_value(m) -> int:
    if m is None:
        return ALL_RANKS
    if isinstance(m, torch.Tensor):
        if m.numel() != 1:
            raise ValueError("active_rank_mask must hold one uint64")
        return int(m.reshape(-1)[0].item()) & ALL_RANKS
    return int(m) & ALL_RANKS


def _addr_array(ptrs) -> np.ndarray:
    """Device addresses as a host uint64 array: the layout of the C ABI's
    arrays of per-rank pointers (0 = NULL) on 64-bit hosts."""
    return np.array([int(p) if p else 0 for p in ptrs], dtype=np.uint64)


def _data(a) -> Optional[int]:
    return None if a is None else a.ctypes.data


def _stream_ptr(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


class EpComm:
    """Rank-major MoE EP dispatch/combine over ``ep_size`` virtual ranks.

    ``dtype`` is the hidden payload type: ``torch.bfloat16``,
    ``torch.float8_e4m3fn`` (fp8 rows usually travel with fp32 scales),
    ``torch.float16`` or ``torch.float32``. ``scale_cols`` is the number of
    fp32 scales per row (default hidden/128 when that divides, else none).
    ``eplb_stats_max_bytes`` reserves room to all-gather that many bytes of
    ``eplb_local_stats`` per rank. ``combine_dtype`` (bf16, fp16 or fp32)
    is the type of the expert outputs combine sums and of its results.
    ``pdl`` launches the kernels with programmatic dependent launch
    (``EP_LAUNCH_PDL``): a combine queued right after its dispatch is
    scheduled while the dispatch drains; results are unchanged. The
    workspace is allocated here with torch, at capacity
    ``max_tokens_per_rank``.

    ``num_partitions`` G > 1 makes this communicator partition ``partition``
    of a partitioned group: it hosts ranks ``first_rank ..
    first_rank+num_ranks-1`` (``num_ranks = ep_size // G``) in a workspace of
    its own, takes per-rank arguments for those ranks only (entry j is rank
    first_rank + j) and must be connected with every partition of the group
    (``connect`` / ``connect_partitions``) before its first dispatch. Its
    combine reads every rank's combine input, wherever it lives.

    Different communicators may be used from different threads at once; one
    communicator must not (it holds the state of its pending dispatch).
    """

    def __init__(self, ep_size: int, num_experts: int, top_k: int, hidden: int,
                 max_tokens_per_rank: int, dtype: torch.dtype = torch.bfloat16,
                 enable_rank_mask: bool = False, device=None, scale_cols: Optional[int] = None,
                 eplb_stats_max_bytes: int = 0, combine_dtype: torch.dtype = torch.bfloat16,
                 pdl: bool = False, num_partitions: int = 1, partition: int = 0):
        self._L = _lib.load()
        if dtype not in _DTYPES:
            raise ValueError(f"dtype {dtype} not supported (bfloat16, float8_e4m3fn, float16, float32)")
        self.ep_size, self.num_experts, self.top_k = int(ep_size), int(num_experts), int(top_k)
        self.hidden, self.max_tokens_per_rank = int(hidden), int(max_tokens_per_rank)
        self.dtype, self.enable_rank_mask = dtype, bool(enable_rank_mask)
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        self._h = None
        if scale_cols is None:
            scale_cols = self.hidden // _lib.EP_SCALE_GROUP if self.hidden % _lib.EP_SCALE_GROUP == 0 else 0
        self.scale_cols = int(scale_cols)
        self.eplb_stats_max_bytes = int(eplb_stats_max_bytes)
        if combine_dtype not in _COMBINE_DTYPES:
            raise ValueError(f"combine_dtype {combine_dtype} not supported (bfloat16, float16, float32)")
        self.combine_dtype = combine_dtype
        self.pdl = bool(pdl)
        self.num_partitions, self.partition = max(1, int(num_partitions)), int(partition)
        if self.ep_size % self.num_partitions or not 0 <= self.partition < self.num_partitions:
            raise ValueError(f"partition {partition} of {num_partitions} does not split ep_size={ep_size}")
        self.num_ranks = self.ep_size // self.num_partitions
        self.first_rank = self.partition * self.num_ranks
        cfg = _lib.EpConfigC(self.ep_size, self.num_experts, self.top_k, self.hidden,
                             self.max_tokens_per_rank, _DTYPES[dtype], int(self.enable_rank_mask),
                             self.scale_cols, self.eplb_stats_max_bytes, _DTYPES[combine_dtype],
                             _lib.EP_LAUNCH_PDL if self.pdl else 0, self.num_partitions, self.partition)
        self._cfg = cfg
        nbytes = ctypes.c_size_t(0)
        check(self._L.ep_workspace_size_ex(ctypes.byref(cfg), ctypes.byref(nbytes)))
        with torch.cuda.device(self.device):
            self._ws = torch.empty(nbytes.value, dtype=torch.uint8, device=self.device)
            h = ctypes.c_void_p()
            check(self._L.ep_create_ex(ctypes.byref(cfg), ctypes.c_void_p(self._ws.data_ptr()),
                                       nbytes.value, ctypes.byref(h)))
        self._h = h
        self._counts: Optional[List[int]] = None
        self._T = 0
        self._stacked = False
        self._dev_index = self.device.index if self.device.index is not None else torch.cuda.current_device()
        self._views = {}  # (kind, T) -> per-rank views of the workspace
        self._peer_ws = None  # peers' workspaces mapped into this process (connect_across_processes)

    # -- MoEEpCommunication.is_platform_supported ---------------------------
    @classmethod
    def is_platform_supported(cls) -> bool:
        if not torch.cuda.is_available():
            return False
        return bool(_lib.load().ep_is_supported())

    # -- NVLinkOneSidedAlltoAll.active_rank_mask ----------------------------
    @staticmethod
    def active_rank_mask(active_ranks: Sequence[int]) -> torch.Tensor:
        """CPU uint64 bit mask of ``active_ranks``."""
        arr = (ctypes.c_int * len(active_ranks))(*[int(r) for r in active_ranks])
        m = _lib.load().ep_rank_mask(arr, len(active_ranks))
        return torch.tensor([m], dtype=torch.uint64)

    def _view(self, ptr: int, rows: int, cols: int, dtype: torch.dtype) -> torch.Tensor:
        off = int(ptr) - self._ws.data_ptr()
        nbytes = rows * cols * torch.empty((), dtype=dtype).element_size()
        return self._ws[off:off + nbytes].view(dtype).view(rows, cols)

    def _live(self):
        if self._h is None:
            raise EpError(_lib.EP_ERR_STATE, "the communicator was destroyed")

    def _check_rank_tensor(self, name, t, s, n, cols, dtype, rows_any_shape=False):
        """A per-rank operand: contiguous [n, cols] of `dtype` on the device. With
        rows_any_shape, [n, *] whose trailing dimensions hold `cols` elements per
        row (the pages give hidden_states and its scales as [local_num_tokens, *])."""
        if t.dtype is not dtype or not t.is_cuda or t.get_device() != self._dev_index:
            raise ValueError(f"{name}[{s}] is {t.dtype} on {t.device}, expected {dtype} on {self.device}")
        if rows_any_shape and t.dim() >= 2 and t.shape[0] == n and t.numel() == n * cols and t.is_contiguous():
            return
        if t.shape != (n, cols) or not t.is_contiguous():
            raise ValueError(f"{name}[{s}] must be a contiguous [{n}, {cols}] tensor, got "
                             f"{tuple(t.shape)}")

    # -- partitioned groups (C ABI ep_partition_*) ----------------------------
    def partition_info(self) -> "_lib.EpPartitionInfoC":
        """This communicator's partition as its peers see it (ep_partition_describe)."""
        self._live()
        info = _lib.EpPartitionInfoC()
        check(self._L.ep_partition_describe(ctypes.byref(self._cfg), ctypes.c_void_p(self._ws.data_ptr()),
                                            self._ws.numel(), ctypes.byref(info)))
        return info

    def connect(self, infos: Sequence["_lib.EpPartitionInfoC"]) -> None:
        """Connect with every partition of the group (``infos`` in partition
        order, this one's included): ep_partition_connect."""
        self._live()
        arr = (_lib.EpPartitionInfoC * len(infos))(*infos)
        check(self._L.ep_partition_connect(self._h, arr, len(infos)))

    def connect_across_processes(self, group=None) -> None:
        """Connect with every partition of the group when each partition lives
        in a process of its own (one per partition, on this GPU or on GPUs that
        can map each other's memory) of a torch.distributed ``group``: the
        workspaces are shared as CUDA IPC handles (the way torch.multiprocessing
        shares CUDA tensors), every peer's is mapped into this process, and the
        descriptions are gathered and checked (gather_partition_infos). The
        mapped peer workspaces are held until destroy(); every process must keep
        its communicator alive until all of them are done with it (e.g. a
        barrier before destroy())."""
        import pickle
        from multiprocessing.reduction import ForkingPickler

        import torch.distributed as dist
        self._live()
        world = dist.get_world_size(group)
        mine = (self.partition, bytes(ForkingPickler.dumps(self._ws)))
        gathered = [None] * world
        dist.all_gather_object(gathered, mine, group=group)
        self._peer_ws = {p: pickle.loads(b) for p, b in gathered if p != self.partition}
        infos = gather_partition_infos(self.partition_info(), group,
                                       addresses={p: t.data_ptr() for p, t in self._peer_ws.items()})
        self.connect(infos)

    def _check_stacked(self, name, t, M, cols, dtype):
        """Checks one stacked operand, [num_ranks, M, cols] (M from the tensor when
        None); returns M."""
        ep = self.num_ranks
        if not isinstance(t, torch.Tensor) or t.dim() != 3 or t.shape[0] != ep or t.shape[2] != cols \
                or (M is not None and t.shape[1] != M):
            want = f"[{ep}, {'M' if M is None else M}, {cols}]"
            got = tuple(t.shape) if isinstance(t, torch.Tensor) else type(t).__name__
            raise ValueError(f"{name} must be a stacked {want} tensor like hidden_states, got {got}")
        if t.dtype is not dtype or not t.is_cuda or t.get_device() != self._dev_index or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dtype} tensor on {self.device}")
        return int(t.shape[1])

    @staticmethod
    def _stacked_ptrs(t, M, cols):
        """Device addresses of every rank's rows in a stacked [ep_size, M, cols] tensor."""
        step = np.uint64(M * cols * t.element_size())
        return np.uint64(t.data_ptr()) + step * np.arange(t.shape[0], dtype=np.uint64)

    def _rank_views(self, kind, ptrs, T, cols, dtype):
        key = (kind, T)
        v = self._views.get(key)
        if v is None:
            rows = self.ep_size * T
            v = [self._view(ptrs[j], rows, cols, dtype) for j in range(self.num_ranks)]
            self._views[key] = v
        return list(v)

    # -- MoEEpCommunication.dispatch ----------------------------------------
    def dispatch(self, hidden_states, topk_ids, topk_weights=None, *,
                 hidden_states_scale=None,
                 runtime_max_tokens_per_rank: Optional[int] = None,
                 eplb_local_stats: Optional[Sequence[torch.Tensor]] = None,
                 active_rank_mask=None,
                 num_tokens_device: Optional[torch.Tensor] = None,
                 num_tokens: Optional[Sequence[int]] = None) -> EpDispatchResult:
        """Scatter each rank's tokens to the ranks holding one of their top-k experts.

        Per rank s (of the communicator's ranks: all ``ep_size`` of them, or
        a partition's ``num_ranks``, entry j being rank ``first_rank + j``):
        ``hidden_states[s]`` [n_s, hidden] (dtype of the
        communicator), ``topk_ids[s]`` int32 [n_s, top_k], optional
        ``topk_weights[s]`` fp32 [n_s, top_k] and ``hidden_states_scale[s]``
        fp32 [n_s, scale_cols]. Weights and scales are all-or-none over ranks.
        Hidden rows and scale rows may also come as [n_s, *] with that many
        elements per row (e.g. [n_s, heads, head_dim]).
        ``eplb_local_stats[s]`` (optional, every rank the same dtype and shape,
        a multiple of 4 bytes) is gathered into ``eplb_global_stats``.

        Stacked form: every operand may instead be one contiguous tensor with
        all ranks' rows, ``hidden_states`` [ep_size, M, hidden], ``topk_ids``
        [ep_size, M, top_k] and so on, and ``num_tokens`` (default M for every
        rank) gives each rank's count n_s <= M. One tensor is checked per
        operand instead of one per rank, so a call costs far less host time
        at large ep_size; the results are the same.

        ``num_tokens_device`` (optional, int32 CUDA tensor of ``ep_size``
        counts) is read by the kernels when they run: rank s then has
        ``min(max(num_tokens_device[s], 0), n_s)`` tokens, ``n_s`` (the row
        count of its tensors) being its maximum. For CUDA graphs whose token
        counts change between replays; the following combine() writes only
        the first count rows of each output.
        """
        self._live()
        ep, K, H = self.num_ranks, self.top_k, self.hidden  # ep: source ranks of this communicator
        G = self.scale_cols
        stacked = isinstance(hidden_states, torch.Tensor)
        if stacked:
            M = self._check_stacked("hidden_states", hidden_states, None, H, self.dtype)
            if num_tokens is None:
                counts = [M] * ep
            else:
                counts = [int(n) for n in num_tokens]
                if len(counts) != ep or any(n < 0 or n > M for n in counts):
                    raise ValueError(f"num_tokens needs {ep} counts in [0, {M}] (the stacked tensors' rows)")
            self._check_stacked("topk_ids", topk_ids, M, K, torch.int32)
            for name, t, cols in (("topk_weights", topk_weights, K), ("hidden_states_scale", hidden_states_scale, G)):
                if t is not None:
                    self._check_stacked(name, t, M, cols, torch.float32)
            hp = self._stacked_ptrs(hidden_states, M, H)
            ip = self._stacked_ptrs(topk_ids, M, K)
            wp = self._stacked_ptrs(topk_weights, M, K) if topk_weights is not None else None
            sp = self._stacked_ptrs(hidden_states_scale, M, G) if hidden_states_scale is not None else None
        else:
            if num_tokens is not None:
                raise ValueError("num_tokens goes with stacked tensors; per-rank tensors give their counts by shape")
            if len(hidden_states) != ep or len(topk_ids) != ep:
                raise ValueError(f"hidden_states and topk_ids need {ep} per-rank tensors")
            for name, lst in (("topk_weights", topk_weights), ("hidden_states_scale", hidden_states_scale)):
                if lst is not None and (len(lst) != ep or any(x is None for x in lst)):
                    raise ValueError(f"{name}: every rank passes it or none does "
                                     "(an empty rank passes an empty tensor)")
            counts = [int(x.shape[0]) for x in hidden_states]
            for s in range(ep):
                n = counts[s]
                self._check_rank_tensor("hidden_states", hidden_states[s], s, n, H, self.dtype, True)
                self._check_rank_tensor("topk_ids", topk_ids[s], s, n, K, torch.int32)
                if topk_weights is not None:
                    self._check_rank_tensor("topk_weights", topk_weights[s], s, n, K, torch.float32)
                if hidden_states_scale is not None:
                    self._check_rank_tensor("hidden_states_scale", hidden_states_scale[s], s, n, G,
                                            torch.float32, True)
            hp = _addr_array([x.data_ptr() for x in hidden_states])
            ip = _addr_array([x.data_ptr() for x in topk_ids])
            wp = _addr_array([x.data_ptr() for x in topk_weights]) if topk_weights is not None else None
            sp = _addr_array([x.data_ptr() for x in hidden_states_scale]) if hidden_states_scale is not None else None
        eplb_ptrs, eplb_bytes, eplb_meta = None, 0, None
        if eplb_local_stats is not None:
            if len(eplb_local_stats) != ep or any(x is None for x in eplb_local_stats):
                raise ValueError("eplb_local_stats: every rank passes its statistics")
            first = eplb_local_stats[0]
            for s, x in enumerate(eplb_local_stats):
                if x.dtype is not first.dtype or x.shape != first.shape or not x.is_contiguous() \
                        or not x.is_cuda or x.get_device() != self._dev_index:
                    raise ValueError(f"eplb_local_stats[{s}] must be a contiguous {first.dtype} "
                                     f"{tuple(first.shape)} tensor on {self.device}")
            eplb_bytes = first.numel() * first.element_size()
            eplb_ptrs = _addr_array([x.data_ptr() for x in eplb_local_stats])
            eplb_meta = (first.dtype, tuple(first.shape))
        dev_counts_ptr = None
        if num_tokens_device is not None:
            t = num_tokens_device
            if t.dtype is not torch.int32 or not t.is_cuda or t.get_device() != self._dev_index \
                    or t.numel() != ep or not t.is_contiguous():
                raise ValueError(f"num_tokens_device must be a contiguous int32 tensor of {ep} counts "
                                 f"on {self.device}")
            dev_counts_ptr = t.data_ptr()
        c_counts = np.array(counts, dtype=np.int32)
        res = _lib.EpDispatchResultC()
        rt = -1 if runtime_max_tokens_per_rank is None else int(runtime_max_tokens_per_rank)
        if rt < -1:
            raise ValueError("runtime_max_tokens_per_rank must be >= 0")
        args = _lib.EpDispatchArgsC(_data(hp), _data(sp), _data(ip), _data(wp), _data(c_counts), rt,
                                    _mask_value(active_rank_mask), _data(eplb_ptrs), eplb_bytes,
                                    dev_counts_ptr)
        with torch.cuda.device(self.device):
            st = self._L.ep_dispatch_ex(self._h, ctypes.byref(args),
                                        ctypes.c_void_p(_stream_ptr(self.device)), ctypes.byref(res))
        if st == _lib.EP_ERR_DEVICE_CHECK:  # checked build: the dispatch happened; keep its state
            self._counts, self._T, self._stacked = counts, res.tokens_per_rank, stacked
        check(st)
        T = res.tokens_per_rank
        self._counts, self._T = counts, T
        self._stacked = stacked
        hs = self._rank_views("hidden", res.recv_hidden, T, H, self.dtype)
        ids = self._rank_views("ids", res.recv_topk_ids, T, K, torch.int32)
        sc = self._rank_views("scale", res.recv_scale, T, G, torch.float32) if res.recv_scale else None
        w = self._rank_views("weights", res.recv_topk_weights, T, K, torch.float32) \
            if res.recv_topk_weights else None
        stats = None
        if eplb_meta is not None:
            n = self.ep_size  # every rank's statistics, this partition's and its peers'
            off = int(res.eplb_global_stats) - self._ws.data_ptr()
            stats = self._ws[off:off + n * eplb_bytes].view(eplb_meta[0]).view((n,) + eplb_meta[1])
        return EpDispatchResult(T, hs, sc, ids, w, stats)

    # -- MoEEpCommunication.get_combine_input_buffer ------------------------
    def get_combine_input_buffer(self, dtype: Optional[torch.dtype] = None, *,
                                 rank: Optional[int] = None):
        """Rank ``rank``'s [ep_size*tokens_per_rank, hidden] combine input of
        the communicator's combine dtype (all of its ranks as a list when
        ``rank`` is None); None when ``dtype`` names another type (no such
        buffer). Usable from a dispatch() until the combine() that follows it."""
        self._live()
        if dtype is not None and dtype != self.combine_dtype:
            return None
        ranks = range(self.first_rank, self.first_rank + self.num_ranks) if rank is None else [int(rank)]
        out = []
        for r in ranks:
            p = ctypes.c_void_p()
            check(self._L.ep_get_combine_input_buffer(self._h, r, ctypes.byref(p)))
            key = ("combine_in", r, self._T)
            v = self._views.get(key)
            if v is None:
                v = self._views[key] = self._view(p.value, self.ep_size * self._T, self.hidden,
                                                  self.combine_dtype)
            out.append(v)
        return out if rank is None else out[0]

    # -- MoEEpCommunication.combine -----------------------------------------
    def combine(self, expert_output=None, *, output=None, active_rank_mask=None):
        """Per source rank, [n_s, hidden] of the combine dtype: the sum over
        the ranks each token was routed to (ascending, fp32, one rounding) of
        their expert_output rows.

        ``expert_output[d]`` is rank d's [ep_size*tokens_per_rank, hidden] (or
        [ep_size, tokens_per_rank, hidden]) tensor of the combine dtype; None,
        or a None entry, means the backend combine input buffer (no copy).
        It may also be one stacked tensor of all ranks' rows,
        [ep_size, ep_size*tokens_per_rank, hidden]. ``output`` may be a list
        of [n_s, hidden] tensors or one stacked [ep_size, M, hidden] tensor
        with M >= every n_s; after a stacked dispatch the default output is
        one such tensor. The result is the list of per-rank [n_s, hidden]
        tensors, or the stacked output itself (rank s's result in its first
        n_s rows; the rows past them are not written)."""
        self._live()
        ep, H = self.ep_size, self.hidden
        nr = self.num_ranks  # source ranks of this communicator (outputs)
        if self._counts is None:
            raise EpError(_lib.EP_ERR_STATE, "combine called without a pending dispatch")
        rows = ep * self._T
        eo_ptrs = None
        if isinstance(expert_output, torch.Tensor):
            e = expert_output
            if e.dtype is not self.combine_dtype or not e.is_cuda or e.get_device() != self._dev_index \
                    or not e.is_contiguous() or e.shape[0] != ep or e.numel() != ep * rows * H or e.shape[-1] != H:
                raise ValueError(f"a stacked expert_output must be a contiguous {self.combine_dtype} "
                                 f"[{ep}, {rows}, {H}] tensor on {self.device}")
            eo_ptrs = self._stacked_ptrs(e, rows, H)
        elif expert_output is not None:
            if len(expert_output) != ep:
                raise ValueError(f"expert_output needs {ep} per-rank tensors")
            eo_ptrs = []
            for d, e in enumerate(expert_output):
                if e is None:
                    eo_ptrs.append(0)
                    continue
                if e.dtype is not self.combine_dtype or not e.is_cuda or e.get_device() != self._dev_index \
                        or not e.is_contiguous() or e.numel() != rows * H or e.shape[-1] != H:
                    raise ValueError(f"expert_output[{d}] must be contiguous {self.combine_dtype} "
                                     f"[{rows}, {H}] on {self.device}")
                eo_ptrs.append(e.data_ptr())
            eo_ptrs = _addr_array(eo_ptrs)
        if output is None and self._stacked:
            output = torch.empty(nr, max(self._counts, default=0), H, dtype=self.combine_dtype,
                                 device=self.device)
        if isinstance(output, torch.Tensor):
            o = output
            if o.dim() != 3 or o.shape[0] != nr or o.shape[2] != H or o.shape[1] < max(self._counts, default=0) \
                    or o.dtype is not self.combine_dtype or not o.is_cuda or o.get_device() != self._dev_index \
                    or not o.is_contiguous():
                raise ValueError(f"a stacked output must be a contiguous {self.combine_dtype} [{nr}, M, {H}] "
                                 f"tensor on {self.device} with M >= {max(self._counts, default=0)}")
            out_ptrs = self._stacked_ptrs(o, int(o.shape[1]), H)
        else:
            if output is None:
                output = [torch.empty(n, H, dtype=self.combine_dtype, device=self.device) for n in self._counts]
            else:
                if len(output) != nr:
                    raise ValueError(f"output needs {nr} per-rank tensors")
                for s in range(nr):
                    self._check_rank_tensor("output", output[s], s, self._counts[s], H, self.combine_dtype)
            out_ptrs = _addr_array([o.data_ptr() for o in output])
        with torch.cuda.device(self.device):
            st = self._L.ep_combine(self._h, _data(eo_ptrs), _data(out_ptrs), _mask_value(active_rank_mask),
                                    ctypes.c_void_p(_stream_ptr(self.device)))
        if st == _lib.EP_ERR_DEVICE_CHECK:  # checked build: the combine happened
            self._counts = None
        check(st)
        self._counts = None
        return output if isinstance(output, torch.Tensor) else list(output)

    # -- MoEEpCommunication.destroy -----------------------------------------
    def destroy(self) -> None:
        """Release the handle and workspace; calling it again does nothing."""
        if self._h is None:
            return
        torch.cuda.synchronize(self.device)
        check(self._L.ep_destroy(self._h))
        self._h = None
        self._views = {}
        self._ws = None
        self._peer_ws = None

    def __del__(self):
        try:
            if getattr(self, "_h", None) is not None:
                # work queued on any stream may still use the workspace, which
                # torch frees (and may hand out again) once this object is gone
                torch.cuda.synchronize(self.device)
                self._L.ep_destroy(self._h)
                self._h = None
        except Exception:
            pass


def connect_partitions(comms: Sequence[EpComm]) -> None:
    """Connects the communicators of every partition of one group, all in
    this process (``comms[p]`` is partition p)."""
    infos = [c.partition_info() for c in comms]
    for c in comms:
        c.connect(infos)


def gather_partition_infos(info: "_lib.EpPartitionInfoC", group=None,
                           addresses: Optional[dict] = None) -> List["_lib.EpPartitionInfoC"]:
    """All partitions' descriptions, in partition order, from one process per
    partition of a torch.distributed group: each process passes its own
    (``EpComm.partition_info()``). ``addresses`` maps a partition to the
    device address at which this process reaches that partition's workspace
    (a peer's memory mapped into this process); it replaces the address the
    owner reported. The result is checked with ep_partition_check, so every
    process learns of a mismatch in the group's configuration."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    gathered = [None] * world
    dist.all_gather_object(gathered, bytes(info), group=group)
    infos = sorted((_lib.EpPartitionInfoC.from_buffer_copy(b) for b in gathered),
                   key=lambda x: x.config.partition)
    for x in infos:
        if addresses and x.config.partition in addresses:
            x.workspace = int(addresses[x.config.partition])
    arr = (_lib.EpPartitionInfoC * len(infos))(*infos)
    check(_lib.load().ep_partition_check(arr, len(infos)))
    return infos


def combine_noalloc(num_experts: int, top_k: int, topk_ids: Sequence[torch.Tensor],
                    expert_output: Sequence[torch.Tensor], output: Sequence[torch.Tensor], *,
                    tokens_per_rank: int, active_rank_mask=None) -> List[torch.Tensor]:
    """The combine without a communicator and without any device allocation
    (C ABI ep_combine_noalloc): for callers that may not allocate where they
    combine. ``topk_ids[s]`` int32 [n_s, top_k] are the ids the dispatch
    routed; ``expert_output[d]`` bf16 [ep_size*tokens_per_rank, hidden];
    ``output[s]`` bf16 [n_s, hidden], written in place and returned. The
    result equals EpComm.combine after EpComm.dispatch of the same ids and
    mask. Runs on torch's current stream of the tensors' device."""
    L = _lib.load()
    ep = len(topk_ids)
    if len(expert_output) != ep or len(output) != ep:
        raise ValueError("topk_ids, expert_output and output need one tensor per rank")
    counts = [int(x.shape[0]) for x in topk_ids]
    hidden = int(output[0].shape[-1]) if ep else 0
    dev = expert_output[0].device
    for name, lst, dtype, cols in (("topk_ids", topk_ids, torch.int32, top_k), ("output", output, torch.bfloat16, hidden)):
        for s, t in enumerate(lst):
            if t.dtype is not dtype or t.device != dev or not t.is_contiguous() or t.dim() != 2 or t.shape != (counts[s], cols):
                raise ValueError(f"{name}[{s}] must be a contiguous {dtype} [{counts[s]}, {cols}] tensor on {dev}")
    rows = ep * int(tokens_per_rank)
    for d, e in enumerate(expert_output):
        if e.dtype is not torch.bfloat16 or e.device != dev or not e.is_contiguous() or e.numel() != rows * hidden:
            raise ValueError(f"expert_output[{d}] must be a contiguous bf16 [{rows}, {hidden}] tensor on {dev}")
    ids = _addr_array([x.data_ptr() for x in topk_ids])
    eo = _addr_array([x.data_ptr() for x in expert_output])
    out = _addr_array([x.data_ptr() for x in output])
    c_counts = np.array(counts, dtype=np.int32)
    with torch.cuda.device(dev):
        check(L.ep_combine_noalloc(ep, int(num_experts), int(top_k), hidden, int(tokens_per_rank),
                                   _data(c_counts), _data(ids), _mask_value(active_rank_mask), _data(eo), _data(out),
                                   ctypes.c_void_p(_stream_ptr(dev))))
    return list(output)
