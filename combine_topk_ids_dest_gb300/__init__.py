"""GB300 (sm_103a) rank-major MoE expert-parallel dispatch/combine.

All ``ep_size`` ranks of an EP group are virtual ranks in one GPU's memory.
The work runs in hand-written CUDA kernels behind the C ABI of
``include/ep.h`` (``libep_gb300.so``); :class:`EpComm` is its PyTorch binding.
"""
from ._lib import (ALL_RANKS, EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3, EP_ERR_CUDA, EP_ERR_INVALID_ARG,
                   EP_ERR_OOM, EP_ERR_STATE, EP_ERR_UNSUPPORTED, EP_INVALID_EXPERT_ID,
                   EP_MAX_EP_SIZE, EP_MAX_TOP_K, EP_OK, EP_SCALE_GROUP, EXPORTS, EpError, load)
from .ep import (EpComm, EpDispatchResult, MoEEpDispatchResult, combine_noalloc, connect_partitions,
                 gather_partition_infos)

__all__ = ["EpComm", "EpDispatchResult", "MoEEpDispatchResult", "combine_noalloc", "connect_partitions",
           "gather_partition_infos", "EpError", "load", "EXPORTS", "ALL_RANKS",
           "EP_INVALID_EXPERT_ID", "EP_MAX_EP_SIZE", "EP_MAX_TOP_K", "EP_SCALE_GROUP", "EP_OK",
           "EP_ERR_INVALID_ARG", "EP_ERR_STATE", "EP_ERR_CUDA", "EP_ERR_OOM", "EP_ERR_UNSUPPORTED",
           "EP_DTYPE_BF16", "EP_DTYPE_FP8_E4M3"]
