// ep_internal.h -- kernel argument blocks and launchers shared by the C ABI
// (ep_host.cu) and the kernels (ep_kernels.cu). Not installed; not part of
// the public interface.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "ep.h"

namespace epk {

constexpr int kMaxEp = EP_MAX_EP_SIZE;

// Everything one dispatch launch needs, passed by value as a __grid_constant__
// kernel parameter (about 2.4 KB), so no host->device copy precedes a launch
// and the launch can be captured in a CUDA graph as is.
struct DispatchArgs {
    const uint8_t *hidden[kMaxEp];  // source rank s: [num_tokens[s], row_bytes]
    const float *scale[kMaxEp];     // [num_tokens[s], G] or unused
    const int32_t *ids[kMaxEp];     // [num_tokens[s], K]
    const float *weights[kMaxEp];   // [num_tokens[s], K] or unused
    int num_tokens[kMaxEp];

    // Destination rank d's receive buffer of each kind starts at base + d*stride
    // (strides in elements of the buffer's type); row r = s*T + t.
    uint8_t *recv_hidden;
    long long hidden_stride;
    float *recv_scale;
    long long scale_stride;
    int32_t *recv_ids;
    long long ids_stride;
    float *recv_weights;
    long long weights_stride;

    uint64_t *route_mask;  // [ep*T] destination-rank bit set of each slot
    uint64_t active;       // ranks allowed as destinations

    int ep, num_experts, experts_per_rank, top_k, T;
    int row_bytes;  // hidden row bytes, a multiple of 16
    int G;          // scale columns per row (0 when no scales are sent)
    int has_weights;

    // eplb_local_stats all-gather: rank r's eplb_bytes bytes -> eplb_dst + r*eplb_bytes
    const uint8_t *eplb_src[kMaxEp];
    uint8_t *eplb_dst;
    int eplb_bytes;  // 0 = nothing to gather; else a multiple of 4
};

struct CombineArgs {
    const void *eo[kMaxEp];  // rank d's combine input, [ep*T, H] of ctype
    void *out[kMaxEp];       // source rank s's output, [num_tokens[s], H] of ctype
    int num_tokens[kMaxEp];
    int token_offset[kMaxEp + 1];  // prefix sums of num_tokens: live token g of rank s has
                                   // token_offset[s] <= g < token_offset[s+1]
    const uint64_t *route_mask;    // [ep*T], written by the dispatch
    int ep, T, H;
    int ctype;  // element type of eo/out: EP_DTYPE_BF16, EP_DTYPE_FP16 or EP_DTYPE_FP32
};

// Records `fmt` as the calling thread's ep_last_error() message (cleared for
// EP_OK) and returns `st`.
ep_status set_error(ep_status st, const char *fmt, ...);

// Queue one launch on `stream`; returns the launch's cudaError_t.
cudaError_t launch_dispatch(const DispatchArgs &a, cudaStream_t stream);
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t stream);

}  // namespace epk
