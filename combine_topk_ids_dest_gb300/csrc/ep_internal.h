// ep_internal.h -- kernel argument blocks and launchers shared by the C ABI
// (ep_host.cu) and the kernels (ep_kernels.cu). Not installed; not part of
// the public interface.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "ep.h"

#ifndef EP_CHECKED
#define EP_CHECKED 0
#endif

namespace epk {

constexpr int kMaxEp = EP_MAX_EP_SIZE;

// Checked build (EP_CHECKED=1, libep_gb300_checked.so): every global access
// of the kernels is tested against the extent of the buffer it belongs to
// (the extents the C ABI documents); an access outside is skipped and
// recorded, and the host turns the record into EP_ERR_DEVICE_CHECK. In the
// normal build the tests compile to nothing. Access sites, for the record:
enum CheckSite {
    kSiteSrcHidden = 0, kSiteSrcIds, kSiteSrcScale, kSiteSrcWeights,
    kSiteRecvHidden, kSiteRecvIds, kSiteRecvScale, kSiteRecvWeights,
    kSiteRouteWrite, kSiteEplbSrc, kSiteEplbDst,
    kSiteRouteRead, kSiteCombineIn, kSiteCombineOut,
    kSiteNoallocIds, kSiteNoallocRoute, kSiteDevCounts, kSiteLiveCounts,
    kNumSites
};

// What a checked launch needs: the device record {violations, first site,
// first offset (signed, bytes from the buffer's start), that buffer's
// extent in bytes}, and a test hook that declares one site's buffers
// `trim_bytes` shorter than they are.
struct CheckCtx {
    unsigned long long *rec;  // 4 entries, device; NULL in the normal build
    int trim_site;            // -1: none
    long long trim_bytes;
};

// Name of a check site, for messages.
const char *check_site_name(int site);

#if EP_CHECKED && defined(__CUDACC__)
// True when [p, p + nb) lies inside [lo, lo + extent) (the extent shortened
// by the test hook's trim at its site); otherwise records the access and
// returns false, so the caller skips it.
static __device__ __noinline__ bool in_bounds(const CheckCtx &c, int site, const void *p, int nb,
                                          const void *lo, long long extent)
{
    if (site == c.trim_site)
        extent -= c.trim_bytes;
    const long long off = static_cast<const char *>(p) - static_cast<const char *>(lo);
    if (off >= 0 && off + nb <= extent)
        return true;
    if (atomicAdd(&c.rec[0], 1ULL) == 0ULL) {
        c.rec[1] = static_cast<unsigned long long>(site);
        c.rec[2] = static_cast<unsigned long long>(off);
        c.rec[3] = static_cast<unsigned long long>(extent);
    }
    return false;
}
#define EP_IN_BOUNDS(ctx, site, p, nb, lo, extent) ::epk::in_bounds((ctx), (site), (p), (nb), (lo), (extent))
#else
#define EP_IN_BOUNDS(ctx, site, p, nb, lo, extent) true
#endif

// Everything one dispatch launch needs, passed by value as a __grid_constant__
// kernel parameter (5488 bytes; the combine's block is 1616), so no
// host->device copy precedes a launch and the launch can be captured in a
// CUDA graph as is.
//
// A launch handles the source ranks [src_first, src_first + n_src) of an EP
// group of `ep` ranks (all of them for an unpartitioned handle; one
// partition's ranks otherwise). Per-source arrays are indexed by the local
// source i (rank src_first + i); per-destination arrays by the global rank d.
struct DispatchArgs {
    const uint8_t *hidden[kMaxEp];  // local source i: [num_tokens[i], row_bytes]
    const float *scale[kMaxEp];     // [num_tokens[i], G] or unused
    const int32_t *ids[kMaxEp];     // [num_tokens[i], K]
    const float *weights[kMaxEp];   // [num_tokens[i], K] or unused
    int num_tokens[kMaxEp];         // tokens of local source i; with dev_counts, its maximum

    // Device-side counts (NULL: num_tokens is exact): local source i has
    // clamp(dev_counts[i], 0, num_tokens[i]) tokens; the kernel stores that
    // into live_counts[i] for the combine.
    const int32_t *dev_counts;
    int32_t *live_counts;

    // Destination rank d's receive buffers, wherever they live (this
    // handle's workspace or a connected partition's), each of ep*T rows with
    // row s*T + t for token t of global source rank s. The pointers are
    // advanced to row row0 = src_first*T, the first row of this launch's
    // sources, so own slot i*T + t indexes them directly.
    uint8_t *recv_hidden[kMaxEp];
    float *recv_scale[kMaxEp];
    int32_t *recv_ids[kMaxEp];
    float *recv_weights[kMaxEp];
    long long row0;

    uint64_t *route_mask;  // [n_src*T] destination-rank bit set of each own slot i*T + t
    uint64_t active;       // ranks allowed as destinations

    int ep, src_first, n_src, num_experts, experts_per_rank, top_k, T;
    int row_bytes;  // hidden row bytes, a multiple of 16
    int G;          // scale columns per row (0 when no scales are sent)
    int has_weights;

    // eplb_local_stats all-gather: local source i's eplb_bytes bytes -> row
    // src_first + i of every gathered buffer eplb_dst[p] ([ep][eplb_bytes],
    // one per partition, n_eplb_dst of them)
    const uint8_t *eplb_src[kMaxEp];
    uint8_t *eplb_dst[kMaxEp];
    int n_eplb_dst;
    int eplb_bytes;  // 0 = nothing to gather; else a multiple of 4

    CheckCtx chk;
};

struct CombineArgs {
    const void *eo[kMaxEp];  // global rank d's combine input, [ep*T, H] of ctype, advanced
                             // to row row0 = src_first*T (own slot i*T + t indexes it)
    long long row0;
    void *out[kMaxEp];       // local source i's output, [num_tokens[i], H] of ctype
    int num_tokens[kMaxEp];
    int token_offset[kMaxEp + 1];  // prefix sums of num_tokens: live token g of local source i
                                   // has token_offset[i] <= g < token_offset[i+1]
    const uint64_t *route_mask;    // [n_src*T], written by the dispatch
    const int32_t *live_counts;    // NULL, or [n_src] device counts the dispatch stored
                                   // (num_tokens are then maxima: rows past the count
                                   // are skipped)
    int ep, src_first, n_src, T, H;
    int ctype;  // element type of eo/out: EP_DTYPE_BF16, EP_DTYPE_FP16 or EP_DTYPE_FP32

    CheckCtx chk;
};

// Records `fmt` as the calling thread's ep_last_error() message (cleared for
// EP_OK) and returns `st`.
ep_status set_error(ep_status st, const char *fmt, ...);

// binaryVersion (compute capability major*10 + minor of the loaded code) of
// every dispatch and combine kernel instance, as cudaFuncGetAttributes reports
// it on the current device: up to `max` values into `out`, the number of
// kernels into *n. The no-alloc routing kernel reports through
// noalloc_binary_version.
cudaError_t kernel_binary_versions(int *out, int max, int *n);
cudaError_t noalloc_binary_version(int *out);

// Queue one launch on `stream`; returns the launch's cudaError_t. `pdl`:
// launch with programmatic dependent launch (EP_LAUNCH_PDL); the kernels
// wait for their predecessor with griddepcontrol.wait before touching global
// memory either way (a no-op without the launch attribute).
cudaError_t launch_dispatch(const DispatchArgs &a, cudaStream_t stream, bool pdl);
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t stream, bool pdl);

// Checked build: the CheckCtx for a launch recording into `rec`, with the
// test hook's trim applied; and, after the launch, EP_OK or
// EP_ERR_DEVICE_CHECK from the record (which is then cleared). `what` names
// the call for the message. Outside stream capture it synchronizes
// `stream`; during a capture it returns EP_OK and leaves the record for the
// next check. The normal build returns {NULL, -1, 0} and EP_OK.
CheckCtx check_ctx(unsigned long long *rec);
ep_status check_after(unsigned long long *rec, cudaStream_t stream, const char *what);

// Checked build: device address of the library's check record on the
// current device (one static record per device, shared by every handle and
// call); NULL on failure (ep_last_error set). The normal build returns NULL.
unsigned long long *check_record();

}  // namespace epk
