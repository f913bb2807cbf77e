// ep_noalloc.cu -- ep_combine_noalloc: a combine for callers that cannot
// allocate device memory.
//
// Some callers of this library may not call cudaMalloc (or any allocator)
// at the point where they combine: code inside a memory arena that owns all
// device memory after start-up, and plug-ins hosted by an inference runtime
// that forbids allocations of their own. They also may not hold an
// ep_handle, whose workspace is an allocation. This entry
// point needs neither: the caller passes the ids, the expert outputs and the
// result buffers, and the only scratch -- the destination-rank bit set of
// every slot -- lives in a file-scope __device__ array of fixed size that
// every GPU loading the library holds until the process exits.
//
// Host code never hands that array's name to a kernel (on the host it is a
// stand-in, not a device address): the first call on each device, with that
// device current, asks for the array's device address with
// cudaGetSymbolAddress and caches it; kernels receive that pointer. A small
// routing kernel fills the array from the ids; the sums are then made by the
// library's own combine kernel, which reads the routing from it.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ep_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Routing state of up to EP_NOALLOC_MAX_SLOTS source slots (512 KB).
static __device__ __align__(256) uint64_t g_noalloc_route[EP_NOALLOC_MAX_SLOTS];

std::mutex g_setup_mu;
void *g_route_ptr[kMaxDevices] = {nullptr};

// What the routing pass needs; the sums are computed by the library's
// combine kernel, reading the routing bit sets from the static array.
struct NoallocRouteArgs {
    const int32_t *ids[epk::kMaxEp];  // source rank s: [num_tokens[s], top_k]
    int num_tokens[epk::kMaxEp];
    uint64_t *route;                  // device address of g_noalloc_route
    uint64_t active;
    int ep, num_experts, experts_per_rank, top_k, T;
    epk::CheckCtx chk;
};

// One thread per slot s*T+t: the set of active ranks owning one of the
// token's valid expert ids (0 for padding slots). Every slot of the call is
// written, so nothing left by an earlier call is ever read.
__global__ void noalloc_route_kernel(const __grid_constant__ NoallocRouteArgs a)
{
    const long long n = (long long)a.ep * a.T;
    for (long long slot = (long long)blockIdx.x * blockDim.x + threadIdx.x; slot < n;
         slot += (long long)gridDim.x * blockDim.x) {
        const int s = (int)(slot / a.T);
        const int t = (int)(slot - (long long)s * a.T);
        uint64_t m = 0;
        if (t < a.num_tokens[s]) {
            const int32_t *row = a.ids[s] + (long long)t * a.top_k;
            for (int k = 0; k < a.top_k; ++k) {
                int e = -1;
                if (EP_IN_BOUNDS(a.chk, epk::kSiteNoallocIds, row + k, 4, a.ids[s],
                                 (long long)a.num_tokens[s] * a.top_k * 4))
                    e = row[k];
                if (e >= 0 && e < a.num_experts)
                    m |= 1ULL << (e / a.experts_per_rank);
            }
            m &= a.active;
        }
        if (EP_IN_BOUNDS(a.chk, epk::kSiteNoallocRoute, a.route + slot, 8, a.route,
                         (long long)EP_NOALLOC_MAX_SLOTS * 8))
            a.route[slot] = m;
    }
}

bool is_aligned(const void *p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// Device address of g_noalloc_route on the current device, looked up once
// per device (with that device current) and cached for the life of the
// process, on the assumption that the device's primary context lives as long
// as the process.
ep_status route_scratch(uint64_t **out)
{
    int dev = -1;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess)
        return epk::set_error(EP_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
    if (dev < 0 || dev >= kMaxDevices)
        return epk::set_error(EP_ERR_UNSUPPORTED, "device index %d is beyond %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_route_ptr[dev]) {
        if (!ep_is_supported())
            return epk::set_error(EP_ERR_UNSUPPORTED, "device %d is not compute capability 10.3", dev);
        void *p = nullptr;
        ce = cudaGetSymbolAddress(&p, g_noalloc_route);
        if (ce != cudaSuccess || !p) {
            cudaGetLastError();
            return epk::set_error(EP_ERR_CUDA, "cudaGetSymbolAddress of the routing scratch: %s",
                                  cudaGetErrorString(ce));
        }
        g_route_ptr[dev] = p;
    }
    *out = static_cast<uint64_t *>(g_route_ptr[dev]);
    return EP_OK;
}

int sm_count_here()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 152;
    return n;
}

}  // namespace

cudaError_t epk::noalloc_binary_version(int *out)
{
    cudaFuncAttributes attr;
    cudaError_t ce = cudaFuncGetAttributes(&attr, reinterpret_cast<const void *>(noalloc_route_kernel));
    if (ce == cudaSuccess)
        *out = attr.binaryVersion;
    return ce;
}

extern "C" ep_status ep_combine_noalloc(int ep_size, int num_experts, int top_k, int hidden,
                                        int tokens_per_rank, const int32_t *num_tokens,
                                        const int32_t *const *topk_ids, uint64_t active_rank_mask,
                                        const void *const *expert_output, void *const *output,
                                        void *stream)
{
    if (ep_size < 1 || ep_size > EP_MAX_EP_SIZE)
        return epk::set_error(EP_ERR_INVALID_ARG, "ep_size=%d outside [1, %d]", ep_size, EP_MAX_EP_SIZE);
    if (num_experts < ep_size || num_experts % ep_size)
        return epk::set_error(EP_ERR_INVALID_ARG, "num_experts=%d is not a positive multiple of ep_size=%d",
                              num_experts, ep_size);
    if (top_k < 1 || top_k > EP_MAX_TOP_K)
        return epk::set_error(EP_ERR_INVALID_ARG, "top_k=%d outside [1, %d]", top_k, EP_MAX_TOP_K);
    if (hidden < 8 || hidden % 8)
        return epk::set_error(EP_ERR_INVALID_ARG, "hidden=%d must be a positive multiple of 8", hidden);
    if (tokens_per_rank < 0)
        return epk::set_error(EP_ERR_INVALID_ARG, "tokens_per_rank=%d < 0", tokens_per_rank);
    if ((long long)ep_size * tokens_per_rank > EP_NOALLOC_MAX_SLOTS)
        return epk::set_error(EP_ERR_INVALID_ARG,
                              "ep_size*tokens_per_rank=%lld exceeds the %d routing slots of the "
                              "static scratch of ep_combine_noalloc",
                              (long long)ep_size * tokens_per_rank, EP_NOALLOC_MAX_SLOTS);
    if (!num_tokens || !topk_ids || !expert_output || !output)
        return epk::set_error(EP_ERR_INVALID_ARG,
                              "num_tokens, topk_ids, expert_output and output must not be NULL");
    const uint64_t full = ep_size >= 64 ? ~0ULL : ((1ULL << ep_size) - 1);
    uint64_t mask = active_rank_mask == ~0ULL ? full : active_rank_mask;
    if (mask & ~full)
        return epk::set_error(EP_ERR_INVALID_ARG, "active_rank_mask 0x%llx has bits at or above ep_size=%d",
                              (unsigned long long)mask, ep_size);

    NoallocRouteArgs a;
    std::memset(&a, 0, sizeof a);
    epk::CombineArgs c;
    std::memset(&c, 0, sizeof c);
    for (int d = 0; d < ep_size; ++d) {
        if (!expert_output[d] || !is_aligned(expert_output[d], 16))
            return epk::set_error(EP_ERR_INVALID_ARG, "expert_output[%d] is NULL or not 16-byte aligned", d);
        c.eo[d] = expert_output[d];
    }
    c.token_offset[0] = 0;
    for (int s = 0; s < ep_size; ++s) {
        const int n = num_tokens[s];
        if (n < 0 || n > tokens_per_rank)
            return epk::set_error(EP_ERR_INVALID_ARG, "num_tokens[%d]=%d outside [0, tokens_per_rank=%d]", s,
                                  n, tokens_per_rank);
        a.num_tokens[s] = c.num_tokens[s] = n;
        c.token_offset[s + 1] = c.token_offset[s] + n;
        if (n == 0)
            continue;
        if (!topk_ids[s] || !is_aligned(topk_ids[s], 4))
            return epk::set_error(EP_ERR_INVALID_ARG, "topk_ids[%d] is NULL or not 4-byte aligned", s);
        if (!output[s] || !is_aligned(output[s], 16))
            return epk::set_error(EP_ERR_INVALID_ARG, "output[%d] is NULL or not 16-byte aligned", s);
        a.ids[s] = topk_ids[s];
        c.out[s] = output[s];
    }
    uint64_t *route = nullptr;
    ep_status st = route_scratch(&route);
    if (st != EP_OK)
        return st;
    a.route = route;
    a.active = mask;
    a.ep = ep_size;
    a.num_experts = num_experts;
    a.experts_per_rank = num_experts / ep_size;
    a.top_k = top_k;
    a.T = tokens_per_rank;
    c.route_mask = route;
    c.ep = ep_size;
    c.row0 = 0;
    c.src_first = 0;
    c.n_src = ep_size;
    c.T = tokens_per_rank;
    c.H = hidden;
    c.ctype = EP_DTYPE_BF16;
    unsigned long long *rec = nullptr;
#if EP_CHECKED
    rec = epk::check_record();
    if (!rec)
        return EP_ERR_CUDA;
#endif
    a.chk = c.chk = epk::check_ctx(rec);

    const long long n_slots = (long long)ep_size * tokens_per_rank;
    if (n_slots == 0)
        return epk::set_error(EP_OK, "");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    long long route_blocks = (n_slots + 255) / 256;
    const long long cap = (long long)sm_count_here() * 8;
    if (route_blocks > cap)
        route_blocks = cap;
    noalloc_route_kernel<<<(unsigned)route_blocks, 256, 0, s>>>(a);
    cudaError_t ce = cudaGetLastError();
    if (ce != cudaSuccess)
        return epk::set_error(EP_ERR_CUDA, "ep_combine_noalloc routing launch: %s", cudaGetErrorString(ce));
    ce = epk::launch_combine(c, s, false);  // the library's combine, reading the static routing array
    if (ce != cudaSuccess)
        return epk::set_error(EP_ERR_CUDA, "ep_combine_noalloc combine launch: %s", cudaGetErrorString(ce));
    st = epk::check_after(rec, s, "ep_combine_noalloc");
    if (st != EP_OK)
        return st;
    return epk::set_error(EP_OK, "");
}
