// ep_host.cu -- the C ABI of include/ep.h: handle, workspace layout, argument
// and state checks, kernel launches.
//
// Contract followed (FlashInfer moe_ep pages):
//  - "flashinfer.moe_ep.MoEEpCommunication", class description: an instance
//    alternates dispatch() and combine(), one pair at a time.
//    dispatch(): runtime_max_tokens_per_rank may not exceed
//    max_tokens_per_rank and fixes tokens_per_rank (the capacity when not
//    given). get_combine_input_buffer(): usable from a dispatch() until its
//    combine(). destroy(): calling it again is harmless.
//  - "flashinfer.moe_ep.NVLinkOneSidedAlltoAll", dispatch(): a rank mask
//    needs a handle created with enable_rank_mask; weights come from all
//    ranks or from none (a rank without tokens sends an empty tensor).
//    combine(): its mask is the dispatch's. get_combine_input_buffer(): the
//    rank's combine-input region seen as [ep_size * tokens_per_rank, hidden].
//
// Workspace (one device allocation, regions 256-byte aligned, each sized at
// capacity C = max_tokens_per_rank), for the n ranks the handle hosts (all
// ep of them, or one partition's ep/G):
//   recv_hidden  [n][ep*C][row_bytes]
//   recv_scale   [n][ep*C][scale_cols] fp32  (scale_cols = H/128 by default)
//   recv_ids     [n][ep*C][K] int32
//   recv_weights [n][ep*C][K] fp32
//   combine_in   [n][ep*C][H] of the combine dtype (bf16 by default)
//   route_mask   [n*C] uint64  (routing state of the hosted source ranks' slots)
//   live_counts  [n] int32  (token counts of a dispatch with device-side counts)
//   eplb_stats   [ep][eplb_stats_max_bytes]  (the gathered eplb_local_stats)
// A step with tokens_per_rank T uses the first ep*T rows of each region, so
// receive row s*T+t of hosted rank j sits at region base + j*stride +
// (s*T+t)*row. The kernels reach every rank's regions, this workspace's or a
// connected partition's, through per-rank address tables held in the handle.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "ep_internal.h"

struct ep_handle {
    int ep, num_experts, top_k, hidden, capacity, experts_per_rank;
    ep_dtype dtype;
    int elem_bytes, row_bytes, scale_cols;
    ep_dtype combine_dtype;
    int mask_enabled;
    int eplb_max_bytes;
    bool pdl;  // EP_LAUNCH_PDL
    int device;
    ep_config cfg;  // as created

    // partition: hosted ranks [first, first + nloc) of num_parts (1: all ranks)
    int num_parts, part, first, nloc;
    bool connected;  // destination tables complete (always, unless partitioned)

    uint8_t *ws;
    size_t ws_bytes;
    bool owns_ws;
    size_t off_hidden, off_scale, off_ids, off_weights, off_comb, off_mask, off_counts, off_eplb;
    size_t st_hidden, st_scale, st_ids, st_weights, st_comb;  // bytes per rank region

    // state of the pending dispatch
    bool pending;
    bool dev_counts;  // its token counts are device-side (live_counts region)
    int T;
    uint64_t mask;
    int32_t counts[EP_MAX_EP_SIZE];

    // hosted ranks' receive buffers (entry j = rank first + j), for results
    void *r_hidden[EP_MAX_EP_SIZE];
    float *r_scale[EP_MAX_EP_SIZE];
    int32_t *r_ids[EP_MAX_EP_SIZE];
    float *r_weights[EP_MAX_EP_SIZE];

    // every rank's buffers by global rank, and each partition's eplb buffer
    uint8_t *t_hidden[EP_MAX_EP_SIZE];
    float *t_scale[EP_MAX_EP_SIZE];
    int32_t *t_ids[EP_MAX_EP_SIZE];
    float *t_weights[EP_MAX_EP_SIZE];
    void *t_comb[EP_MAX_EP_SIZE];
    uint8_t *t_eplb[EP_MAX_EP_SIZE];
};

namespace {

thread_local char g_err[512] = "";

ep_status fail(ep_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

ep_status ok()
{
    g_err[0] = '\0';
    return EP_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

uint64_t full_mask(int ep) { return ep >= 64 ? ~0ULL : ((1ULL << ep) - 1); }

struct Layout {
    int num_parts, part, first, nloc;  // partition and hosted ranks
    int elem_bytes, row_bytes, scale_cols, combine_elem;
    size_t off_hidden, off_scale, off_ids, off_weights, off_comb, off_mask, off_counts, off_eplb, total;
    size_t st_hidden, st_scale, st_ids, st_weights, st_comb;
};

int dtype_bytes(ep_dtype dtype)
{
    switch (dtype) {
    case EP_DTYPE_BF16:
    case EP_DTYPE_FP16:
        return 2;
    case EP_DTYPE_FP8_E4M3:
        return 1;
    case EP_DTYPE_FP32:
        return 4;
    }
    return 0;
}

ep_config default_config(int ep, int E, int K, int H, int C, ep_dtype dtype, int enable_rank_mask)
{
    ep_config c;
    c.ep_size = ep;
    c.num_experts = E;
    c.top_k = K;
    c.hidden = H;
    c.max_tokens_per_rank = C;
    c.dtype = dtype;
    c.enable_rank_mask = enable_rank_mask;
    c.scale_cols = EP_SCALE_COLS_DEFAULT;
    c.eplb_stats_max_bytes = 0;
    c.combine_dtype = EP_DTYPE_BF16;
    c.launch_flags = 0;
    c.num_partitions = 0;
    c.partition = 0;
    return c;
}

ep_status plan(const ep_config *cfg, Layout *L)
{
    if (!cfg)
        return fail(EP_ERR_INVALID_ARG, "config is NULL");
    const int ep = cfg->ep_size, E = cfg->num_experts, K = cfg->top_k, H = cfg->hidden;
    const int C = cfg->max_tokens_per_rank;
    const ep_dtype dtype = cfg->dtype;
    if (ep < 1 || ep > EP_MAX_EP_SIZE)
        return fail(EP_ERR_INVALID_ARG, "ep_size=%d outside [1, %d]", ep, EP_MAX_EP_SIZE);
    if (E < ep || E % ep != 0)
        return fail(EP_ERR_INVALID_ARG, "num_experts=%d is not a positive multiple of ep_size=%d", E, ep);
    if (K < 1 || K > EP_MAX_TOP_K)
        return fail(EP_ERR_INVALID_ARG, "top_k=%d outside [1, %d]", K, EP_MAX_TOP_K);
    const int elem = dtype_bytes(dtype);
    if (elem == 0)
        return fail(EP_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (H < 1 || ((long long)H * elem) % 16 != 0)
        return fail(EP_ERR_INVALID_ARG, "hidden=%d: a row must be a positive multiple of 16 bytes", H);
    if ((long long)H * 4 > (1LL << 30))  // row byte counts are 32-bit in the kernels
        return fail(EP_ERR_INVALID_ARG, "hidden=%d: rows are limited to 2^28 columns", H);
    const ep_dtype cdt = cfg->combine_dtype;
    if (cdt != EP_DTYPE_BF16 && cdt != EP_DTYPE_FP16 && cdt != EP_DTYPE_FP32)
        return fail(EP_ERR_INVALID_ARG, "combine_dtype %d: use bf16, fp16 or fp32", (int)cdt);
    const int ce = dtype_bytes(cdt);
    if (((long long)H * ce) % 16 != 0)
        return fail(EP_ERR_INVALID_ARG, "hidden=%d: the combine rows need hidden %% %d == 0", H, 16 / ce);
    if (C < 0)
        return fail(EP_ERR_INVALID_ARG, "max_tokens_per_rank=%d < 0", C);
    if ((long long)ep * C > (1LL << 30))  // slot and token indices are 32-bit in the kernels
        return fail(EP_ERR_INVALID_ARG, "ep_size*max_tokens_per_rank=%lld exceeds 2^30 slots",
                    (long long)ep * C);
    if (cfg->scale_cols < EP_SCALE_COLS_DEFAULT)
        return fail(EP_ERR_INVALID_ARG, "scale_cols=%d: use -1 (default), 0 or a positive count",
                    cfg->scale_cols);
    if (cfg->eplb_stats_max_bytes < 0 || cfg->eplb_stats_max_bytes % 4 != 0)
        return fail(EP_ERR_INVALID_ARG, "eplb_stats_max_bytes=%d must be a non-negative multiple of 4",
                    cfg->eplb_stats_max_bytes);
    if (cfg->launch_flags & ~EP_LAUNCH_PDL)
        return fail(EP_ERR_INVALID_ARG, "launch_flags=0x%x has unknown bits", (unsigned)cfg->launch_flags);
    const int G = cfg->num_partitions <= 1 ? 1 : cfg->num_partitions;
    if (cfg->num_partitions < 0 || ep % G != 0)
        return fail(EP_ERR_INVALID_ARG, "num_partitions=%d must be 0, 1 or a divisor of ep_size=%d",
                    cfg->num_partitions, ep);
    if (cfg->partition < 0 || cfg->partition >= G)
        return fail(EP_ERR_INVALID_ARG, "partition=%d outside [0, %d)", cfg->partition, G);
    L->num_parts = G;
    L->part = cfg->partition;
    L->nloc = ep / G;
    L->first = cfg->partition * L->nloc;
    L->elem_bytes = elem;
    L->row_bytes = H * elem;
    if (cfg->scale_cols == EP_SCALE_COLS_DEFAULT)
        L->scale_cols = (H % EP_SCALE_GROUP == 0) ? H / EP_SCALE_GROUP : 0;
    else
        L->scale_cols = cfg->scale_cols;
    const size_t rows = (size_t)ep * (size_t)C;
    L->st_hidden = align256(rows * L->row_bytes);
    L->st_scale = align256(rows * L->scale_cols * sizeof(float));
    L->st_ids = align256(rows * K * sizeof(int32_t));
    L->st_weights = align256(rows * K * sizeof(float));
    L->combine_elem = ce;
    L->st_comb = align256(rows * H * ce);
    const size_t n = (size_t)L->nloc;
    size_t off = 0;
    L->off_hidden = off;
    off += L->st_hidden * n;
    L->off_scale = off;
    off += L->st_scale * n;
    L->off_ids = off;
    off += L->st_ids * n;
    L->off_weights = off;
    off += L->st_weights * n;
    L->off_comb = off;
    off += L->st_comb * n;
    L->off_mask = off;
    off += align256(n * (size_t)C * sizeof(uint64_t));
    L->off_counts = off;
    off += align256(n * sizeof(int32_t));
    L->off_eplb = off;
    off += align256((size_t)ep * (size_t)cfg->eplb_stats_max_bytes);
    L->total = off < 256 ? 256 : off;
    return EP_OK;
}

ep_status make_handle(const ep_config *cfg, void *ws, size_t ws_bytes, bool own, ep_handle **out)
{
    if (!out)
        return fail(EP_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    Layout L{};
    ep_status st = plan(cfg, &L);
    if (st != EP_OK)
        return st;
    const int ep = cfg->ep_size, E = cfg->num_experts, K = cfg->top_k, H = cfg->hidden;
    const int C = cfg->max_tokens_per_rank;
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess)
        return fail(EP_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
    if (!ep_is_supported())
        return fail(EP_ERR_UNSUPPORTED, "device %d is not compute capability 10.3 (sm_103)", dev);
#if EP_CHECKED
    // look the check record up now, outside any stream capture a later call may be in
    if (!epk::check_record())
        return EP_ERR_CUDA;
#endif
    if (own) {
        void *p = nullptr;
        ce = cudaMalloc(&p, L.total);
        if (ce != cudaSuccess) {
            cudaGetLastError();
            return fail(ce == cudaErrorMemoryAllocation ? EP_ERR_OOM : EP_ERR_CUDA,
                        "cudaMalloc(%zu): %s", L.total, cudaGetErrorString(ce));
        }
        ws = p;
        ws_bytes = L.total;
    } else {
        if (!ws || !aligned(ws, 256))
            return fail(EP_ERR_INVALID_ARG, "workspace is NULL or not 256-byte aligned");
        if (ws_bytes < L.total)
            return fail(EP_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", ws_bytes, L.total);
    }
    ep_handle *h = new (std::nothrow) ep_handle();
    if (!h) {
        if (own)
            cudaFree(ws);
        return fail(EP_ERR_OOM, "host allocation of the handle failed");
    }
    h->ep = ep;
    h->num_experts = E;
    h->top_k = K;
    h->hidden = H;
    h->capacity = C;
    h->experts_per_rank = E / ep;
    h->dtype = cfg->dtype;
    h->elem_bytes = L.elem_bytes;
    h->row_bytes = L.row_bytes;
    h->scale_cols = L.scale_cols;
    h->mask_enabled = cfg->enable_rank_mask ? 1 : 0;
    h->eplb_max_bytes = cfg->eplb_stats_max_bytes;
    h->pdl = (cfg->launch_flags & EP_LAUNCH_PDL) != 0;
    h->cfg = *cfg;
    h->num_parts = L.num_parts;
    h->part = L.part;
    h->first = L.first;
    h->nloc = L.nloc;
    h->connected = L.num_parts == 1;
    h->combine_dtype = cfg->combine_dtype;
    h->device = dev;
    h->ws = static_cast<uint8_t *>(ws);
    h->ws_bytes = ws_bytes;
    h->owns_ws = own;
    h->off_hidden = L.off_hidden;
    h->off_scale = L.off_scale;
    h->off_ids = L.off_ids;
    h->off_weights = L.off_weights;
    h->off_comb = L.off_comb;
    h->off_mask = L.off_mask;
    h->off_counts = L.off_counts;
    h->off_eplb = L.off_eplb;
    h->st_hidden = L.st_hidden;
    h->st_scale = L.st_scale;
    h->st_ids = L.st_ids;
    h->st_weights = L.st_weights;
    h->st_comb = L.st_comb;
    h->pending = false;
    h->dev_counts = false;
    h->T = 0;
    h->mask = 0;
    for (int j = 0; j < h->nloc; ++j) {
        h->r_hidden[j] = h->ws + h->off_hidden + j * h->st_hidden;
        h->r_scale[j] = reinterpret_cast<float *>(h->ws + h->off_scale + j * h->st_scale);
        h->r_ids[j] = reinterpret_cast<int32_t *>(h->ws + h->off_ids + j * h->st_ids);
        h->r_weights[j] = reinterpret_cast<float *>(h->ws + h->off_weights + j * h->st_weights);
        const int d = h->first + j;
        h->t_hidden[d] = static_cast<uint8_t *>(h->r_hidden[j]);
        h->t_scale[d] = h->r_scale[j];
        h->t_ids[d] = h->r_ids[j];
        h->t_weights[d] = h->r_weights[j];
        h->t_comb[d] = h->ws + h->off_comb + j * h->st_comb;
    }
    h->t_eplb[h->part] = h->ws + h->off_eplb;
    *out = h;
    return ok();
}

ep_status check_device(const ep_handle *h)
{
    int dev = -1;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess)
        return fail(EP_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
    if (dev != h->device)
        return fail(EP_ERR_INVALID_ARG, "handle lives on device %d but device %d is current", h->device,
                    dev);
    return EP_OK;
}

// Normalises a caller's mask: UINT64_MAX means "all ranks". With masking
// disabled only "all ranks" is accepted.
ep_status resolve_mask(const ep_handle *h, uint64_t in, uint64_t *out)
{
    const uint64_t full = full_mask(h->ep);
    if (in == ~0ULL)
        in = full;
    if (!h->mask_enabled) {
        if (in != full)
            return fail(EP_ERR_INVALID_ARG,
                        "active_rank_mask 0x%llx given but the handle was created without "
                        "enable_rank_mask",
                        (unsigned long long)in);
    } else if (in & ~full) {
        return fail(EP_ERR_INVALID_ARG, "active_rank_mask 0x%llx has bits at or above ep_size=%d",
                    (unsigned long long)in, h->ep);
    }
    *out = in;
    return EP_OK;
}

}  // namespace

ep_status epk::set_error(ep_status st, const char *fmt, ...)
{
    if (st == EP_OK) {
        g_err[0] = '\0';
        return st;
    }
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

const char *epk::check_site_name(int site)
{
    static const char *const names[kNumSites] = {
        "dispatch: source hidden row", "dispatch: source id row", "dispatch: source scale row",
        "dispatch: source weight row", "dispatch: receive hidden row", "dispatch: receive id row",
        "dispatch: receive scale row", "dispatch: receive weight row", "dispatch: routing state",
        "dispatch: eplb_local_stats", "dispatch: gathered eplb stats", "combine: routing state",
        "combine: expert output row", "combine: output row", "ep_combine_noalloc: id row",
        "ep_combine_noalloc: routing scratch", "dispatch: device token counts", "live token counts"};
    return (site >= 0 && site < kNumSites) ? names[site] : "unknown site";
}

#if EP_CHECKED
namespace {

// One check record per device for the whole library: {violations, first
// site, first offset, that buffer's extent}.
__device__ unsigned long long g_check_rec[4];

std::mutex g_check_mu;
void *g_check_ptr[64] = {nullptr};
int g_trim_site = -1;
long long g_trim_bytes = 0;

}  // namespace

unsigned long long *epk::check_record()
{
    int dev = -1;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess || dev < 0 || dev >= 64) {
        set_error(EP_ERR_CUDA, "check record: no usable current device");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_check_mu);
    if (!g_check_ptr[dev]) {
        void *p = nullptr;
        ce = cudaGetSymbolAddress(&p, g_check_rec);
        if (ce != cudaSuccess || !p) {
            cudaGetLastError();
            set_error(EP_ERR_CUDA, "cudaGetSymbolAddress of the check record: %s", cudaGetErrorString(ce));
            return nullptr;
        }
        g_check_ptr[dev] = p;
    }
    return static_cast<unsigned long long *>(g_check_ptr[dev]);
}

epk::CheckCtx epk::check_ctx(unsigned long long *rec)
{
    std::lock_guard<std::mutex> lock(g_check_mu);
    return CheckCtx{rec, g_trim_site, g_trim_bytes};
}

ep_status epk::check_after(unsigned long long *rec, cudaStream_t stream, const char *what)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t ce = cudaStreamIsCapturing(stream, &cs);
    if (ce != cudaSuccess)
        return set_error(EP_ERR_CUDA, "%s: cudaStreamIsCapturing: %s", what, cudaGetErrorString(ce));
    if (cs != cudaStreamCaptureStatusNone)
        return EP_OK;  // checked at the next call outside the capture
    ce = cudaStreamSynchronize(stream);
    unsigned long long h[4] = {0, 0, 0, 0};
    if (ce == cudaSuccess)
        ce = cudaMemcpy(h, rec, sizeof h, cudaMemcpyDeviceToHost);
    if (ce != cudaSuccess)
        return set_error(EP_ERR_CUDA, "%s: reading the check record: %s", what, cudaGetErrorString(ce));
    if (h[0] == 0)
        return EP_OK;
    cudaMemset(rec, 0, sizeof h);
    return set_error(EP_ERR_DEVICE_CHECK,
                     "%s: %llu device accesses fell outside their buffers and were skipped; the first: %s, "
                     "byte offset %lld of a %lld-byte buffer",
                     what, h[0], check_site_name((int)h[1]), (long long)h[2], (long long)h[3]);
}

// Test hook of the checked build (not part of include/ep.h): declares every
// buffer of one access site `bytes` shorter than it is, so that accesses
// near its end, which stay inside the real buffer, are reported and
// skipped. site = -1 clears it.
extern "C" __attribute__((visibility("default"))) ep_status ep_checked_trim_extent(int site, long long bytes)
{
    if (site < -1 || site >= epk::kNumSites || bytes < 0)
        return epk::set_error(EP_ERR_INVALID_ARG, "site %d / bytes %lld", site, bytes);
    std::lock_guard<std::mutex> lock(g_check_mu);
    g_trim_site = site;
    g_trim_bytes = site < 0 ? 0 : bytes;
    return epk::set_error(EP_OK, "");
}
#else
unsigned long long *epk::check_record() { return nullptr; }

epk::CheckCtx epk::check_ctx(unsigned long long *) { return CheckCtx{nullptr, -1, 0}; }

ep_status epk::check_after(unsigned long long *, cudaStream_t, const char *) { return EP_OK; }
#endif

extern "C" {

int ep_is_supported(void)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return (major == 10 && minor == 3) ? 1 : 0;
}

ep_status ep_workspace_size(int ep_size, int num_experts, int top_k, int hidden,
                            int max_tokens_per_rank, ep_dtype dtype, size_t *bytes)
{
    const ep_config cfg = default_config(ep_size, num_experts, top_k, hidden, max_tokens_per_rank, dtype, 0);
    return ep_workspace_size_ex(&cfg, bytes);
}

ep_status ep_workspace_size_ex(const ep_config *cfg, size_t *bytes)
{
    if (!bytes)
        return fail(EP_ERR_INVALID_ARG, "bytes is NULL");
    Layout L{};
    ep_status st = plan(cfg, &L);
    if (st != EP_OK)
        return st;
    *bytes = L.total;
    return ok();
}

ep_status ep_create(int ep_size, int num_experts, int top_k, int hidden, int max_tokens_per_rank,
                    ep_dtype dtype, int enable_rank_mask, ep_handle **out)
{
    const ep_config cfg = default_config(ep_size, num_experts, top_k, hidden, max_tokens_per_rank, dtype,
                                         enable_rank_mask);
    return make_handle(&cfg, nullptr, 0, true, out);
}

ep_status ep_create_with_workspace(int ep_size, int num_experts, int top_k, int hidden,
                                   int max_tokens_per_rank, ep_dtype dtype, int enable_rank_mask,
                                   void *workspace, size_t bytes, ep_handle **out)
{
    const ep_config cfg = default_config(ep_size, num_experts, top_k, hidden, max_tokens_per_rank, dtype,
                                         enable_rank_mask);
    return make_handle(&cfg, workspace, bytes, false, out);
}

ep_status ep_create_ex(const ep_config *cfg, void *workspace, size_t bytes, ep_handle **out)
{
    return make_handle(cfg, workspace, bytes, workspace == nullptr, out);
}

ep_status ep_dispatch(ep_handle *h, const void *const *hidden, const float *const *hidden_scale,
                      const int32_t *const *topk_ids, const float *const *topk_weights,
                      const int32_t *num_tokens, int runtime_max_tokens_per_rank,
                      uint64_t active_rank_mask, void *stream, ep_dispatch_result *out)
{
    ep_dispatch_args args;
    args.hidden = hidden;
    args.hidden_scale = hidden_scale;
    args.topk_ids = topk_ids;
    args.topk_weights = topk_weights;
    args.num_tokens = num_tokens;
    args.runtime_max_tokens_per_rank = runtime_max_tokens_per_rank;
    args.active_rank_mask = active_rank_mask;
    args.eplb_local_stats = nullptr;
    args.eplb_stats_bytes = 0;
    args.num_tokens_device = nullptr;
    return ep_dispatch_ex(h, &args, stream, out);
}

ep_status ep_dispatch_ex(ep_handle *h, const ep_dispatch_args *args, void *stream, ep_dispatch_result *out)
{
    if (!h)
        return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    if (!args)
        return fail(EP_ERR_INVALID_ARG, "args is NULL");
    if (h->pending)
        return fail(EP_ERR_STATE, "dispatch called while the previous dispatch has not been combined");
    if (!h->connected)
        return fail(EP_ERR_STATE, "partition %d of %d is not connected with its group (ep_partition_connect)",
                    h->part, h->num_parts);
    const void *const *hidden = args->hidden;
    const float *const *hidden_scale = args->hidden_scale;
    const int32_t *const *topk_ids = args->topk_ids;
    const float *const *topk_weights = args->topk_weights;
    const int32_t *num_tokens = args->num_tokens;
    const int runtime_max_tokens_per_rank = args->runtime_max_tokens_per_rank;
    if (!hidden || !topk_ids || !num_tokens)
        return fail(EP_ERR_INVALID_ARG, "hidden, topk_ids and num_tokens must not be NULL");
    ep_status st = check_device(h);
    if (st != EP_OK)
        return st;
    const int T = runtime_max_tokens_per_rank < 0 ? h->capacity : runtime_max_tokens_per_rank;
    if (T > h->capacity)
        return fail(EP_ERR_INVALID_ARG, "runtime_max_tokens_per_rank=%d exceeds max_tokens_per_rank=%d",
                    T, h->capacity);
    uint64_t mask = 0;
    st = resolve_mask(h, args->active_rank_mask, &mask);
    if (st != EP_OK)
        return st;
    if (hidden_scale && h->scale_cols == 0)
        return fail(EP_ERR_INVALID_ARG, "hidden_scale given but the handle has no scale columns "
                                        "(hidden %% %d != 0 or scale_cols = 0)", EP_SCALE_GROUP);
    if (args->num_tokens_device && !aligned(args->num_tokens_device, 4))
        return fail(EP_ERR_INVALID_ARG, "num_tokens_device is not 4-byte aligned");
    const int eplb_bytes = args->eplb_local_stats ? args->eplb_stats_bytes : 0;
    if (args->eplb_local_stats) {
        if (h->eplb_max_bytes == 0)
            return fail(EP_ERR_INVALID_ARG, "eplb_local_stats given but the handle was created without "
                                            "eplb_stats_max_bytes");
        if (eplb_bytes <= 0 || eplb_bytes % 4 != 0 || eplb_bytes > h->eplb_max_bytes)
            return fail(EP_ERR_INVALID_ARG, "eplb_stats_bytes=%d must be a positive multiple of 4 "
                                            "and at most %d", eplb_bytes, h->eplb_max_bytes);
    }

    epk::DispatchArgs a;
    std::memset(&a, 0, sizeof a);
    for (int s = 0; s < h->nloc; ++s) {  // hosted source ranks; rank h->first + s
        if (eplb_bytes) {
            if (!args->eplb_local_stats[s] || !aligned(args->eplb_local_stats[s], 4))
                return fail(EP_ERR_INVALID_ARG, "eplb_local_stats[%d] is NULL or not 4-byte aligned "
                                                "(every rank passes its statistics)", s);
            a.eplb_src[s] = static_cast<const uint8_t *>(args->eplb_local_stats[s]);
        }
        const int n = num_tokens[s];
        if (n < 0 || n > T)
            return fail(EP_ERR_INVALID_ARG, "num_tokens[%d]=%d outside [0, tokens_per_rank=%d]", s, n, T);
        a.num_tokens[s] = n;
        if (n == 0)
            continue;
        if (!hidden[s] || !aligned(hidden[s], 16))
            return fail(EP_ERR_INVALID_ARG, "hidden[%d] is NULL or not 16-byte aligned", s);
        if (!topk_ids[s] || !aligned(topk_ids[s], 4))
            return fail(EP_ERR_INVALID_ARG, "topk_ids[%d] is NULL or not 4-byte aligned", s);
        if (hidden_scale && (!hidden_scale[s] || !aligned(hidden_scale[s], 4)))
            return fail(EP_ERR_INVALID_ARG,
                        "hidden_scale[%d] is NULL while other ranks pass scales (all or none)", s);
        if (topk_weights && (!topk_weights[s] || !aligned(topk_weights[s], 4)))
            return fail(EP_ERR_INVALID_ARG,
                        "topk_weights[%d] is NULL while other ranks pass weights (all or none)", s);
        a.hidden[s] = static_cast<const uint8_t *>(hidden[s]);
        a.ids[s] = topk_ids[s];
        a.scale[s] = hidden_scale ? hidden_scale[s] : nullptr;
        a.weights[s] = topk_weights ? topk_weights[s] : nullptr;
    }
    // every rank's receive buffers, advanced to the first row of the hosted sources
    a.row0 = (long long)h->first * T;
    for (int d = 0; d < h->ep; ++d) {
        a.recv_hidden[d] = h->t_hidden[d] + a.row0 * h->row_bytes;
        a.recv_scale[d] = h->t_scale[d] + a.row0 * h->scale_cols;
        a.recv_ids[d] = h->t_ids[d] + a.row0 * h->top_k;
        a.recv_weights[d] = h->t_weights[d] + a.row0 * h->top_k;
    }
    a.route_mask = reinterpret_cast<uint64_t *>(h->ws + h->off_mask);
    a.active = mask;
    a.ep = h->ep;
    a.src_first = h->first;
    a.n_src = h->nloc;
    a.num_experts = h->num_experts;
    a.experts_per_rank = h->experts_per_rank;
    a.top_k = h->top_k;
    a.T = T;
    a.row_bytes = h->row_bytes;
    a.G = hidden_scale ? h->scale_cols : 0;
    a.has_weights = topk_weights ? 1 : 0;
    for (int p = 0; p < h->num_parts; ++p)
        a.eplb_dst[p] = h->t_eplb[p];
    a.n_eplb_dst = h->num_parts;
    a.eplb_bytes = eplb_bytes;
    a.dev_counts = args->num_tokens_device;
    a.live_counts = args->num_tokens_device ? reinterpret_cast<int32_t *>(h->ws + h->off_counts) : nullptr;
    unsigned long long *rec = nullptr;
#if EP_CHECKED
    rec = epk::check_record();
    if (!rec)
        return EP_ERR_CUDA;
#endif
    a.chk = epk::check_ctx(rec);

    nvtxRangePushA("ep_dispatch");  // host-side range around the launch, for profilers
    cudaError_t ce = epk::launch_dispatch(a, static_cast<cudaStream_t>(stream), h->pdl);
    nvtxRangePop();
    if (ce != cudaSuccess)
        return fail(EP_ERR_CUDA, "dispatch launch: %s", cudaGetErrorString(ce));

    h->pending = true;
    h->dev_counts = args->num_tokens_device != nullptr;
    h->T = T;
    h->mask = mask;
    for (int s = 0; s < h->nloc; ++s)
        h->counts[s] = a.num_tokens[s];
    if (out) {
        out->tokens_per_rank = T;
        out->ep_size = h->ep;
        out->first_rank = h->first;
        out->num_ranks = h->nloc;
        out->recv_hidden = h->r_hidden;
        out->recv_scale = hidden_scale ? h->r_scale : nullptr;
        out->recv_topk_ids = h->r_ids;
        out->recv_topk_weights = topk_weights ? h->r_weights : nullptr;
        out->eplb_global_stats = eplb_bytes ? h->ws + h->off_eplb : nullptr;
        out->eplb_stats_bytes = eplb_bytes;
    }
    st = epk::check_after(rec, static_cast<cudaStream_t>(stream), "ep_dispatch");
    return st == EP_OK ? ok() : st;
}

ep_status ep_get_combine_input_buffer(ep_handle *h, int rank, void **out)
{
    if (!h || !out)
        return fail(EP_ERR_INVALID_ARG, "handle or out is NULL");
    *out = nullptr;
    if (!h->pending)
        return fail(EP_ERR_STATE, "the combine input buffer exists only from a dispatch until its combine");
    if (rank < h->first || rank >= h->first + h->nloc)
        return fail(EP_ERR_INVALID_ARG, "rank=%d outside the handle's ranks [%d, %d)", rank, h->first,
                    h->first + h->nloc);
    *out = h->ws + h->off_comb + (size_t)(rank - h->first) * h->st_comb;
    return ok();
}

ep_status ep_combine(ep_handle *h, const void *const *expert_output, void *const *output,
                     uint64_t active_rank_mask, void *stream)
{
    if (!h)
        return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    if (!h->pending)
        return fail(EP_ERR_STATE, "combine called without a pending dispatch");
    if (!output)
        return fail(EP_ERR_INVALID_ARG, "output is NULL");
    ep_status st = check_device(h);
    if (st != EP_OK)
        return st;
    uint64_t mask = 0;
    st = resolve_mask(h, active_rank_mask, &mask);
    if (st != EP_OK)
        return st;
    if (mask != h->mask)
        return fail(EP_ERR_INVALID_ARG, "combine active_rank_mask 0x%llx differs from dispatch's 0x%llx",
                    (unsigned long long)mask, (unsigned long long)h->mask);

    epk::CombineArgs a;
    std::memset(&a, 0, sizeof a);
    // every rank's combine input, advanced to the first row of the hosted sources
    a.row0 = (long long)h->first * h->T;
    const long long row0_bytes = a.row0 * h->hidden * (h->combine_dtype == EP_DTYPE_FP32 ? 4 : 2);
    for (int d = 0; d < h->ep; ++d) {
        const void *p = expert_output ? expert_output[d] : nullptr;
        if (!p)
            p = h->t_comb[d];
        else if (!aligned(p, 16))
            return fail(EP_ERR_INVALID_ARG, "expert_output[%d] is not 16-byte aligned", d);
        a.eo[d] = static_cast<const uint8_t *>(p) + row0_bytes;
    }
    a.token_offset[0] = 0;
    for (int s = 0; s < h->nloc; ++s) {  // hosted source ranks
        a.num_tokens[s] = h->counts[s];
        a.token_offset[s + 1] = a.token_offset[s] + h->counts[s];
        if (h->counts[s] == 0)
            continue;
        if (!output[s] || !aligned(output[s], 16))
            return fail(EP_ERR_INVALID_ARG, "output[%d] is NULL or not 16-byte aligned", s);
        a.out[s] = output[s];
    }
    a.route_mask = reinterpret_cast<const uint64_t *>(h->ws + h->off_mask);
    a.live_counts = h->dev_counts ? reinterpret_cast<const int32_t *>(h->ws + h->off_counts) : nullptr;
    a.ep = h->ep;
    a.src_first = h->first;
    a.n_src = h->nloc;
    a.T = h->T;
    a.H = h->hidden;
    a.ctype = (int)h->combine_dtype;
    unsigned long long *rec = nullptr;
#if EP_CHECKED
    rec = epk::check_record();
    if (!rec)
        return EP_ERR_CUDA;
#endif
    a.chk = epk::check_ctx(rec);

    nvtxRangePushA("ep_combine");
    cudaError_t ce = epk::launch_combine(a, static_cast<cudaStream_t>(stream), h->pdl);
    nvtxRangePop();
    if (ce != cudaSuccess)
        return fail(EP_ERR_CUDA, "combine launch: %s", cudaGetErrorString(ce));
    h->pending = false;
    st = epk::check_after(rec, static_cast<cudaStream_t>(stream), "ep_combine");
    return st == EP_OK ? ok() : st;
}

ep_status ep_destroy(ep_handle *h)
{
    if (!h)
        return ok();
    ep_status st = EP_OK;
    if (h->owns_ws && h->ws) {
        int prev = -1;
        cudaGetDevice(&prev);
        if (prev != h->device)
            cudaSetDevice(h->device);
        cudaError_t ce = cudaFree(h->ws);
        if (prev >= 0 && prev != h->device)
            cudaSetDevice(prev);
        if (ce != cudaSuccess)
            st = fail(EP_ERR_CUDA, "cudaFree: %s", cudaGetErrorString(ce));
    }
    delete h;
    return st == EP_OK ? ok() : st;
}

uint64_t ep_rank_mask(const int *ranks, int n)
{
    uint64_t m = 0;
    if (!ranks)
        return 0;
    for (int i = 0; i < n; ++i)
        if (ranks[i] >= 0 && ranks[i] < 64)
            m |= 1ULL << ranks[i];
    return m;
}

const char *ep_last_error(void) { return g_err; }

ep_status ep_partition_describe(const ep_config *cfg, void *workspace, size_t bytes, ep_partition_info *out)
{
    if (!out)
        return fail(EP_ERR_INVALID_ARG, "out is NULL");
    Layout L{};
    ep_status st = plan(cfg, &L);
    if (st != EP_OK)
        return st;
    std::memset(out, 0, sizeof *out);
    out->config = *cfg;
    out->first_rank = L.first;
    out->num_ranks = L.nloc;
    out->workspace = workspace;
    out->workspace_bytes = bytes;
    out->off_recv_hidden = L.off_hidden;
    out->off_recv_scale = L.off_scale;
    out->off_recv_ids = L.off_ids;
    out->off_recv_weights = L.off_weights;
    out->off_combine_in = L.off_comb;
    out->off_eplb = L.off_eplb;
    out->stride_recv_hidden = L.st_hidden;
    out->stride_recv_scale = L.st_scale;
    out->stride_recv_ids = L.st_ids;
    out->stride_recv_weights = L.st_weights;
    out->stride_combine_in = L.st_comb;
    return ok();
}

ep_status ep_partition_info_of(const ep_handle *h, ep_partition_info *out)
{
    if (!h)
        return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    return ep_partition_describe(&h->cfg, h->ws, h->ws_bytes, out);
}

namespace {

// Name of the first field in which two configurations of one group differ
// (the partition index and the launch flags may differ), or NULL.
const char *group_config_differs(const ep_config &a, const ep_config &b)
{
    const int ga = a.num_partitions <= 1 ? 1 : a.num_partitions;
    const int gb = b.num_partitions <= 1 ? 1 : b.num_partitions;
    if (a.ep_size != b.ep_size) return "ep_size";
    if (a.num_experts != b.num_experts) return "num_experts";
    if (a.top_k != b.top_k) return "top_k";
    if (a.hidden != b.hidden) return "hidden";
    if (a.max_tokens_per_rank != b.max_tokens_per_rank) return "max_tokens_per_rank";
    if (a.dtype != b.dtype) return "dtype";
    if ((a.enable_rank_mask != 0) != (b.enable_rank_mask != 0)) return "enable_rank_mask";
    if (a.scale_cols != b.scale_cols) return "scale_cols";
    if (a.eplb_stats_max_bytes != b.eplb_stats_max_bytes) return "eplb_stats_max_bytes";
    if (a.combine_dtype != b.combine_dtype) return "combine_dtype";
    if (ga != gb) return "num_partitions";
    return nullptr;
}

}  // namespace

ep_status ep_partition_check(const ep_partition_info *infos, int n)
{
    if (!infos || n < 1 || n > EP_MAX_EP_SIZE)
        return fail(EP_ERR_INVALID_ARG, "need 1 to %d partition descriptions, got %d", EP_MAX_EP_SIZE, n);
    const ep_config &c0 = infos[0].config;
    const int G = c0.num_partitions <= 1 ? 1 : c0.num_partitions;
    if (n != G)
        return fail(EP_ERR_INVALID_ARG, "%d descriptions for a group of %d partitions", n, G);
    for (int p = 0; p < n; ++p) {
        const ep_partition_info &x = infos[p];
        if (x.config.partition != p)
            return fail(EP_ERR_INVALID_ARG, "description %d is of partition %d", p, x.config.partition);
        if (const char *f = group_config_differs(x.config, c0))
            return fail(EP_ERR_INVALID_ARG, "partition %d has another %s than partition 0", p, f);
        Layout L{};
        if (plan(&x.config, &L) != EP_OK)
            return EP_ERR_INVALID_ARG;  // message set by plan
        if (x.first_rank != L.first || x.num_ranks != L.nloc || x.off_recv_hidden != L.off_hidden ||
            x.off_recv_scale != L.off_scale || x.off_recv_ids != L.off_ids ||
            x.off_recv_weights != L.off_weights || x.off_combine_in != L.off_comb || x.off_eplb != L.off_eplb ||
            x.stride_recv_hidden != L.st_hidden || x.stride_recv_scale != L.st_scale ||
            x.stride_recv_ids != L.st_ids || x.stride_recv_weights != L.st_weights ||
            x.stride_combine_in != L.st_comb)
            return fail(EP_ERR_INVALID_ARG, "partition %d: the layout differs from the one its configuration gives", p);
        if (!x.workspace || !aligned(x.workspace, 256))
            return fail(EP_ERR_INVALID_ARG, "partition %d: workspace is NULL or not 256-byte aligned", p);
        if (x.workspace_bytes < L.total)
            return fail(EP_ERR_INVALID_ARG, "partition %d: workspace has %zu bytes, needs %zu", p,
                        x.workspace_bytes, L.total);
        const uintptr_t lo = reinterpret_cast<uintptr_t>(x.workspace), hi = lo + x.workspace_bytes;
        for (int q = 0; q < p; ++q) {
            const uintptr_t qlo = reinterpret_cast<uintptr_t>(infos[q].workspace);
            const uintptr_t qhi = qlo + infos[q].workspace_bytes;
            if (lo < qhi && qlo < hi)
                return fail(EP_ERR_INVALID_ARG, "the workspaces of partitions %d and %d overlap", q, p);
        }
    }
    return ok();
}

ep_status ep_partition_connect(ep_handle *h, const ep_partition_info *infos, int n)
{
    if (!h)
        return fail(EP_ERR_INVALID_ARG, "handle is NULL");
    if (h->pending)
        return fail(EP_ERR_STATE, "connect called while a dispatch is pending");
    ep_status st = ep_partition_check(infos, n);
    if (st != EP_OK)
        return st;
    if (n != h->num_parts)
        return fail(EP_ERR_INVALID_ARG, "%d descriptions but the handle is one of %d partitions", n, h->num_parts);
    const ep_partition_info &me = infos[h->part];  // h->part < num_parts == n
    if (me.workspace != h->ws)
        return fail(EP_ERR_INVALID_ARG, "description %d is not of this handle's workspace", h->part);
    if (const char *f = group_config_differs(me.config, h->cfg))
        return fail(EP_ERR_INVALID_ARG, "description %d has another %s than the handle", h->part, f);
    for (int p = 0; p < n; ++p) {
        const ep_partition_info &x = infos[p];
        uint8_t *base = static_cast<uint8_t *>(x.workspace);
        for (int j = 0; j < x.num_ranks; ++j) {
            const int d = x.first_rank + j;
            h->t_hidden[d] = base + x.off_recv_hidden + j * x.stride_recv_hidden;
            h->t_scale[d] = reinterpret_cast<float *>(base + x.off_recv_scale + j * x.stride_recv_scale);
            h->t_ids[d] = reinterpret_cast<int32_t *>(base + x.off_recv_ids + j * x.stride_recv_ids);
            h->t_weights[d] = reinterpret_cast<float *>(base + x.off_recv_weights + j * x.stride_recv_weights);
            h->t_comb[d] = base + x.off_combine_in + j * x.stride_combine_in;
        }
        h->t_eplb[p] = base + x.off_eplb;
    }
    h->connected = true;
    return ok();
}

ep_status ep_binary_version(int *version)
{
    if (!version)
        return fail(EP_ERR_INVALID_ARG, "version is NULL");
    *version = 0;
    int v[16], n = 0;
    cudaError_t ce = epk::kernel_binary_versions(v, 15, &n);
    if (ce == cudaSuccess && n < 16)
        ce = epk::noalloc_binary_version(&v[n++]);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return fail(EP_ERR_CUDA, "cudaFuncGetAttributes: %s", cudaGetErrorString(ce));
    }
    for (int i = 1; i < n; ++i)
        if (v[i] != v[0])
            return fail(EP_ERR_UNSUPPORTED, "kernel %d reports binary version %d, kernel 0 %d", i, v[i], v[0]);
    *version = v[0];
    return ok();
}

}  // extern "C"
