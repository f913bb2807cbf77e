// ep_kernels.cu -- sm_103a kernels of rank-major MoE EP dispatch/combine with
// every EP rank a virtual rank in this GPU's memory.
//
// dispatch_kernel (one warp per (source slot s*T+t, column chunk of its
// hidden row) work item, grid-stride):
//   payload   -- the item's chunk of the hidden row is read once with
//                non-caching 32-byte loads (16-byte ones when a row or source
//                pointer is only 16-byte aligned), issued first so they
//                overlap the routing, and stored to every routed rank's row
//                s*T+t.
//   routing   -- lane k reads expert id k; the owners' bits are OR-reduced
//                across the warp (two 32-bit halves for up to 64 ranks) and
//                ANDed with active_rank_mask (page "flashinfer.moe_ep.
//                NVLinkOneSidedAlltoAll", dispatch(): a masked-off rank
//                receives nothing). The slot's first chunk keeps the bit set
//                for combine.
//   id plane  -- the slot's first chunk writes the slot's id row in every
//                destination rank: the token's ids where it is routed,
//                invalid_expert_id elsewhere and on padding slots (same page,
//                class description), then the scale and weight rows (one
//                dispatch carries all four payloads).
//
// combine_kernel (each thread owns 64 bytes of one live token's output row,
// as 4 16-byte or, for large aligned combines, 2 32-byte vectors):
//   reads the row's slot in each routed rank's combine input in ascending
//   rank order, two ranks' loads in flight before their adds, adds in fp32
//   from +0.0 and rounds once to the combine type (bf16 or fp16; fp32 sums
//   are stored as they are) (page "flashinfer.moe_ep.MoEEpCommunication",
//   combine(): per token, the ranks' expert outputs are added up).
//
// A launch handles a range of source ranks (all of them, or one partition's
// of a partitioned group) and reaches every destination rank's buffers
// through per-rank address tables, advanced on the host to the range's first
// row so that the launch's own slot index addresses them; where each rank's
// buffers live (one workspace or several) does not matter to the kernels.
// Both kernels open with griddepcontrol.launch_dependents / .wait, which let
// a programmatically dependent launch (EP_LAUNCH_PDL) be scheduled early and
// are no-ops otherwise.
//
// With device-side token counts the dispatch reads each rank's count when it
// runs (clamped to the host maximum) and leaves it for the combine, whose
// blocks past it exit. In the checked build (EP_CHECKED) every global access
// is tested against its buffer first (EP_IN_BOUNDS); in the normal build
// those tests compile to nothing.
//
// Nothing here is a dense contraction; both kernels are bound by HBM
// bandwidth, so the design is about coalesced 16- and 32-byte accesses and
// enough bytes in flight per SM. Launch shapes come from sweeps on GB300.
#include <atomic>

#include "ep_internal.h"

namespace epk {
namespace {

// Launch shapes (compile-time; -D overrides exist for tuning sweeps).
#ifndef EP_DISPATCH_THREADS
#define EP_DISPATCH_THREADS 256
#endif
#ifndef EP_DISPATCH_VEC_PER_LANE
#define EP_DISPATCH_VEC_PER_LANE 8
#endif
#ifndef EP_DISPATCH_BLOCKS_PER_SM
#define EP_DISPATCH_BLOCKS_PER_SM 64
#endif
#ifndef EP_DISPATCH_WIDE
#define EP_DISPATCH_WIDE 1  // 32-byte row accesses when rows and sources are 32-byte aligned
#endif
#ifndef EP_COMBINE_WIDE
#define EP_COMBINE_WIDE 1  // 32-byte accesses when every row and pointer is 32-byte aligned
#endif
#ifndef EP_COMBINE_MAX_THREADS
#define EP_COMBINE_MAX_THREADS 256
#endif
#ifndef EP_COMBINE_VPT
#define EP_COMBINE_VPT 4
#endif
#ifndef EP_COMBINE_BATCH
#define EP_COMBINE_BATCH 2
#endif

constexpr unsigned kFull = 0xffffffffu;
constexpr int kDispatchThreads = EP_DISPATCH_THREADS;          // one warp per work item
constexpr int kDispatchVecPerLane = EP_DISPATCH_VEC_PER_LANE;  // 16-byte vectors per lane per chunk
constexpr int kDispatchBlocksPerSm = EP_DISPATCH_BLOCKS_PER_SM;  // grid cap, in blocks per SM
constexpr int kCombineMaxThreads = EP_COMBINE_MAX_THREADS;
constexpr int kCombineVpt = EP_COMBINE_VPT;      // 16-byte column vectors per combine thread
constexpr int kCombineBatch = EP_COMBINE_BATCH;  // ranks whose rows are loaded before their adds

// Programmatic dependent launch (sm_90+). launch_dependents: the next kernel
// of the stream may be scheduled once every block of this grid has issued it
// (or exited). wait: block until the previous kernel of the stream has
// completed and its memory operations are visible. Both are no-ops when the
// grid was launched without the programmatic-serialization attribute.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// 32-byte vector (sm_100+ 256-bit global access): half the load/store
// instructions of 16-byte vectors for the same bytes.
struct alignas(32) Vec32 {
    uint32_t w[8];
};

template <int VB>
struct RowVec;

template <>
struct RowVec<16> {
    using T = uint4;
    __device__ static T load(const void *p) { return ld_stream(p); }
    __device__ static void store(void *p, const T &v) { *static_cast<uint4 *>(p) = v; }
};

template <>
struct RowVec<32> {
    using T = Vec32;
    __device__ static T load(const void *p)
    {
        T v;
        asm("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
            : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
              "=r"(v.w[6]), "=r"(v.w[7])
            : "l"(p));
        return v;
    }
    __device__ static void store(void *p, const T &v)
    {
        asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v.w[0]),
                     "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
                     "r"(v.w[7])
                     : "memory");
    }
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 -> packed bf16x2, round to nearest even (cvt.rn.bf16x2.f32; no
// flush of subnormals). `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// binary16 halves of a 32-bit word, widened exactly (cvt.f32.f16).
__device__ __forceinline__ float f16_lo(uint32_t w)
{
    float f;
    asm("{ .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.f32.f16 %0, lo; }" : "=f"(f) : "r"(w));
    return f;
}
__device__ __forceinline__ float f16_hi(uint32_t w)
{
    float f;
    asm("{ .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %1;\n cvt.f32.f16 %0, hi; }" : "=f"(f) : "r"(w));
    return f;
}

// Two fp32 -> packed binary16x2, round to nearest even (cvt.rn.f16x2.f32;
// subnormal results kept). `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Element codec of the combine, per storage type: how many elements a
// 16-byte vector holds, how to widen them to fp32 and how to narrow the sums.
template <int CT>
struct CombineCodec;

template <>
struct CombineCodec<EP_DTYPE_BF16> {
    static constexpr int kPerVec = 8;
    __device__ static void widen(const uint4 &x, float *f)
    {
        f[0] = bf16_lo(x.x), f[1] = bf16_hi(x.x), f[2] = bf16_lo(x.y), f[3] = bf16_hi(x.y);
        f[4] = bf16_lo(x.z), f[5] = bf16_hi(x.z), f[6] = bf16_lo(x.w), f[7] = bf16_hi(x.w);
    }
    __device__ static uint4 narrow(const float *a)
    {
        return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                          pack_bf16x2(a[6], a[7]));
    }
};

template <>
struct CombineCodec<EP_DTYPE_FP16> {
    static constexpr int kPerVec = 8;
    __device__ static void widen(const uint4 &x, float *f)
    {
        f[0] = f16_lo(x.x), f[1] = f16_hi(x.x), f[2] = f16_lo(x.y), f[3] = f16_hi(x.y);
        f[4] = f16_lo(x.z), f[5] = f16_hi(x.z), f[6] = f16_lo(x.w), f[7] = f16_hi(x.w);
    }
    __device__ static uint4 narrow(const float *a)
    {
        return make_uint4(pack_f16x2(a[0], a[1]), pack_f16x2(a[2], a[3]), pack_f16x2(a[4], a[5]),
                          pack_f16x2(a[6], a[7]));
    }
};

template <>
struct CombineCodec<EP_DTYPE_FP32> {
    static constexpr int kPerVec = 4;
    __device__ static void widen(const uint4 &x, float *f)
    {
        f[0] = __uint_as_float(x.x), f[1] = __uint_as_float(x.y);
        f[2] = __uint_as_float(x.z), f[3] = __uint_as_float(x.w);
    }
    __device__ static uint4 narrow(const float *a)
    {
        return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                          __float_as_uint(a[3]));
    }
};

// VB: bytes per row access of one lane (16, or 32 when every source row and
// destination row is 32-byte aligned); a chunk is 32 lanes x kVpl accesses
// = 4 KB either way.
template <int VB>
__global__ void __launch_bounds__(kDispatchThreads)
    dispatch_kernel(const __grid_constant__ DispatchArgs a)
{
    using RV = RowVec<VB>;
    constexpr int kVpl = kDispatchVecPerLane * 16 / VB;
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const long long n_slots = (long long)a.n_src * a.T;  // this launch's source slots
#if EP_CHECKED
    const long long n_rows = (long long)a.ep * a.T;  // rows of every receive buffer (extents)
#endif
    const long long warp_stride = (long long)gridDim.x * wpb;
    const int K = a.top_k;
    // Nothing below may touch global memory before the previous kernel is done:
    // it may have produced the inputs, or still read the buffers written here.
    pdl_launch_dependents();
    pdl_wait();

    // ---- eplb_local_stats all-gather: one warp per (own rank i, gathered
    // buffer p) copies rank src_first+i's statistics into row src_first+i of
    // buffer p (a few hundred bytes per rank).
    if (a.eplb_bytes > 0) {
        const long long gw = (long long)blockIdx.x * wpb + (threadIdx.x >> 5);
        if (gw < (long long)a.n_src * a.n_eplb_dst) {
            const int i = (int)(gw / a.n_eplb_dst);
            const int p = (int)(gw - (long long)i * a.n_eplb_dst);
            const uint32_t *src = reinterpret_cast<const uint32_t *>(a.eplb_src[i]);
            uint32_t *dst = reinterpret_cast<uint32_t *>(a.eplb_dst[p] + (long long)(a.src_first + i) * a.eplb_bytes);
            for (int w = lane; w < (a.eplb_bytes >> 2); w += 32) {
                uint32_t x = 0;
                if (EP_IN_BOUNDS(a.chk, kSiteEplbSrc, src + w, 4, a.eplb_src[i], a.eplb_bytes))
                    x = src[w];
                if (EP_IN_BOUNDS(a.chk, kSiteEplbDst, dst + w, 4, a.eplb_dst[p], (long long)a.ep * a.eplb_bytes))
                    dst[w] = x;
            }
        }
    }

    // Work items are (slot, column chunk) pairs: the hidden row is split into
    // chunks of 32*kDispatchVecPerLane 16-byte vectors, one warp per chunk,
    // so the work divides finely over the resident warps even when there are
    // few slots. Every item routes its slot; the first chunk's item also
    // writes the routing state, the id plane and the scale/weight rows.
    const int nvec = a.row_bytes / VB;
    const int chunk_vecs = 32 * kVpl;
    const int nchunks = (nvec + chunk_vecs - 1) / chunk_vecs;
    const long long n_items = n_slots * nchunks;
    for (long long item = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); item < n_items;
         item += warp_stride) {
        const long long slot = item / nchunks;  // own slot i*T + t
        const int chunk = (int)(item - slot * nchunks);
        const int c0 = chunk * chunk_vecs;
        const int s = (int)(slot / a.T);  // local source index
        const int t = (int)(slot - (long long)s * a.T);
        int n_s = a.num_tokens[s];
        if (a.dev_counts) {  // counts read at run time, clamped to [0, the host maximum]
            int c = 0;
            if (EP_IN_BOUNDS(a.chk, kSiteDevCounts, a.dev_counts + s, 4, a.dev_counts, (long long)a.n_src * 4))
                c = a.dev_counts[s];
            n_s = c < 0 ? 0 : (c < n_s ? c : n_s);
            if (t == 0 && chunk == 0 && lane == 0 &&
                EP_IN_BOUNDS(a.chk, kSiteLiveCounts, a.live_counts + s, 4, a.live_counts, (long long)a.n_src * 4))
                a.live_counts[s] = n_s;  // for the combine
        }
        const bool live = t < n_s;

        // ---- this chunk of the hidden row, loaded before the routing so the
        // two memory round trips overlap (almost every live token is routed)
        const uint8_t *src = a.hidden[s] + (long long)t * a.row_bytes;
        typename RV::T v[kVpl];
#if EP_CHECKED
#pragma unroll
        for (int j = 0; j < kVpl; ++j)
            v[j] = typename RV::T{};
#endif
        if (live) {
#pragma unroll
            for (int j = 0; j < kVpl; ++j) {
                const int idx = c0 + j * 32 + lane;
                if (idx < nvec && EP_IN_BOUNDS(a.chk, kSiteSrcHidden, src + VB * (long long)idx, VB, a.hidden[s],
                                               (long long)a.num_tokens[s] * a.row_bytes))
                    v[j] = RV::load(src + VB * (long long)idx);
            }
        }

        // ---- routing: destination-rank bit set of this slot
        int my_id = EP_INVALID_EXPERT_ID;
        unsigned lo = 0, hi = 0;
        if (live && lane < K) {
            const int32_t *ip = a.ids[s] + (long long)t * K + lane;
            if (EP_IN_BOUNDS(a.chk, kSiteSrcIds, ip, 4, a.ids[s], (long long)a.num_tokens[s] * K * 4))
                my_id = *ip;
            if (my_id >= 0 && my_id < a.num_experts) {
                const int owner = my_id / a.experts_per_rank;
                if (owner < 32)
                    lo = 1u << owner;
                else
                    hi = 1u << (owner - 32);
            }
        }
        lo = __reduce_or_sync(kFull, lo);
        hi = __reduce_or_sync(kFull, hi);
        const uint64_t m = ((((uint64_t)hi) << 32) | lo) & a.active;
        if (chunk == 0 && lane == 0 &&
            EP_IN_BOUNDS(a.chk, kSiteRouteWrite, a.route_mask + slot, 8, a.route_mask, n_slots * 8))
            a.route_mask[slot] = m;

        // ---- id rows of this slot in all destination ranks (first chunk's item)
        if (chunk != 0) {
            // the first chunk's item writes the slot's ids
        } else if ((K & 3) == 0) {
            const int qpr = K >> 2;  // int4 vectors per id row
            const int n = a.ep * qpr;
            for (int base = 0; base < n; base += 32) {
                const int i = base + lane;
                const int d = i / qpr;
                const int q = i - d * qpr;
                int4 v;
                v.x = __shfl_sync(kFull, my_id, 4 * q + 0);
                v.y = __shfl_sync(kFull, my_id, 4 * q + 1);
                v.z = __shfl_sync(kFull, my_id, 4 * q + 2);
                v.w = __shfl_sync(kFull, my_id, 4 * q + 3);
                if (i < n) {
                    if (!((m >> d) & 1u))
                        v = make_int4(EP_INVALID_EXPERT_ID, EP_INVALID_EXPERT_ID,
                                      EP_INVALID_EXPERT_ID, EP_INVALID_EXPERT_ID);
                    int32_t *p = a.recv_ids[d] + slot * K + 4 * q;
                    if (EP_IN_BOUNDS(a.chk, kSiteRecvIds, p, 16, a.recv_ids[d] - a.row0 * K, n_rows * K * 4))
                        *reinterpret_cast<int4 *>(p) = v;
                }
            }
        } else {
            const int n = a.ep * K;
            for (int base = 0; base < n; base += 32) {
                const int i = base + lane;
                const int d = i / K;
                const int k = i - d * K;
                int v = __shfl_sync(kFull, my_id, k);
                if (i < n) {
                    if (!((m >> d) & 1u))
                        v = EP_INVALID_EXPERT_ID;
                    int32_t *p = a.recv_ids[d] + slot * K + k;
                    if (EP_IN_BOUNDS(a.chk, kSiteRecvIds, p, 4, a.recv_ids[d] - a.row0 * K, n_rows * K * 4))
                        *p = v;
                }
            }
        }
        if (m == 0)
            continue;  // warp-uniform: padding, unrouted or fully masked slot

        // ---- this chunk of the hidden row: read once, stored to each routed rank
        for (uint64_t mm = m; mm; mm &= mm - 1) {
            const int d = __ffsll((long long)mm) - 1;
            uint8_t *dst = a.recv_hidden[d] + slot * a.row_bytes;
#pragma unroll
            for (int j = 0; j < kVpl; ++j) {
                const int idx = c0 + j * 32 + lane;
                if (idx < nvec && EP_IN_BOUNDS(a.chk, kSiteRecvHidden, dst + VB * (long long)idx, VB,
                                               a.recv_hidden[d] - a.row0 * a.row_bytes, n_rows * a.row_bytes))
                    RV::store(dst + VB * (long long)idx, v[j]);
            }
        }
        if (chunk != 0)
            continue;

        // ---- scale row (G fp32) and weight row (K fp32)
        if (a.G > 0) {
            const float *ssrc = a.scale[s] + (long long)t * a.G;
            for (int j = lane; j < a.G; j += 32) {
                float x = 0.0f;
                if (EP_IN_BOUNDS(a.chk, kSiteSrcScale, ssrc + j, 4, a.scale[s], (long long)a.num_tokens[s] * a.G * 4))
                    x = ssrc[j];
                for (uint64_t mm = m; mm; mm &= mm - 1) {
                    const int d = __ffsll((long long)mm) - 1;
                    float *p = a.recv_scale[d] + slot * a.G + j;
                    if (EP_IN_BOUNDS(a.chk, kSiteRecvScale, p, 4, a.recv_scale[d] - a.row0 * a.G, n_rows * a.G * 4))
                        *p = x;
                }
            }
        }
        if (a.has_weights && lane < K) {
            const float *wp = a.weights[s] + (long long)t * K + lane;
            float w = 0.0f;
            if (EP_IN_BOUNDS(a.chk, kSiteSrcWeights, wp, 4, a.weights[s], (long long)a.num_tokens[s] * K * 4))
                w = *wp;
            for (uint64_t mm = m; mm; mm &= mm - 1) {
                const int d = __ffsll((long long)mm) - 1;
                float *p = a.recv_weights[d] + slot * K + lane;
                if (EP_IN_BOUNDS(a.chk, kSiteRecvWeights, p, 4, a.recv_weights[d] - a.row0 * K, n_rows * K * 4))
                    *p = w;
            }
        }
    }
}

// Splits a row access of VB bytes into the 16-byte halves the codecs work on.
__device__ __forceinline__ const uint4 &half16(const uint4 &v, int) { return v; }
__device__ __forceinline__ uint4 half16(const Vec32 &v, int h)
{
    return make_uint4(v.w[4 * h], v.w[4 * h + 1], v.w[4 * h + 2], v.w[4 * h + 3]);
}
__device__ __forceinline__ void set_half16(uint4 &v, int, const uint4 &x) { v = x; }
__device__ __forceinline__ void set_half16(Vec32 &v, int h, const uint4 &x)
{
    v.w[4 * h] = x.x, v.w[4 * h + 1] = x.y, v.w[4 * h + 2] = x.z, v.w[4 * h + 3] = x.w;
}

template <int CT, int VB>
__global__ void __launch_bounds__(kCombineMaxThreads)
    combine_kernel(const __grid_constant__ CombineArgs a, int blocks_per_row, long long n_blocks)
{
    using Codec = CombineCodec<CT>;
    using RV = RowVec<VB>;
    constexpr int kEpv = Codec::kPerVec;      // elements per 16 bytes
    constexpr int kH = VB / 16;               // 16-byte halves per access
    constexpr int kV = kCombineVpt / kH;      // accesses per thread (same 64 bytes either way)
    const long long row_bytes = (long long)a.H * (16 / kEpv);
    const int nvec = (int)(row_bytes / VB);
    const int nthr = blockDim.x;
    // the routing state and the expert outputs come from the kernels before this one
    pdl_launch_dependents();
    pdl_wait();
    for (long long b = blockIdx.x; b < n_blocks; b += gridDim.x) {
        // block -> (live token g, column chunk); g -> source rank s by binary
        // search of the token offsets, so no block is spent on padding slots
        const int g = (int)(b / blocks_per_row);
        const int chunk = (int)(b - (long long)g * blocks_per_row);
        int lo = 0, hi = a.n_src - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.token_offset[mid] <= g)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int s = lo;  // local source index
        const int t = g - a.token_offset[s];
        if (a.live_counts) {  // device-side counts: rows past the dispatch's count are skipped
            int c = 0;
            if (EP_IN_BOUNDS(a.chk, kSiteLiveCounts, a.live_counts + s, 4, a.live_counts, (long long)a.n_src * 4))
                c = a.live_counts[s];
            if (t >= c)
                continue;
        }
        const long long slot = (long long)s * a.T + t;  // own slot: routing state
        const int v0 = chunk * (nthr * kV) + threadIdx.x;
        if (v0 >= nvec)
            continue;
        uint64_t m = 0;
        if (EP_IN_BOUNDS(a.chk, kSiteRouteRead, a.route_mask + slot, 8, a.route_mask, (long long)a.n_src * a.T * 8))
            m = a.route_mask[slot];
        // byte offset of the token's row from eo[d], which points at row row0 = src_first*T
        const long long row = slot * row_bytes;

        float acc[kV][kH][kEpv];
#pragma unroll
        for (int j = 0; j < kV; ++j)
#pragma unroll
            for (int h = 0; h < kH; ++h)
#pragma unroll
                for (int e = 0; e < kEpv; ++e)
                    acc[j][h][e] = 0.0f;

        uint64_t mm = m;
        while (mm) {
            typename RV::T x[kCombineBatch][kV];
#if EP_CHECKED
#pragma unroll
            for (int r = 0; r < kCombineBatch; ++r)
#pragma unroll
                for (int j = 0; j < kV; ++j)
                    x[r][j] = typename RV::T{};
#endif
            int nb = 0;
#pragma unroll
            for (int r = 0; r < kCombineBatch; ++r) {
                if (mm) {
                    const int d = __ffsll((long long)mm) - 1;
                    mm &= mm - 1;
                    const uint8_t *base = static_cast<const uint8_t *>(a.eo[d]) + row;
#pragma unroll
                    for (int j = 0; j < kV; ++j) {
                        const int v = v0 + j * nthr;
                        if (v < nvec && EP_IN_BOUNDS(a.chk, kSiteCombineIn, base + VB * (long long)v, VB,
                                                     static_cast<const uint8_t *>(a.eo[d]) - a.row0 * row_bytes,
                                                     (long long)a.ep * a.T * row_bytes))
                            x[r][j] = RV::load(base + VB * (long long)v);
                    }
                    nb = r + 1;
                }
            }
#pragma unroll
            for (int r = 0; r < kCombineBatch; ++r) {
                if (r < nb) {
#pragma unroll
                    for (int j = 0; j < kV; ++j)
#pragma unroll
                        for (int h = 0; h < kH; ++h) {
                            float f[kEpv];
                            Codec::widen(half16(x[r][j], h), f);
#pragma unroll
                            for (int e = 0; e < kEpv; ++e)
                                acc[j][h][e] = __fadd_rn(acc[j][h][e], f[e]);
                        }
                }
            }
        }
        uint8_t *out = static_cast<uint8_t *>(a.out[s]) + (long long)t * row_bytes;
#pragma unroll
        for (int j = 0; j < kV; ++j) {
            const int v = v0 + j * nthr;
            if (v < nvec) {
                typename RV::T o;
#pragma unroll
                for (int h = 0; h < kH; ++h)
                    set_half16(o, h, Codec::narrow(acc[j][h]));
                if (EP_IN_BOUNDS(a.chk, kSiteCombineOut, out + VB * (long long)v, VB, a.out[s],
                                 (long long)a.num_tokens[s] * row_bytes))
                    RV::store(out + VB * (long long)v, o);
            }
        }
    }
}

// Block width of the combine: the row's vectors are split into chunks of
// threads*VPT; a width whose chunks tile the row exactly leaves no idle
// threads (64 for 4096-wide rows, 32 for 7168-wide rows). Preference order
// from measurements on GB300.
// One launch of `kernel` on `stream`, with programmatic dependent launch
// when `pdl` is set.
template <typename Kernel, typename... Args>
cudaError_t launch(Kernel kernel, long long grid, int threads, cudaStream_t stream, bool pdl, Args... args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

int combine_threads(int nvec)
{
    const int per_thread = kCombineVpt;
    const int candidates[] = {64, 32, 128};
    for (int c : candidates)
        if (c <= kCombineMaxThreads && nvec % (c * per_thread) == 0)
            return c;
    return 64;
}

// SM count of the current device, looked up once per device (host threads
// may launch concurrently: the cache is atomic).
int sm_count()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 152;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace

cudaError_t kernel_binary_versions(int *out, int max, int *n)
{
    const void *fns[] = {
        reinterpret_cast<const void *>(dispatch_kernel<16>),
        reinterpret_cast<const void *>(dispatch_kernel<32>),
        reinterpret_cast<const void *>(combine_kernel<EP_DTYPE_BF16, 16>),
        reinterpret_cast<const void *>(combine_kernel<EP_DTYPE_BF16, 32>),
        reinterpret_cast<const void *>(combine_kernel<EP_DTYPE_FP16, 16>),
        reinterpret_cast<const void *>(combine_kernel<EP_DTYPE_FP16, 32>),
        reinterpret_cast<const void *>(combine_kernel<EP_DTYPE_FP32, 16>),
        reinterpret_cast<const void *>(combine_kernel<EP_DTYPE_FP32, 32>),
    };
    *n = 0;
    for (const void *f : fns) {
        cudaFuncAttributes attr;
        cudaError_t ce = cudaFuncGetAttributes(&attr, f);
        if (ce != cudaSuccess)
            return ce;
        if (*n < max)
            out[*n] = attr.binaryVersion;
        ++*n;
    }
    return cudaSuccess;
}

cudaError_t launch_dispatch(const DispatchArgs &a, cudaStream_t stream, bool pdl)
{
    const long long n_slots = (long long)a.n_src * a.T;
    if (n_slots == 0 && a.eplb_bytes == 0)
        return cudaSuccess;
    // 32-byte accesses need every source row and receive row 32-byte aligned:
    // row_bytes % 32 == 0, every receive buffer and every source base pointer
    // of a rank with tokens.
    bool wide = EP_DISPATCH_WIDE && (a.row_bytes % 32 == 0);
    for (int d = 0; wide && d < a.ep; ++d)
        if ((reinterpret_cast<uintptr_t>(a.recv_hidden[d]) % 32) != 0)
            wide = false;
    for (int s = 0; wide && s < a.n_src; ++s)
        if (a.num_tokens[s] > 0 && (reinterpret_cast<uintptr_t>(a.hidden[s]) % 32) != 0)
            wide = false;
    const int wpb = kDispatchThreads / 32;
    const int chunk_vecs = 32 * kDispatchVecPerLane;  // 16-byte units per 4 KB chunk
    const long long n_items = n_slots * (((a.row_bytes >> 4) + chunk_vecs - 1) / chunk_vecs);
    long long blocks = (n_items + wpb - 1) / wpb;
    const long long cap = (long long)sm_count() * kDispatchBlocksPerSm;
    if (blocks > cap)
        blocks = cap;
    // one warp per (own rank, gathered buffer)
    const long long eplb_blocks = a.eplb_bytes > 0 ? ((long long)a.n_src * a.n_eplb_dst + wpb - 1) / wpb : 0;
    if (blocks < eplb_blocks)
        blocks = eplb_blocks;
    cudaError_t ce = wide ? launch(dispatch_kernel<32>, blocks, kDispatchThreads, stream, pdl, a)
                          : launch(dispatch_kernel<16>, blocks, kDispatchThreads, stream, pdl, a);
    return ce != cudaSuccess ? ce : cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t stream, bool pdl)
{
    const int elem = a.ctype == EP_DTYPE_FP32 ? 4 : 2;
    const int nvec = (int)(((long long)a.H * elem) >> 4);
    const int threads = combine_threads(nvec);
    const int per_block = threads * kCombineVpt;
    const int bpr = (nvec + per_block - 1) / per_block;
    const long long n_blocks = (long long)a.token_offset[a.n_src] * bpr;
    if (n_blocks == 0)
        return cudaSuccess;
    long long grid = n_blocks;
    if (grid > (1LL << 30))
        grid = 1LL << 30;
    // 32-byte accesses need every row of every input and output 32-byte aligned.
    // They raise the streaming rate but also the fixed cost of a launch
    // (measured on GB300: ~7.2 vs ~7.0 TB/s incremental, ~17 vs ~11 us fixed;
    // equal at ~117 MB of output, faster from ~235 MB), so they are used only
    // for large combines: output of at least 192 MiB.
    const long long out_bytes = (long long)a.token_offset[a.n_src] * a.H * elem;
    bool wide = EP_COMBINE_WIDE && (((long long)a.H * elem) % 32 == 0) && out_bytes >= (192LL << 20);
    for (int d = 0; wide && d < a.ep; ++d)
        if ((reinterpret_cast<uintptr_t>(a.eo[d]) % 32) != 0)
            wide = false;
    for (int s = 0; wide && s < a.n_src; ++s)
        if (a.num_tokens[s] > 0 && (reinterpret_cast<uintptr_t>(a.out[s]) % 32) != 0)
            wide = false;
#define EP_LAUNCH_COMBINE(CT)                                                          \
    (wide ? launch(combine_kernel<CT, 32>, grid, threads, stream, pdl, a, bpr, n_blocks) \
          : launch(combine_kernel<CT, 16>, grid, threads, stream, pdl, a, bpr, n_blocks))
    cudaError_t ce;
    switch (a.ctype) {
    case EP_DTYPE_BF16:
        ce = EP_LAUNCH_COMBINE(EP_DTYPE_BF16);
        break;
    case EP_DTYPE_FP16:
        ce = EP_LAUNCH_COMBINE(EP_DTYPE_FP16);
        break;
    case EP_DTYPE_FP32:
        ce = EP_LAUNCH_COMBINE(EP_DTYPE_FP32);
        break;
    default:
        return cudaErrorInvalidValue;
    }
#undef EP_LAUNCH_COMBINE
    return ce != cudaSuccess ? ce : cudaGetLastError();
}

}  // namespace epk
