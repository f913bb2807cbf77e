/*
 * ep.h -- C ABI of the GB300 (sm_103a) rank-major MoE expert-parallel
 * dispatch/combine library (libep_gb300.so).
 *
 * The operation is the one FlashInfer's moe_ep API pages define:
 *  - page "flashinfer.moe_ep.MoEEpCommunication": dispatch() delivers every
 *    token to each rank that owns one of its top-k experts; combine() adds up,
 *    per token, what the ranks' experts produced; get_combine_input_buffer()
 *    lends the expert computation a library-owned output buffer; calls
 *    alternate dispatch(), combine(), dispatch(), ...; destroy() may be
 *    repeated.
 *  - page "flashinfer.moe_ep.NVLinkOneSidedAlltoAll": one dispatch carries
 *    the hidden row, its scales, the ids and the weights; a receiving rank
 *    keeps token t of source rank s in row s*tokens_per_rank + t; padding
 *    slots and tokens the rank does not receive are marked with
 *    invalid_expert_id; a rank left out of active_rank_mask receives
 *    nothing, and combine uses the dispatch's mask.
 *
 * All ep_size ranks of the EP group are virtual ranks on ONE GPU: every
 * rank's inputs, receive buffers and combine inputs live in that GPU's
 * memory, and one call handles all ranks at once. The per-rank arguments
 * are therefore host arrays of ep_size device pointers, entry r belonging
 * to rank r.
 *
 * Readings the pages leave open, fixed here:
 *  - invalid_expert_id is EP_INVALID_EXPERT_ID (-1); ids are int32, weights
 *    and scales fp32; a scale row has hidden/128 entries.
 *  - experts are split contiguously: rank d owns ids [d*E/ep, (d+1)*E/ep);
 *    ids outside [0, E) route nowhere; duplicate ids reach a rank once.
 *  - a routed receive row carries the token's whole top-k id row unchanged;
 *    only the id row of a padding/unrouted row is defined (all -1); its
 *    hidden, scale and weight rows keep whatever they held.
 *  - the rank mask filters destinations only.
 *  - combine adds, per token, the rows of the ranks it was routed to, in
 *    ascending rank order, in fp32 from +0.0, and rounds once (round to
 *    nearest even) to the combine dtype: bf16 by default, or fp16; fp32
 *    results are not rounded. The result is bit-exact and deterministic.
 *
 * Errors are synchronous: each call checks its arguments and the handle's
 * state on the host before it launches anything, and returns a status;
 * ep_last_error() gives a message. GPU work is queued on the given stream
 * (NULL = the legacy default stream) and is asynchronous to the host.
 *
 * Threads: calls on different handles may come from different host threads
 * at once; calls on one handle must not overlap (a handle holds the state
 * of its pending dispatch). ep_last_error() is per thread. Every call works
 * on the current CUDA device, which must be the handle's.
 *
 * Checked build (libep_gb300_checked.so, compiled with EP_CHECKED=1; same
 * ABI): the kernels test every global access against the extent this
 * header gives its buffer, skip any access outside and record it; after
 * its launches each call waits for its stream and returns
 * EP_ERR_DEVICE_CHECK (with the first access's buffer and offset in
 * ep_last_error) if anything was recorded. The call's other effects
 * (state, results of the accesses that were inside) stand. Inside a stream
 * capture the wait is skipped and the record is reported by the next call
 * outside one. All calls of the library share one record per device, so
 * overlapping work on two streams may report the other's access; its device
 * address is looked up once per device and kept, which assumes the primary
 * context lives as long as the process. It is for testing: slower, and
 * synchronous.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1, /* bad sizes, pointers, masks, or weights/scales on some ranks only */
    EP_ERR_STATE = 2,       /* dispatch while one is pending, combine without dispatch */
    EP_ERR_CUDA = 3,        /* a CUDA runtime call failed (message has the CUDA error) */
    EP_ERR_OOM = 4,         /* workspace allocation failed */
    EP_ERR_UNSUPPORTED = 5, /* no sm_103 device current */
    EP_ERR_DEVICE_CHECK = 6 /* checked build only (below): a kernel access fell outside its buffer */
} ep_status;

typedef enum {
    EP_DTYPE_BF16 = 0,      /* hidden rows of bfloat16 */
    EP_DTYPE_FP8_E4M3 = 1,  /* hidden rows of OCP fp8 e4m3fn */
    EP_DTYPE_FP16 = 2,      /* hidden rows of IEEE binary16 */
    EP_DTYPE_FP32 = 3       /* hidden rows of IEEE binary32 */
} ep_dtype;

#define EP_INVALID_EXPERT_ID (-1)
#define EP_MAX_EP_SIZE 64 /* the rank mask is one uint64 */
#define EP_MAX_TOP_K 32
#define EP_SCALE_GROUP 128 /* hidden columns per fp32 scale (the default scale width) */
#define EP_SCALE_COLS_DEFAULT (-1) /* ep_config.scale_cols: hidden/128 if that divides, else none */

typedef struct ep_handle ep_handle;

/* Where one dispatch left its results. All arrays are host arrays owned by
 * the handle, each with one device pointer per rank of the handle (entry j =
 * destination rank first_rank + j; every rank unless the handle is a
 * partition). Each buffer holds ep_size*tokens_per_rank rows; row
 * s*tokens_per_rank+t is token t of source rank s. The pointers stay valid
 * until ep_destroy; the contents until the next ep_dispatch. */
typedef struct {
    int tokens_per_rank;
    int ep_size;
    int first_rank;                   /* the arrays' entry j is rank first_rank + j ... */
    int num_ranks;                    /* ... for j < num_ranks (0 and ep_size unless partitioned) */
    void *const *recv_hidden;         /* rows of `hidden` elements of the payload dtype */
    float *const *recv_scale;         /* rows of scale_cols fp32, or NULL if none were sent */
    int32_t *const *recv_topk_ids;    /* rows of top_k int32 */
    float *const *recv_topk_weights;  /* rows of top_k fp32, or NULL if none were sent */
    /* eplb_local_stats of all ranks, row r = rank r's bytes: device [ep_size,
     * eplb_stats_bytes], one buffer every rank reads (treat as read-only), or
     * NULL when the dispatch sent none (ep_dispatch_ex only). */
    const void *eplb_global_stats;
    int eplb_stats_bytes;
} ep_dispatch_result;

/* Everything a handle is created with (ep_create_ex). */
typedef struct {
    int ep_size;               /* 1..64 ranks */
    int num_experts;           /* a positive multiple of ep_size */
    int top_k;                 /* 1..32 */
    int hidden;                /* payload columns, <= 2^28; hidden*elem_bytes a multiple of 16
                                  for the payload and for the combine dtype (so hidden % 8 == 0
                                  for a bf16 or fp16 combine, hidden % 4 == 0 for fp32) */
    int max_tokens_per_rank;   /* capacity C >= 0 */
    ep_dtype dtype;            /* payload type of the hidden rows */
    int enable_rank_mask;      /* 0/1 */
    int scale_cols;            /* fp32 scales per row: EP_SCALE_COLS_DEFAULT, 0 (none) or > 0 */
    int eplb_stats_max_bytes;  /* eplb_local_stats bytes per rank the handle can gather, a
                                  multiple of 4 (0: not supported) */
    ep_dtype combine_dtype;    /* type of the expert outputs combine sums and of its results:
                                  EP_DTYPE_BF16 (0, the default), EP_DTYPE_FP16 or EP_DTYPE_FP32;
                                  hidden*elem_bytes of it must be a multiple of 16 */
    int launch_flags;          /* 0 or EP_LAUNCH_PDL (below) */
    int num_partitions;        /* 0 or 1: one handle holds every rank. G > 1 (dividing ep_size):
                                  the handle is one partition of the group (below) */
    int partition;             /* which partition, 0 <= partition < num_partitions */
} ep_config;

/* ep_config.launch_flags bit: launch the dispatch and combine kernels with
 * programmatic dependent launch (cudaLaunchAttributeProgrammaticStream-
 * Serialization). Each kernel lets the next kernel of its stream be launched
 * as soon as all of its own blocks are running, and itself waits
 * (griddepcontrol.wait) for the kernel before it to complete and its memory
 * to be visible before touching global memory. So a combine queued right
 * after its dispatch is launched and scheduled while the dispatch drains,
 * and results are the same as with ordinary stream order. A kernel before
 * it that does not let dependents launch early (any ordinary kernel) is
 * simply waited for, so the flag is safe with any producer on the stream.
 * Also honoured inside stream capture (the graph keeps the programmatic
 * edge). Not on the pages: a launch-latency option for small (decode-size)
 * rounds. */
#define EP_LAUNCH_PDL 1

/* Everything one dispatch takes (ep_dispatch_ex); see ep_dispatch for the
 * first seven fields. eplb_local_stats: NULL, or eplb_local_stats[r] =
 * device pointer to rank r's eplb_stats_bytes bytes of expert-load
 * statistics (4-byte aligned; every rank passes the same size), gathered
 * into ep_dispatch_result.eplb_global_stats by the same launch
 * (MoEEpCommunication.dispatch, parameter eplb_local_stats). A partition
 * handle writes its ranks' rows into every partition's gathered buffer, so
 * each holds all ranks' rows once every partition has dispatched (all pass
 * the same eplb_stats_bytes).
 * num_tokens_device: NULL, or a device int32 [ep_size] array (one entry per
 * hosted rank for a partition handle) the kernels
 * read when they run: rank s then has min(max(num_tokens_device[s], 0),
 * num_tokens[s]) tokens, and num_tokens (host) gives each rank's maximum
 * (its source tensors hold that many rows). This lets one captured CUDA
 * graph serve steps whose token counts change: the caller writes the new
 * counts into the array before each replay. The routing, the receive rows
 * and the combine all follow the device counts; the ep_combine that follows
 * writes only the first count rows of each output. (An extension for CUDA
 * graphs; the pages' dispatch takes counts from its tensors' shapes.) */
typedef struct {
    const void *const *hidden;
    const float *const *hidden_scale;
    const int32_t *const *topk_ids;
    const float *const *topk_weights;
    const int32_t *num_tokens;
    int runtime_max_tokens_per_rank;
    uint64_t active_rank_mask;
    const void *const *eplb_local_stats;
    int eplb_stats_bytes;
    const int32_t *num_tokens_device;
} ep_dispatch_args;

/* 1 when the current CUDA device can run this library (compute capability
 * 10.3, the sm_103a build), else 0. Does no GPU work.
 * (MoEEpCommunication.is_platform_supported) */
int ep_is_supported(void);

/* Bytes of device workspace a handle with these parameters needs: for every
 * rank, receive buffers and a bf16 combine-input buffer of ep_size *
 * max_tokens_per_rank rows, plus 8 bytes of routing state per slot and a
 * 256-byte block for the live token counts. Validates the parameters like
 * ep_create. */
ep_status ep_workspace_size(int ep_size, int num_experts, int top_k, int hidden,
                            int max_tokens_per_rank, ep_dtype dtype, size_t *bytes);

/* ep_workspace_size for a full configuration (scale width, eplb capacity). */
ep_status ep_workspace_size_ex(const ep_config *cfg, size_t *bytes);

/* Creates a handle for one EP group (MoEEpCommunication constructor with
 * MoEEpCommParams). Requirements: 1 <= ep_size <= 64; num_experts a
 * positive multiple of ep_size; 1 <= top_k <= 32; hidden > 0 with
 * hidden*elem_bytes a multiple of 16, hidden % 8 == 0 and hidden <= 2^28;
 * max_tokens_per_rank >= 0 with ep_size*max_tokens_per_rank <= 2^30.
 * enable_rank_mask (0/1) allows active_rank_mask on dispatch/combine.
 * Allocates the workspace with cudaMalloc on the current device; *out
 * receives the handle (NULL on error). */
ep_status ep_create(int ep_size, int num_experts, int top_k, int hidden,
                    int max_tokens_per_rank, ep_dtype dtype, int enable_rank_mask,
                    ep_handle **out);

/* As ep_create, but uses caller-owned device memory `workspace` of `bytes`
 * (>= ep_workspace_size, 256-byte aligned) on the current device. The
 * caller frees it after ep_destroy. */
ep_status ep_create_with_workspace(int ep_size, int num_experts, int top_k, int hidden,
                                   int max_tokens_per_rank, ep_dtype dtype, int enable_rank_mask,
                                   void *workspace, size_t bytes, ep_handle **out);

/* Creates a handle from a full configuration. workspace == NULL: allocate
 * with cudaMalloc (freed by ep_destroy); else caller-owned device memory of
 * `bytes` >= ep_workspace_size_ex, 256-byte aligned. ep_create(...) equals
 * ep_create_ex with scale_cols = EP_SCALE_COLS_DEFAULT,
 * eplb_stats_max_bytes = 0 and launch_flags = 0. */
ep_status ep_create_ex(const ep_config *cfg, void *workspace, size_t bytes, ep_handle **out);

/* Dispatch of all ep_size source ranks (MoEEpCommunication.dispatch;
 * NVLinkOneSidedAlltoAll.dispatch for active_rank_mask). For a partition
 * handle: of the ranks it hosts, and every per-rank array below has one
 * entry per hosted rank (see "Partitioned EP groups").
 *  hidden[s]       device [num_tokens[s], hidden] payload dtype, 16-byte aligned
 *  hidden_scale    NULL, or hidden_scale[s] device fp32 [num_tokens[s], scale_cols]
 *                  (scale_cols = hidden/128 for ep_create handles; needs scale_cols > 0)
 *  topk_ids[s]     device int32 [num_tokens[s], top_k], global expert ids
 *  topk_weights    NULL, or topk_weights[s] device fp32 [num_tokens[s], top_k]
 *  num_tokens      host int32 [ep_size], 0 <= num_tokens[s] <= tokens_per_rank
 *  runtime_max_tokens_per_rank  tokens_per_rank of this step, <= max_tokens_per_rank;
 *                  negative means max_tokens_per_rank (static shapes)
 *  active_rank_mask  bit d set = rank d active; UINT64_MAX = all ranks. Any
 *                  other value needs a handle created with enable_rank_mask and
 *                  no bit at or above ep_size (else EP_ERR_INVALID_ARG).
 *  stream          cudaStream_t to queue the work on
 *  out             filled with the receive buffers (may be NULL)
 * Scales and weights are all-or-none: if the array is given, every rank with
 * tokens must pass a non-NULL pointer (an empty rank may pass anything).
 * Rows of ranks with zero tokens are never read. Inputs must stay valid until
 * the queued work has run. Returns EP_ERR_STATE if a dispatch is pending. */
ep_status ep_dispatch(ep_handle *h, const void *const *hidden, const float *const *hidden_scale,
                      const int32_t *const *topk_ids, const float *const *topk_weights,
                      const int32_t *num_tokens, int runtime_max_tokens_per_rank,
                      uint64_t active_rank_mask, void *stream, ep_dispatch_result *out);

/* ep_dispatch with its arguments in a struct, plus the eplb_local_stats
 * all-gather and device-side token counts. Same checks and errors;
 * additionally EP_ERR_INVALID_ARG when stats are given to a handle without
 * eplb capacity, exceed it, are not a multiple of 4 bytes, or are missing
 * for some rank, or when num_tokens_device is not 4-byte aligned. */
ep_status ep_dispatch_ex(ep_handle *h, const ep_dispatch_args *args, void *stream,
                         ep_dispatch_result *out);

/* Device pointer to rank `rank`'s backend-owned combine input (a rank the
 * handle hosts: any rank, unless the handle is a partition): [ep_size *
 * tokens_per_rank, hidden] elements of the handle's combine dtype (bf16
 * unless ep_config.combine_dtype says otherwise) for the pending dispatch. Passing it (or
 * NULL) to ep_combine avoids one copy. Valid between ep_dispatch and
 * ep_combine; EP_ERR_STATE outside (MoEEpCommunication.get_combine_input_buffer,
 * NVLinkOneSidedAlltoAll.get_combine_input_buffer). */
ep_status ep_get_combine_input_buffer(ep_handle *h, int rank, void **out);

/* Combine of the pending dispatch (MoEEpCommunication.combine). For a
 * partition handle: of the source ranks it hosts (output has one entry per
 * hosted rank), reading every rank's expert outputs (expert_output keeps
 * ep_size entries; NULL ones are that rank's backend buffer, wherever its
 * partition's workspace is).
 *  expert_output   NULL = every rank's backend combine input buffer; else
 *                  expert_output[d] is rank d's [ep_size*tokens_per_rank, hidden]
 *                  device buffer of the combine dtype (NULL entry = that rank's
 *                  backend buffer), 16-byte aligned; only routed rows are read.
 *  output[s]       device [num_tokens[s], hidden] of the combine dtype, 16-byte
 *                  aligned, caller-owned; may be NULL when num_tokens[s] == 0.
 *                  After a dispatch with num_tokens_device, num_tokens[s] is the
 *                  maximum and only the rows below the device count are written.
 *  active_rank_mask  must equal the dispatch's (when masking is enabled).
 * output[s][t] = round( sum over routed ranks d ascending of expert_output[d]
 * [s*tokens_per_rank + t] ) with an fp32 accumulator from +0.0 and one
 * round-to-nearest-even to the combine dtype (none for fp32). A token routed
 * nowhere gets +0.0. Returns the handle to the idle state. */
ep_status ep_combine(ep_handle *h, const void *const *expert_output, void *const *output,
                     uint64_t active_rank_mask, void *stream);

/* Frees the handle and, when the library allocated the workspace (ep_create,
 * or ep_create_ex with workspace NULL), that workspace: cudaFree waits for
 * work using it. With a caller-owned workspace nothing is synchronised:
 * finish the streams that used it before reusing or freeing that memory.
 * NULL is a no-op; the Python binding makes repeated destroy() calls no-ops
 * (MoEEpCommunication.destroy). */
ep_status ep_destroy(ep_handle *h);

/* Bit set of the listed ranks, for active_rank_mask; ranks outside [0, 64)
 * are ignored (NVLinkOneSidedAlltoAll.active_rank_mask). */
uint64_t ep_rank_mask(const int *ranks, int n);

/* Message of the calling thread's last failed call ("" if none). */
const char *ep_last_error(void);

/* The architecture of the device code the CUDA runtime loaded for this
 * library on the current device: *version = major*10 + minor of the binary
 * (103 for the sm_103a build), as cudaFuncGetAttributes reports it for every
 * kernel of the library. EP_ERR_CUDA when the kernels cannot be loaded on
 * the current device (e.g. no sm_103 GPU), EP_ERR_UNSUPPORTED when two
 * kernels report different versions. Runs no kernel. (Not on the pages: a
 * build check.) */
ep_status ep_binary_version(int *version);

/* ---- Partitioned EP groups -------------------------------------------------
 * The pages' backends (NVLinkOneSidedAlltoAll, class description) run one
 * rank per GPU and move rows between the GPUs' buffers with one-sided
 * stores and loads. A partitioned group is that layout for virtual ranks:
 * the ep_size ranks are split into G = num_partitions contiguous blocks of
 * ep_size/G ranks; partition g hosts ranks [g*ep_size/G, (g+1)*ep_size/G)
 * in a workspace of its own (its ranks' receive and combine-input buffers,
 * the routing state of its own source tokens) and has a handle of its own.
 * Its dispatch scatters its own ranks' tokens into the receive rows of every
 * rank, in whichever partition's workspace those live, through a table of
 * destination addresses; its combine sums its own tokens' rows from every
 * rank's combine input, in ascending rank order, exactly as the unpartitioned
 * combine does. Results are bit for bit those of one handle over all ranks.
 *
 * Per-rank arguments of a partition handle have one entry per rank it hosts
 * (entry j = rank first_rank + j): ep_dispatch's hidden, hidden_scale,
 * topk_ids, topk_weights, num_tokens (and ep_dispatch_args'
 * eplb_local_stats and num_tokens_device), and ep_combine's output.
 * ep_combine's expert_output keeps ep_size entries (every rank's rows are
 * read); ep_get_combine_input_buffer takes a rank the partition hosts.
 *
 * Set-up: each partition describes itself (ep_partition_describe: its
 * configuration and the layout of its workspace), the descriptions of all
 * G partitions are brought together, and every handle is connected with all
 * of them (ep_partition_connect), which checks that they form one group. An
 * address in a description must be valid on the device of the handle that
 * is connected with it; on one GPU the workspaces are simply separate
 * allocations. Every partition dispatches once per step with the same
 * runtime_max_tokens_per_rank and mask; a partition's receive buffers are
 * complete once every partition's dispatch has completed, and a combine may
 * start only after every rank's expert outputs are written: ordering across
 * partitions is the caller's (stream order, or events between streams).
 * A connected handle keeps its peers' addresses: a partition's workspace must
 * stay allocated while any handle of the group may still dispatch or combine,
 * so destroy a group's handles together, after their last work has run. */

/* One partition as its peers see it. */
typedef struct {
    ep_config config;           /* the partition's configuration */
    int first_rank, num_ranks;  /* the ranks it hosts */
    void *workspace;            /* device address of its workspace */
    size_t workspace_bytes;     /* its size (at least ep_workspace_size_ex) */
    /* byte offsets of its regions in the workspace, and bytes per hosted rank
     * (receive hidden/scale/ids/weights, combine input); the eplb buffer */
    size_t off_recv_hidden, off_recv_scale, off_recv_ids, off_recv_weights, off_combine_in, off_eplb;
    size_t stride_recv_hidden, stride_recv_scale, stride_recv_ids, stride_recv_weights, stride_combine_in;
} ep_partition_info;

/* Fills *out for the partition cfg->partition of a group configured by
 * `cfg`, whose workspace is `workspace` (bytes as given). Host only; needs
 * no GPU. EP_ERR_INVALID_ARG on a bad configuration. */
ep_status ep_partition_describe(const ep_config *cfg, void *workspace, size_t bytes, ep_partition_info *out);

/* ep_partition_describe of a handle: its configuration and its workspace
 * (also one the library allocated). Host only. */
ep_status ep_partition_info_of(const ep_handle *h, ep_partition_info *out);

/* Checks that infos[0..n) describe one partitioned group: n ==
 * num_partitions, infos[p] is partition p, all configurations equal but for
 * `partition` and `launch_flags` (a local choice), each layout is the one
 * its configuration gives, workspaces
 * are large enough, 256-byte aligned and do not overlap. Host only;
 * EP_ERR_INVALID_ARG with the first problem in ep_last_error otherwise. */
ep_status ep_partition_check(const ep_partition_info *infos, int n);

/* Connects a partition handle with all partitions of its group (its own
 * description included, which must match the handle): ep_partition_check,
 * then the handle's destination tables are filled. Required once before the
 * first dispatch of a partition handle (EP_ERR_STATE otherwise); may be
 * repeated while no dispatch is pending. An unpartitioned handle needs no
 * connection (connecting it with its own description is accepted). */
ep_status ep_partition_connect(ep_handle *h, const ep_partition_info *infos, int n);

/* Largest ep_size * tokens_per_rank that ep_combine_noalloc accepts. */
#define EP_NOALLOC_MAX_SLOTS 65536

/* Combine for callers that cannot allocate device memory. The pages have no
 * counterpart: it exists for code that may not call cudaMalloc or any
 * allocator where it combines (code inside an arena that owns all device
 * memory after start-up, or a plug-in of a runtime that forbids allocations
 * of its own) and that holds no ep_handle, whose workspace is an allocation.
 *
 * It computes what ep_combine computes, from the same ids instead of a
 * pending dispatch: output[s][t] = bf16( sum over the active ranks d that own
 * one of topk_ids[s][t]'s valid expert ids, ascending, of expert_output[d]
 * [s*tokens_per_rank + t] ), fp32 accumulator from +0.0, one
 * round-to-nearest-even; a token routed nowhere gets +0.0. Results are bit
 * for bit those of ep_combine after ep_dispatch with the same ids and mask.
 *  topk_ids[s]      device int32 [num_tokens[s], top_k] (read only)
 *  num_tokens       host int32 [ep_size], each in [0, tokens_per_rank]
 *  active_rank_mask bit d = rank d active; UINT64_MAX = all; no bit >= ep_size
 *  expert_output[d] device bf16 [ep_size*tokens_per_rank, hidden], 16-byte aligned
 *  output[s]        device bf16 [num_tokens[s], hidden], 16-byte aligned
 *  stream           cudaStream_t to queue the two kernels on
 * Scratch: the routing bit set of every slot lives in one file-scope device
 * array of EP_NOALLOC_MAX_SLOTS entries (512 KB), held by every GPU that
 * loads the library until the process exits; ep_size * tokens_per_rank
 * beyond that returns EP_ERR_INVALID_ARG. Each call rewrites every entry it
 * reads, so nothing needs clearing, but all calls on a device share the
 * array: calls whose GPU work overlaps (e.g. on two streams) race.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. The address is kept for the rest of the
 * process: this assumes the device's primary context lives as long as the
 * process (after a cudaDeviceReset the kept address is stale). It calls no
 * allocator: no cudaMalloc, no cudaFree, no allocating library routine. */
ep_status ep_combine_noalloc(int ep_size, int num_experts, int top_k, int hidden,
                             int tokens_per_rank, const int32_t *num_tokens,
                             const int32_t *const *topk_ids, uint64_t active_rank_mask,
                             const void *const *expert_output, void *const *output,
                             void *stream);

#ifdef __cplusplus
}
#endif
#endif /* EP_GB300_H */
