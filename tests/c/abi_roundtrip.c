/*
 * abi_roundtrip.c -- drives the C ABI of include/ep.h from plain C (no
 * Python, no torch): the hand-worked two-rank example of
 * tests/golden/worked_example.json, dispatched and combined on the GPU.
 *
 * ep_size 2, 4 experts (0,1 on rank 0; 2,3 on rank 1), top_k 2, hidden 8
 * bf16, 3 tokens per rank. Rank 0 sends ids {0,1} and {1,3}; rank 1 sends
 * {2,3}. Checks every receive id row, the routed hidden rows, and three
 * combine outputs worked by hand; then a second round through
 * ep_dispatch_ex with device-side token counts (rank 0 sends only its first
 * token); then the first round again as a partitioned group of two
 * partitions. Exit status 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ep.h"

#define H 8
#define T 3
#define EP 2

static int failures = 0;

static void expect(int cond, const char *what)
{
    if (!cond) {
        fprintf(stderr, "FAIL: %s\n", what);
        ++failures;
    }
}

static int ok(ep_status st, const char *call)
{
    if (st != EP_OK) {
        fprintf(stderr, "%s failed: status %d (%s)\n", call, (int)st, ep_last_error());
        return 0;
    }
    return 1;
}

int main(void)
{
    if (!ep_is_supported()) {
        fprintf(stderr, "no sm_103 device\n");
        return 2;
    }
    /* source rows: bf16 bits, distinct per token */
    uint16_t h0[2 * H], h1[1 * H];
    for (int i = 0; i < 2 * H; ++i)
        h0[i] = (uint16_t)(0x3F80 + i);
    for (int i = 0; i < H; ++i)
        h1[i] = (uint16_t)(0x4000 + i);
    const int32_t ids0[4] = {0, 1, 1, 3}, ids1[2] = {2, 3};

    void *d_h0, *d_h1, *d_i0, *d_i1, *d_o0, *d_o1;
    if (cudaMalloc(&d_h0, sizeof h0) || cudaMalloc(&d_h1, sizeof h1) || cudaMalloc(&d_i0, sizeof ids0) ||
        cudaMalloc(&d_i1, sizeof ids1) || cudaMalloc(&d_o0, 2 * H * 2) || cudaMalloc(&d_o1, 1 * H * 2)) {
        fprintf(stderr, "cudaMalloc failed\n");
        return 2;
    }
    cudaMemcpy(d_h0, h0, sizeof h0, cudaMemcpyHostToDevice);
    cudaMemcpy(d_h1, h1, sizeof h1, cudaMemcpyHostToDevice);
    cudaMemcpy(d_i0, ids0, sizeof ids0, cudaMemcpyHostToDevice);
    cudaMemcpy(d_i1, ids1, sizeof ids1, cudaMemcpyHostToDevice);

    ep_handle *h = NULL;
    if (!ok(ep_create(EP, 4, 2, H, T, EP_DTYPE_BF16, 0, &h), "ep_create"))
        return 1;

    const void *hidden[EP] = {d_h0, d_h1};
    const int32_t *ids[EP] = {(const int32_t *)d_i0, (const int32_t *)d_i1};
    const int32_t counts[EP] = {2, 1};
    ep_dispatch_result res;
    if (!ok(ep_dispatch(h, hidden, NULL, ids, NULL, counts, -1, UINT64_MAX, NULL, &res), "ep_dispatch"))
        return 1;
    expect(res.tokens_per_rank == T && res.ep_size == EP, "result geometry");
    expect(res.recv_scale == NULL && res.recv_topk_weights == NULL, "no scales or weights sent");
    expect(ep_dispatch(h, hidden, NULL, ids, NULL, counts, -1, UINT64_MAX, NULL, &res) == EP_ERR_STATE,
           "second dispatch is refused");

    /* receive id planes, rows s*T+t */
    const int32_t want[EP][EP * T][2] = {
        {{0, 1}, {1, 3}, {-1, -1}, {-1, -1}, {-1, -1}, {-1, -1}},
        {{-1, -1}, {1, 3}, {-1, -1}, {2, 3}, {-1, -1}, {-1, -1}},
    };
    for (int d = 0; d < EP; ++d) {
        int32_t got[EP * T][2];
        cudaMemcpy(got, res.recv_topk_ids[d], sizeof got, cudaMemcpyDeviceToHost);
        expect(memcmp(got, want[d], sizeof got) == 0, d == 0 ? "rank 0 id plane" : "rank 1 id plane");
    }
    /* routed hidden rows equal their source rows */
    uint16_t row[H];
    cudaMemcpy(row, (const char *)res.recv_hidden[0] + 1 * H * 2, sizeof row, cudaMemcpyDeviceToHost);
    expect(memcmp(row, h0 + H, sizeof row) == 0, "rank 0 receives token 1 of rank 0");
    cudaMemcpy(row, (const char *)res.recv_hidden[1] + 3 * H * 2, sizeof row, cudaMemcpyDeviceToHost);
    expect(memcmp(row, h1, sizeof row) == 0, "rank 1 receives token 0 of rank 1");

    /* expert outputs written into the combine-input buffers */
    void *cin[EP];
    for (int d = 0; d < EP; ++d)
        if (!ok(ep_get_combine_input_buffer(h, d, &cin[d]), "ep_get_combine_input_buffer"))
            return 1;
    uint16_t eo[EP][EP * T][H];
    for (int d = 0; d < EP; ++d)
        for (int r = 0; r < EP * T; ++r)
            for (int c = 0; c < H; ++c)
                eo[d][r][c] = 0x7FC1; /* NaN where nothing may be read */
    for (int c = 0; c < H; ++c) {
        eo[0][0][c] = 0x4000; /* token (0,0): rank 0 only -> 2.0 */
        eo[0][1][c] = 0x3F80; /* token (0,1): 1.0 + 2^-8 is a tie -> 1.0 */
        eo[1][1][c] = 0x3B80;
        eo[1][3][c] = 0x3FC0; /* token (1,0): rank 1 only -> 1.5 */
    }
    for (int d = 0; d < EP; ++d)
        cudaMemcpy(cin[d], eo[d], sizeof eo[d], cudaMemcpyHostToDevice);
    void *out[EP] = {d_o0, d_o1};
    if (!ok(ep_combine(h, NULL, out, UINT64_MAX, NULL), "ep_combine"))
        return 1;
    uint16_t o0[2][H], o1[1][H];
    cudaMemcpy(o0, d_o0, sizeof o0, cudaMemcpyDeviceToHost);
    cudaMemcpy(o1, d_o1, sizeof o1, cudaMemcpyDeviceToHost);
    for (int c = 0; c < H; ++c) {
        expect(o0[0][c] == 0x4000, "token (0,0) = 2.0");
        expect(o0[1][c] == 0x3F80, "token (0,1) rounds the tie to even");
        expect(o1[0][c] == 0x3FC0, "token (1,0) = 1.5");
    }
    expect(ep_combine(h, NULL, out, UINT64_MAX, NULL) == EP_ERR_STATE, "second combine is refused");

    /* A second round through ep_dispatch_ex with device-side token counts:
     * rank 0 may send 2 tokens (its host count is the maximum) but sends 1. */
    const int32_t dcounts[EP] = {1, 1};
    void *d_counts;
    if (cudaMalloc(&d_counts, 16)) {
        fprintf(stderr, "cudaMalloc failed\n");
        return 2;
    }
    cudaMemcpy(d_counts, dcounts, sizeof dcounts, cudaMemcpyHostToDevice);
    ep_dispatch_args args;
    memset(&args, 0, sizeof args);
    args.hidden = hidden;
    args.topk_ids = ids;
    args.num_tokens = counts;
    args.runtime_max_tokens_per_rank = -1;
    args.active_rank_mask = UINT64_MAX;
    args.num_tokens_device = (const int32_t *)((const char *)d_counts + 2);
    expect(ep_dispatch_ex(h, &args, NULL, &res) == EP_ERR_INVALID_ARG, "misaligned device counts are refused");
    args.num_tokens_device = (const int32_t *)d_counts;
    if (!ok(ep_dispatch_ex(h, &args, NULL, &res), "ep_dispatch_ex with device counts"))
        return 1;
    const int32_t want2[EP][EP * T][2] = {
        {{0, 1}, {-1, -1}, {-1, -1}, {-1, -1}, {-1, -1}, {-1, -1}},
        {{-1, -1}, {-1, -1}, {-1, -1}, {2, 3}, {-1, -1}, {-1, -1}},
    };
    for (int d = 0; d < EP; ++d) {
        int32_t got[EP * T][2];
        cudaMemcpy(got, res.recv_topk_ids[d], sizeof got, cudaMemcpyDeviceToHost);
        expect(memcmp(got, want2[d], sizeof got) == 0, "id planes follow the device counts");
    }
    uint16_t sentinel[2][H];
    for (int i = 0; i < 2 * H; ++i)
        sentinel[i / H][i % H] = 0x7FC1;
    cudaMemcpy(d_o0, sentinel, sizeof sentinel, cudaMemcpyHostToDevice);
    /* the combine-input buffers still hold the expert outputs written above */
    if (!ok(ep_combine(h, NULL, out, UINT64_MAX, NULL), "ep_combine after device counts"))
        return 1;
    cudaMemcpy(o0, d_o0, sizeof o0, cudaMemcpyDeviceToHost);
    cudaMemcpy(o1, d_o1, sizeof o1, cudaMemcpyDeviceToHost);
    for (int c = 0; c < H; ++c) {
        expect(o0[0][c] == 0x4000, "device counts: token (0,0) = 2.0");
        expect(o0[1][c] == 0x7FC1, "device counts: the row past rank 0's count is left alone");
        expect(o1[0][c] == 0x3FC0, "device counts: token (1,0) = 1.5");
    }
    cudaFree(d_counts);
    if (!ok(ep_destroy(h), "ep_destroy"))
        return 1;

    /* The same example as a partitioned group: two partitions of one rank
     * each, every partition with a handle and a workspace of its own. Each
     * dispatch writes its rank's tokens into both ranks' receive rows; each
     * combine reads both ranks' combine inputs. */
    ep_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.ep_size = EP;
    cfg.num_experts = 4;
    cfg.top_k = 2;
    cfg.hidden = H;
    cfg.max_tokens_per_rank = T;
    cfg.dtype = EP_DTYPE_BF16;
    cfg.scale_cols = EP_SCALE_COLS_DEFAULT;
    cfg.combine_dtype = EP_DTYPE_BF16;
    cfg.num_partitions = EP;
    ep_handle *part[EP];
    ep_partition_info info[EP];
    for (int g = 0; g < EP; ++g) {
        cfg.partition = g;
        if (!ok(ep_create_ex(&cfg, NULL, 0, &part[g]), "ep_create_ex (partition)") ||
            !ok(ep_partition_info_of(part[g], &info[g]), "ep_partition_info_of"))
            return 1;
        expect(info[g].first_rank == g && info[g].num_ranks == 1, "one rank per partition");
    }
    expect(ep_dispatch(part[0], hidden, NULL, ids, NULL, counts, -1, UINT64_MAX, NULL, &res) == EP_ERR_STATE,
           "an unconnected partition refuses to dispatch");
    for (int g = 0; g < EP; ++g)
        if (!ok(ep_partition_connect(part[g], info, EP), "ep_partition_connect"))
            return 1;
    ep_dispatch_result pres[EP];
    for (int g = 0; g < EP; ++g)
        if (!ok(ep_dispatch(part[g], &hidden[g], NULL, &ids[g], NULL, &counts[g], -1, UINT64_MAX, NULL, &pres[g]),
                "ep_dispatch (partition)"))
            return 1;
    for (int g = 0; g < EP; ++g) {
        int32_t got[EP * T][2];
        expect(pres[g].first_rank == g && pres[g].num_ranks == 1, "partition result geometry");
        cudaMemcpy(got, pres[g].recv_topk_ids[0], sizeof got, cudaMemcpyDeviceToHost);
        expect(memcmp(got, want[g], sizeof got) == 0, "partition id plane");
        void *buf;
        if (!ok(ep_get_combine_input_buffer(part[g], g, &buf), "ep_get_combine_input_buffer (partition)"))
            return 1;
        cudaMemcpy(buf, eo[g], sizeof eo[g], cudaMemcpyHostToDevice);
    }
    cudaMemcpy(row, (const char *)pres[1].recv_hidden[0] + 3 * H * 2, sizeof row, cudaMemcpyDeviceToHost);
    expect(memcmp(row, h1, sizeof row) == 0, "partition 1 receives token 0 of rank 1");
    cudaMemcpy(row, (const char *)pres[1].recv_hidden[0] + 1 * H * 2, sizeof row, cudaMemcpyDeviceToHost);
    expect(memcmp(row, h0 + H, sizeof row) == 0, "partition 1 receives token 1 of rank 0 from partition 0");
    for (int g = 0; g < EP; ++g)
        if (!ok(ep_combine(part[g], NULL, &out[g], UINT64_MAX, NULL), "ep_combine (partition)"))
            return 1;
    cudaMemcpy(o0, d_o0, sizeof o0, cudaMemcpyDeviceToHost);
    cudaMemcpy(o1, d_o1, sizeof o1, cudaMemcpyDeviceToHost);
    for (int c = 0; c < H; ++c) {
        expect(o0[0][c] == 0x4000, "partitions: token (0,0) = 2.0");
        expect(o0[1][c] == 0x3F80, "partitions: token (0,1) sums ranks 0 and 1 across partitions");
        expect(o1[0][c] == 0x3FC0, "partitions: token (1,0) = 1.5");
    }
    for (int g = 0; g < EP; ++g)
        if (!ok(ep_destroy(part[g]), "ep_destroy (partition)"))
            return 1;
    if (failures)
        return 1;
    printf("abi_roundtrip: ok\n");
    return 0;
}
