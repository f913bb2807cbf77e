/*
 * pdl_graph.c -- what a stream capture of ep_dispatch + ep_combine records,
 * with and without EP_LAUNCH_PDL, from plain C.
 *
 * The hand-worked two-rank example (ep_size 2, experts 0,1 on rank 0 and
 * 2,3 on rank 1, top_k 2, hidden 8 bf16, 3 tokens per rank) is captured into
 * a CUDA graph twice: once from a handle created with launch_flags 0 and
 * once with EP_LAUNCH_PDL. The graph's edges are read back
 * (cudaGraphGetEdges with edge data): with the flag the combine node hangs
 * on the dispatch node by a programmatic edge, without it by an ordinary one.
 * Each graph is then launched and its combine outputs checked against the
 * values worked by hand. Exit status 0 on success.
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

static int run(int flags)
{
    uint16_t h0[2 * H], h1[1 * H];
    for (int i = 0; i < 2 * H; ++i)
        h0[i] = (uint16_t)(0x3F80 + i);
    for (int i = 0; i < H; ++i)
        h1[i] = (uint16_t)(0x4000 + i);
    const int32_t ids0[4] = {0, 1, 1, 3}, ids1[2] = {2, 3};
    void *d_h0, *d_h1, *d_i0, *d_i1, *d_o0, *d_o1;
    if (cudaMalloc(&d_h0, sizeof h0) || cudaMalloc(&d_h1, sizeof h1) || cudaMalloc(&d_i0, sizeof ids0) ||
        cudaMalloc(&d_i1, sizeof ids1) || cudaMalloc(&d_o0, 2 * H * 2) || cudaMalloc(&d_o1, 1 * H * 2))
        return 2;
    cudaMemcpy(d_h0, h0, sizeof h0, cudaMemcpyHostToDevice);
    cudaMemcpy(d_h1, h1, sizeof h1, cudaMemcpyHostToDevice);
    cudaMemcpy(d_i0, ids0, sizeof ids0, cudaMemcpyHostToDevice);
    cudaMemcpy(d_i1, ids1, sizeof ids1, cudaMemcpyHostToDevice);

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
    cfg.launch_flags = flags;
    ep_handle *h = NULL;
    if (ep_create_ex(&cfg, NULL, 0, &h) != EP_OK) {
        fprintf(stderr, "ep_create_ex: %s\n", ep_last_error());
        return 1;
    }
    /* one eager round first: first-use set-up happens outside the capture */
    const void *hidden[EP] = {d_h0, d_h1};
    const int32_t *ids[EP] = {(const int32_t *)d_i0, (const int32_t *)d_i1};
    const int32_t counts[EP] = {2, 1};
    void *out[EP] = {d_o0, d_o1};
    if (ep_dispatch(h, hidden, NULL, ids, NULL, counts, -1, UINT64_MAX, NULL, NULL) != EP_OK ||
        ep_combine(h, NULL, out, UINT64_MAX, NULL) != EP_OK) {
        fprintf(stderr, "eager round: %s\n", ep_last_error());
        return 1;
    }
    cudaDeviceSynchronize();

    cudaStream_t s;
    cudaGraph_t graph;
    cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    void *cin[EP];
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeGlobal) != cudaSuccess)
        return 2;
    int st = ep_dispatch(h, hidden, NULL, ids, NULL, counts, -1, UINT64_MAX, s, NULL);
    for (int d = 0; st == EP_OK && d < EP; ++d)
        st = ep_get_combine_input_buffer(h, d, &cin[d]);
    if (st == EP_OK)
        st = ep_combine(h, NULL, out, UINT64_MAX, s);
    if (cudaStreamEndCapture(s, &graph) != cudaSuccess || st != EP_OK) {
        fprintf(stderr, "capture: %d %s\n", st, ep_last_error());
        return 1;
    }

    /* the captured nodes and edges */
    size_t n_nodes = 0, n_edges = 0;
    cudaGraphGetNodes(graph, NULL, &n_nodes);
    cudaGraphGetEdges(graph, NULL, NULL, NULL, &n_edges);
    expect(n_nodes == 2 && n_edges == 1, "the graph holds the two kernels and one edge between them");
    if (n_edges == 1) {
        cudaGraphNode_t from, to;
        cudaGraphEdgeData data;
        memset(&data, 0, sizeof data);
        if (cudaGraphGetEdges(graph, &from, &to, &data, &n_edges) != cudaSuccess)
            return 2;
        enum cudaGraphNodeType tf, tt;
        cudaGraphNodeGetType(from, &tf);
        cudaGraphNodeGetType(to, &tt);
        expect(tf == cudaGraphNodeTypeKernel && tt == cudaGraphNodeTypeKernel, "kernel to kernel");
        if (flags & EP_LAUNCH_PDL)
            expect(data.type == cudaGraphDependencyTypeProgrammatic, "EP_LAUNCH_PDL: a programmatic edge");
        else
            expect(data.type == cudaGraphDependencyTypeDefault, "without the flag: an ordinary edge");
        printf("flags %d: edge type %d, from port %d\n", flags, (int)data.type, (int)data.from_port);
    }

    /* expert outputs of the worked example, then the graph */
    uint16_t eo[EP][EP * T][H];
    for (int d = 0; d < EP; ++d)
        for (int r = 0; r < EP * T; ++r)
            for (int c = 0; c < H; ++c)
                eo[d][r][c] = 0x7FC1;
    for (int c = 0; c < H; ++c) {
        eo[0][0][c] = 0x4000;
        eo[0][1][c] = 0x3F80;
        eo[1][1][c] = 0x3B80;
        eo[1][3][c] = 0x3FC0;
    }
    for (int d = 0; d < EP; ++d)
        cudaMemcpy(cin[d], eo[d], sizeof eo[d], cudaMemcpyHostToDevice);
    cudaMemset(d_o0, 0, 2 * H * 2);
    cudaMemset(d_o1, 0, 1 * H * 2);
    cudaGraphExec_t exec;
    if (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess || cudaGraphLaunch(exec, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        fprintf(stderr, "graph launch: %s\n", cudaGetErrorString(cudaGetLastError()));
        return 2;
    }
    uint16_t o0[2][H], o1[1][H];
    cudaMemcpy(o0, d_o0, sizeof o0, cudaMemcpyDeviceToHost);
    cudaMemcpy(o1, d_o1, sizeof o1, cudaMemcpyDeviceToHost);
    for (int c = 0; c < H; ++c) {
        expect(o0[0][c] == 0x4000, "graph: token (0,0) = 2.0");
        expect(o0[1][c] == 0x3F80, "graph: token (0,1) rounds the tie to even");
        expect(o1[0][c] == 0x3FC0, "graph: token (1,0) = 1.5");
    }
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    cudaStreamDestroy(s);
    ep_destroy(h);
    cudaFree(d_h0);
    cudaFree(d_h1);
    cudaFree(d_i0);
    cudaFree(d_i1);
    cudaFree(d_o0);
    cudaFree(d_o1);
    return 0;
}

int main(void)
{
    if (!ep_is_supported()) {
        fprintf(stderr, "no sm_103 device\n");
        return 2;
    }
    int rc = run(0);
    if (rc == 0)
        rc = run(EP_LAUNCH_PDL);
    if (rc)
        return rc;
    if (failures)
        return 1;
    printf("pdl_graph: ok\n");
    return 0;
}
