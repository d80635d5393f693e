// graph.cu — a whole decode step (or several) captured once as a CUDA graph and replayed with
// one launch ("DSpark in SGLang", LMSYS blog summary, A2 ragged verify over full CUDA graphs,
// figure 2: the variable windows are packed so that the step replays a captured graph).
//
// The library's kernels size themselves on the device (verify reads M from cu_seqlens; every
// grid is sized from B*gamma), so one graph serves every window allocation and tier. Kernels
// captured with programmatic dependent launch keep their programmatic edges in the graph, so a
// replay overlaps each kernel's start with the previous one's tail as eager launches do.
#include <new>

#include "common.cuh"

struct dspark_graph_s {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

namespace {

int cuda_fail(const char* what, cudaError_t e)
{
    cudaGetLastError();
    return dspark::fail(DSPARK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e),
                        cudaGetErrorName(e));
}

}  // namespace

extern "C" {

int dspark_graph_begin(cudaStream_t stream)
{
    if (stream == nullptr)
        return dspark::fail(DSPARK_ERR_INVALID_ARG,
                            "dspark_graph_begin: the legacy default stream cannot be captured");
    const cudaError_t e = cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail("dspark_graph_begin: cudaStreamBeginCapture", e);
    return DSPARK_OK;
}

int dspark_graph_end(cudaStream_t stream, dspark_graph* out)
{
    if (out == nullptr || stream == nullptr)
        return dspark::fail(DSPARK_ERR_INVALID_ARG, "dspark_graph_end: NULL stream or output");
    *out = nullptr;
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(stream, &g);
    if (e != cudaSuccess) {
        if (g != nullptr) cudaGraphDestroy(g);
        return cuda_fail("dspark_graph_end: cudaStreamEndCapture", e);
    }
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiateWithFlags(&exec, g, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(g);
        return cuda_fail("dspark_graph_end: cudaGraphInstantiateWithFlags", e);
    }
    dspark_graph h = new (std::nothrow) dspark_graph_s;
    if (h == nullptr) {
        cudaGraphExecDestroy(exec);
        cudaGraphDestroy(g);
        return dspark::fail(DSPARK_ERR_CUDA, "dspark_graph_end: out of host memory");
    }
    h->graph = g;
    h->exec = exec;
    *out = h;
    return DSPARK_OK;
}

int dspark_graph_launch(dspark_graph graph, cudaStream_t stream)
{
    if (graph == nullptr || graph->exec == nullptr)
        return dspark::fail(DSPARK_ERR_INVALID_ARG, "dspark_graph_launch: NULL graph");
    const cudaError_t e = cudaGraphLaunch(graph->exec, stream);
    if (e != cudaSuccess) return cuda_fail("dspark_graph_launch: cudaGraphLaunch", e);
    return DSPARK_OK;
}

int dspark_graph_destroy(dspark_graph graph)
{
    if (graph == nullptr) return DSPARK_OK;
    if (graph->exec != nullptr) cudaGraphExecDestroy(graph->exec);
    if (graph->graph != nullptr) cudaGraphDestroy(graph->graph);
    delete graph;
    return DSPARK_OK;
}

}  // extern "C"
