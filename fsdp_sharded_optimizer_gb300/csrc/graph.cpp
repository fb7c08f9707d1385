// graph.cpp -- zero3_graph: one ZeRO-3 step of fixed buffers captured once as
// a CUDA graph (zero3_graph_create) and replayed once per step
// (zero3_graph_launch).
//
// The step is the one zero3_step (or zero3_step_f32grads) issues: the forward gathers, the backward
// gathers and per-unit reduce-scatter + AdamW ("Data parallelism, ZeRO and
// FSDP", "How FSDP implements ZeRO-3", steps 2-5), side-stream prefetch and
// two full-unit buffers.  Stream capture turns its event records and waits
// into graph edges, so a replay hands the GPU the whole dependency structure
// at once instead of one launch and one event at a time.  That matters for
// models of many small units, whose fused launches last tens of microseconds.
//
// What changes from step to step is the step number t (the bias corrections)
// and, with a schedule, lr / betas / eps / weight decay: the fp32 AdamW
// scalars, which the fused kernel takes by value.  The capture records every
// fused-step node it creates, and zero3_graph_launch rewrites those nodes'
// scalars in the instantiated graph before each replay.  The gathers and the
// clipping kernels take nothing that changes.
#include <new>
#include <vector>

#include "zero_internal.h"

struct zero3_graph {
    int device;
    int32_t n_ranks;
    cudaGraph_t graph;
    cudaGraphExec_t exec;
    zero::StepNodeList* nodes;
};

using namespace zero;

namespace {

// Turns the capture's direct edge from -> to (a kernel node to a kernel node,
// default type) into a programmatic one: `to` may start as soon as every block
// of `from` has triggered its dependents.  Nothing changes when the capture
// made no such edge.
int make_programmatic(cudaGraph_t graph, cudaGraphNode_t from, cudaGraphNode_t to)
{
    size_t n = 0;
    int rc = cuda_status(cudaGraphNodeGetDependencies(to, nullptr, nullptr, &n));
    if (rc != ZERO_OK || n == 0) return rc;
    std::vector<cudaGraphNode_t> deps(n);
    std::vector<cudaGraphEdgeData> edges(n);
    if ((rc = cuda_status(cudaGraphNodeGetDependencies(to, deps.data(), edges.data(), &n))) !=
        ZERO_OK)
        return rc;
    for (size_t i = 0; i < n; ++i) {
        if (deps[i] != from || edges[i].type != cudaGraphDependencyTypeDefault ||
            edges[i].from_port != cudaGraphKernelNodePortDefault)
            continue;
        if ((rc = cuda_status(cudaGraphRemoveDependencies(graph, &from, &to, &edges[i], 1))) !=
            ZERO_OK)
            return rc;
        cudaGraphEdgeData e = {};
        e.from_port = cudaGraphKernelNodePortProgrammatic;
        e.type = cudaGraphDependencyTypeProgrammatic;
        return cuda_status(cudaGraphAddDependencies(graph, &from, &to, &e, 1));
    }
    return ZERO_OK;
}

// The backward pass updates the units in reverse order, each unit's fused
// launches following the previous unit's on the main stream.  Consecutive
// units touch disjoint parameters, so the edge from one unit's last launch
// to the next unit's first is made programmatic, like the edges between the
// chunks of one unit: the next unit's blocks take over the SMs the previous
// one's tail leaves idle.  The next unit's edge from its backward gather (the
// gather reads the shard the update writes) stays a full dependency, and every
// fused launch waits for its predecessors before it exits, so completion
// stays ordered.  On GPT-2-sized units (7 M parameters) the launch tails are
// a visible part of the step.
int chain_units(cudaGraph_t graph, const StepNodeList* nodes, const zero_unit_t* units,
                int32_t n_units)
{
    size_t idx = 0;
    cudaGraphNode_t prev_last = nullptr;
    for (int32_t pos = 0; pos < n_units; ++pos) {
        const int32_t u = n_units - 1 - pos;
        const int64_t c = chunk_count(units[u].n_padded / 8);
        cudaGraphNode_t first = step_node_at(nodes, idx);
        if (!first || c < 1) return ZERO_ECUDA;
        if (prev_last) {
            const int rc = make_programmatic(graph, prev_last, first);
            if (rc != ZERO_OK) return rc;
        }
        idx += static_cast<size_t>(c);
        prev_last = step_node_at(nodes, idx - 1);
    }
    return ZERO_OK;
}

// The gathers run one after another on the side stream.  Two consecutive
// gathers that write disjoint bytes (the two full-unit buffers alternate, and
// without resharding each unit has its own region) only read the parameter
// shards, so their stream-order edge is made programmatic too: the next
// gather's blocks fill the SMs as the previous one drains.  Its edge from the
// main stream's release of the buffer it overwrites stays a full dependency,
// so a gather into a buffer still in use waits as before.  A pair that writes
// the same bytes (the last forward and first backward gather of an odd number
// of units, both into the first buffer) keeps its full edge.
int chain_gathers(cudaGraph_t graph, const std::vector<GatherNode>& gathers)
{
    for (size_t i = 1; i < gathers.size(); ++i) {
        const GatherNode& a = gathers[i - 1];
        const GatherNode& b = gathers[i];
        if (a.dst < b.dst + b.size && b.dst < a.dst + a.size) continue;
        const int rc = make_programmatic(graph, a.node, b.node);
        if (rc != ZERO_OK) return rc;
    }
    return ZERO_OK;
}

} // namespace

namespace {

// Captures the step that issue() queues on capture_stream (and side_stream),
// joins its launches with programmatic edges and instantiates the graph.
template <typename Issue>
int create_graph(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                 const zero_hparams_t* hp, bool clip, int32_t reshard_after_forward,
                 cudaStream_t capture_stream, cudaStream_t side_stream, zero3_graph_t** out,
                 Issue issue)
{
    if (!out) return ZERO_EINVAL;
    *out = nullptr;
    // The legacy default stream cannot be captured.
    if (!units || n_units < 1 || n_ranks < 1 || n_ranks > ZERO_MAX_RANKS || !valid_hparams(hp) ||
        !capture_stream || capture_stream == cudaStreamLegacy || capture_stream == side_stream)
        return ZERO_EINVAL;
    cudaStreamCaptureStatus status = cudaStreamCaptureStatusNone;
    int rc = cuda_status(cudaStreamIsCapturing(capture_stream, &status));
    if (rc != ZERO_OK) return rc;
    if (status != cudaStreamCaptureStatusNone) return ZERO_EINVAL; // no nested capture
    int dev = 0;
    if ((rc = cuda_status(cudaGetDevice(&dev))) != ZERO_OK) return rc;
    if ((rc = preload_fused_kernels()) != ZERO_OK || (rc = preload_gather_kernel()) != ZERO_OK ||
        (clip && (rc = preload_clip_kernels()) != ZERO_OK) || (rc = preload_step_events()) != ZERO_OK)
        return rc;

    std::vector<GatherNode> gathers;
    try {
        gathers.reserve(2 * static_cast<size_t>(n_units));
    } catch (...) {
        return ZERO_ECUDA;
    }
    StepNodeList* nodes = step_nodes_begin();
    if (!nodes) return ZERO_ECUDA;
    gather_nodes_begin(&gathers);
    cudaError_t e = cudaStreamBeginCapture(capture_stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        step_nodes_end();
        gather_nodes_end();
        step_nodes_free(nodes);
        return cuda_status(e);
    }
    // The step checks every argument before it issues anything; a rejected
    // call leaves an empty capture behind, which is discarded below.
    rc = issue();
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(capture_stream, &graph);
    step_nodes_end();
    const bool gathers_logged = gather_nodes_end();
    if (rc == ZERO_OK && e != cudaSuccess) rc = cuda_status(e);
    // each unit's fused reduce-scatter + AdamW, in its chained launches
    int64_t expected = 0;
    for (int32_t u = 0; u < n_units && rc == ZERO_OK; ++u)
        expected += chunk_count(units[u].n_padded / 8);
    if (rc == ZERO_OK && !step_nodes_ok(nodes, static_cast<size_t>(expected))) rc = ZERO_ECUDA;
    // a gather per unit in the forward pass, and again in the backward pass
    // when the forward pass reshards
    const size_t expected_gathers =
        static_cast<size_t>(n_units) * (reshard_after_forward ? 2 : 1);
    if (rc == ZERO_OK && (!gathers_logged || gathers.size() != expected_gathers)) rc = ZERO_ECUDA;
    if (rc == ZERO_OK) rc = chain_units(graph, nodes, units, n_units);
    if (rc == ZERO_OK) rc = chain_gathers(graph, gathers);
    cudaGraphExec_t exec = nullptr;
    if (rc == ZERO_OK) rc = cuda_status(cudaGraphInstantiate(&exec, graph, 0));
    zero3_graph_t* g = nullptr;
    if (rc == ZERO_OK) {
        g = new (std::nothrow) zero3_graph_t{dev, n_ranks, graph, exec, nodes};
        if (!g) rc = ZERO_ECUDA;
    }
    if (rc != ZERO_OK) {
        if (exec) cudaGraphExecDestroy(exec);
        if (graph) cudaGraphDestroy(graph);
        step_nodes_free(nodes);
        return rc;
    }
    *out = g;
    return ZERO_OK;
}

} // namespace

extern "C" int zero3_graph_create(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                                  const uint16_t* const* grads, float* const* master,
                                  float* const* m, float* const* v,
                                  uint16_t* const* shard_bf16, uint16_t* full_a,
                                  uint16_t* full_b, const zero_hparams_t* hp,
                                  const zero_clip_t* clip, int32_t reshard_after_forward,
                                  cudaStream_t capture_stream, cudaStream_t side_stream,
                                  zero3_graph_t** out)
{
    return create_graph(units, n_units, n_ranks, hp, clip != nullptr, reshard_after_forward,
                        capture_stream, side_stream, out, [&] {
                            return zero3_step(units, n_units, n_ranks, grads, 1, master, m, v,
                                              shard_bf16, full_a, full_b, hp, nullptr, clip,
                                              reshard_after_forward, capture_stream,
                                              side_stream);
                        });
}

extern "C" int zero3_graph_create_f32grads(const zero_unit_t* units, int32_t n_units,
                                           int32_t n_ranks, const float* const* grads,
                                           float* const* master, float* const* m,
                                           float* const* v, uint16_t* const* shard_bf16,
                                           uint16_t* full_a, uint16_t* full_b,
                                           const zero_hparams_t* hp,
                                           int32_t reshard_after_forward,
                                           cudaStream_t capture_stream, cudaStream_t side_stream,
                                           zero3_graph_t** out)
{
    return create_graph(units, n_units, n_ranks, hp, false, reshard_after_forward,
                        capture_stream, side_stream, out, [&] {
                            return zero3_step_f32grads(units, n_units, n_ranks, grads, master, m,
                                                       v, shard_bf16, full_a, full_b, hp,
                                                       reshard_after_forward, capture_stream,
                                                       side_stream);
                        });
}

extern "C" int zero3_graph_launch(zero3_graph_t* graph, const zero_hparams_t* hp,
                                  cudaStream_t stream)
{
    if (!graph || !valid_hparams(hp)) return ZERO_EINVAL;
    int dev = 0;
    int rc = cuda_status(cudaGetDevice(&dev));
    if (rc != ZERO_OK) return rc;
    if (dev != graph->device) return ZERO_EINVAL;
    // Only later launches see the new scalars; a replay already queued keeps
    // the ones it was launched with.
    if ((rc = step_nodes_set_scalars(graph->nodes, graph->exec, make_scalars(hp, graph->n_ranks))) !=
        ZERO_OK)
        return rc;
    return cuda_status(cudaGraphLaunch(graph->exec, stream));
}

extern "C" int zero3_graph_destroy(zero3_graph_t* graph)
{
    if (!graph) return ZERO_OK;
    int rc = cuda_status(cudaGraphExecDestroy(graph->exec));
    const int rc2 = cuda_status(cudaGraphDestroy(graph->graph));
    if (rc == ZERO_OK) rc = rc2;
    step_nodes_free(graph->nodes);
    delete graph;
    return rc;
}
