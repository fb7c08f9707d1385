// zero_internal.h -- host-side helpers shared by the library's translation
// units (argument checks, per-device launch geometry, the fp32 step scalars).
#pragma once

#include <cmath>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "zero.h"

namespace zero {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks a host table of n device pointers: non-null and 16-byte aligned.
// Returns ZERO_OK, ZERO_EINVAL or ZERO_EALIGN.
template <typename T>
int check_table(T const* table, int32_t n)
{
    if (!table) return ZERO_EINVAL;
    for (int32_t i = 0; i < n; ++i) {
        if (!table[i]) return ZERO_EINVAL;
        if (!aligned16(table[i])) return ZERO_EALIGN;
    }
    return ZERO_OK;
}

// Hyper-parameters a step accepts: finite, step >= 1, betas in [0, 1),
// lr and eps and weight decay >= 0 (eps > 0 keeps the division defined).
bool valid_hparams(const zero_hparams_t* hp);

// The fp32 constants of one AdamW step, each computed in double from the
// double hyper-parameters and rounded once to fp32.
struct StepScalars {
    float b1, b2, omb1, omb2, bc1, bc2, lr, eps, wd, inv_n;
};
StepScalars make_scalars(const zero_hparams_t* hp, int32_t n_ranks);

// Persistent-grid size for a kernel on the current device: the SM count
// times the resident blocks per SM (computed once per device and kernel).
int persistent_blocks(const void* kernel, int block_threads, size_t dyn_smem);

// Splits a grid stride (in vectors) into whole shards and a remainder so
// that a grid-stride loop can advance (owner, position) without dividing.
struct StrideSplit {
    int64_t k, j;
};
inline StrideSplit split_stride(int64_t stride, int64_t shard_vec)
{
    return {stride / shard_vec, stride % shard_vec};
}

int cuda_status(cudaError_t e);

// Global-norm clipping: a fixed grid of kNormBlocks blocks writes one fp64
// partial sum each, so scratch holds kNormBlocks doubles (152 SMs x 8).
constexpr int kNormBlocks = 1216;
constexpr int64_t kNormScratchBytes = kNormBlocks * static_cast<int64_t>(sizeof(double));
// chained: the previous kernel on `stream` is a norm pass over other
// gradients; this one may start while it drains (programmatic dependent
// launch) and adds to the partials only once it has completed.
int grad_sqnorm(int32_t n_ranks, int64_t n_elems, const uint16_t* const* grads, int32_t accumulate,
                double* scratch, int64_t scratch_bytes, cudaStream_t stream,
                bool chained = false);
int clip_coef(const double* scratch, int64_t scratch_bytes, double max_norm, float* norm_coef,
              cudaStream_t stream);
int grad_reduce_sqnorm(int32_t n_ranks, int64_t n_elems, const uint16_t* const* grads,
                       float* const* grad_shard, int32_t accumulate, double* scratch,
                       int64_t scratch_bytes, cudaStream_t stream, bool chained = false);

// One unit's fused reduce-scatter + AdamW + bf16 shard write, as
// zero3_reduce_scatter_unit and its variants issue it: g from the rank
// gradients (bf16, or fp32 with f32) or, with g32, from the fp32 gradient
// shard storage (grads then holds its per-rank base pointers); clip = the
// device coefficient or nullptr.  chain_first: the last thing issued on
// `stream` was another unit's update and nothing else has been issued on it
// since (no event record or wait); the first chunk is then chained to it
// (programmatic dependent launch; the units touch disjoint elements).
// nonfinite: nullptr, or the device flag words of the fused finite check
// (bf16 rank gradients without clipping only).
int unit_update(const zero_unit_t* unit, int32_t n_ranks, const void* const* grads,
                float* const* master, float* const* m, float* const* v,
                uint16_t* const* shard_bf16, const zero_hparams_t* hp, const float* clip,
                cudaStream_t stream, bool f32, bool g32, bool chain_first,
                uint32_t* nonfinite = nullptr);

// CUDA-graph support (zero3_graph).  Between step_nodes_begin and
// step_nodes_end, every fused-step launch made on this thread into a stream
// that is being captured records its graph node and a copy of its arguments
// in the returned list; step_nodes_set_scalars later rewrites the AdamW
// scalars of all of them in an instantiated graph.  step_nodes_ok: no
// recording failed and exactly `expected` launches were recorded.
// Number of chained launches the fused step uses for n_vec vectors (a vector
// = 8 elements): ceil(n_vec / (ZERO_CHUNK_ELEMS / 8)); all but the last cover
// ZERO_CHUNK_ELEMS elements.
int64_t chunk_count(int64_t n_vec);

struct StepNodeList;
StepNodeList* step_nodes_begin(); // nullptr when out of host memory
void step_nodes_end();
bool step_nodes_ok(const StepNodeList* log, size_t expected);
int step_nodes_set_scalars(StepNodeList* log, cudaGraphExec_t exec, const StepScalars& s);
void step_nodes_free(StepNodeList* log);
cudaGraphNode_t step_node_at(const StepNodeList* log, size_t i); // nullptr past the end

// Between gather_nodes_begin and gather_nodes_end, every gather launched on
// this thread into a stream being captured appends its graph node and the
// byte range it writes to `log`.  gather_nodes_end: false when a record
// failed (the log is then incomplete).
struct GatherNode {
    cudaGraphNode_t node;
    uintptr_t dst;  // first byte written
    uintptr_t size; // bytes written
};
void gather_nodes_begin(std::vector<GatherNode>* log);
bool gather_nodes_end();

// Load the kernels a ZeRO-3 step launches and cache their launch geometry,
// so that nothing is loaded or queried for the first time inside a capture.
int preload_fused_kernels();
int preload_gather_kernel();
int preload_clip_kernels();
int preload_step_events(); // zero3_step's per-thread events

} // namespace zero
