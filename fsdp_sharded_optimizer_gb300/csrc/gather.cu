// gather.cu -- ZeRO-3 unit all-gather (zero3_gather_unit).
//
// Method: "Data parallelism, ZeRO and FSDP", "How FSDP implements ZeRO-3",
// steps 2-3 (a pre-forward hook, and again the backward pass, all-gathers the
// unit's bf16 parameters); "Data parallelism, collectives and ZeRO/FSDP",
// "Collectives" (every rank gets all shards).
//
// On one GPU the all-gather is a bit copy of the N_d rank shards of a unit
// into one full buffer: 2 bytes read + 2 bytes written per parameter.  The
// grid is two-dimensional -- y is the source rank, x the tiles of that rank's
// shard -- so no thread divides to find its owner.  Each block copies one
// tile of kBlock x kUnroll 16-byte vectors (32 KB), each thread keeping its
// kUnroll loads in flight before it stores.  One block per tile, not a
// persistent grid: a persistent grid gives every block the same number of
// tiles and ends with a partial round (4.4 tiles per block on a Llama-1.1B
// unit), while single-tile blocks are balanced by the block scheduler.
// Measured on GB300 (gathers alone, back to back): Llama-7B units 6.12 ->
// 6.87 TB/s, Llama-1.1B 5.82 -> 6.17 TB/s, GPT-2 blocks unchanged.
#include "device.cuh"
#include "zero_internal.h"

namespace zero {
namespace {

constexpr int kBlock = 256;
constexpr int kUnroll = 8;

struct Sources {
    const uint4* src[ZERO_MAX_RANKS]; // rank k's shard of this unit
};

__global__ void __launch_bounds__(kBlock)
gather_kernel(const __grid_constant__ Sources S, uint4* __restrict__ dst, int64_t shard_vec)
{
    // In a graph, consecutive gathers may be joined by a programmatic edge
    // (they write different buffers): this gather lets the next one start
    // once all its blocks run, and completes only after its predecessor.  Both
    // instructions do nothing otherwise.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int k = blockIdx.y;
    const uint4* __restrict__ src = S.src[k];
    uint4* __restrict__ out = dst + static_cast<int64_t>(k) * shard_vec;
    const int64_t tile = static_cast<int64_t>(kBlock) * kUnroll;
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * tile; base < shard_vec;
         base += static_cast<int64_t>(gridDim.x) * tile) {
        uint4 x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t j = base + u * kBlock + threadIdx.x;
            if (j < shard_vec) x[u] = dev::ld_stream(src + j);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t j = base + u * kBlock + threadIdx.x;
            if (j < shard_vec) dev::st_stream(out + j, x[u]);
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The gathers launched on this thread while a capture log is installed
// (zero3_graph_create), in issue order.
thread_local std::vector<GatherNode>* t_gather_log = nullptr;
thread_local bool t_gather_log_failed = false;

} // namespace

void gather_nodes_begin(std::vector<GatherNode>* log)
{
    t_gather_log = log;
    t_gather_log_failed = false;
}

bool gather_nodes_end()
{
    t_gather_log = nullptr;
    return !t_gather_log_failed;
}

int preload_gather_kernel()
{
    cudaFuncAttributes a;
    return cudaFuncGetAttributes(&a, gather_kernel) == cudaSuccess ? ZERO_OK : ZERO_ECUDA;
}

} // namespace zero

using namespace zero;

extern "C" int zero3_gather_unit(const zero_unit_t* unit, int32_t n_ranks,
                                 const uint16_t* const* shard_bf16, uint16_t* full_unit,
                                 cudaStream_t stream)
{
    if (!unit || n_ranks < 1 || n_ranks > ZERO_MAX_RANKS || unit->shard_len <= 0 ||
        unit->shard_len % 8 != 0 || unit->shard_len * n_ranks != unit->n_padded ||
        unit->shard_offset < 0 || unit->shard_offset % 8 != 0 || !full_unit)
        return ZERO_EINVAL;
    int rc = check_table(shard_bf16, n_ranks);
    if (rc != ZERO_OK) return rc;
    if (!aligned16(full_unit)) return ZERO_EALIGN;

    Sources S = {};
    for (int32_t k = 0; k < n_ranks; ++k)
        S.src[k] = reinterpret_cast<const uint4*>(shard_bf16[k] + unit->shard_offset);
    const int64_t shard_vec = unit->shard_len / 8;
    const int64_t tiles = (shard_vec + kBlock * kUnroll - 1) / (kBlock * kUnroll);
    if (tiles > 0x7FFFFFFF) return ZERO_EINVAL; // grid.x limit (a shard of > 2^40 elements)
    const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(n_ranks));
    gather_kernel<<<grid, kBlock, 0, stream>>>(S, reinterpret_cast<uint4*>(full_unit), shard_vec);
    rc = cuda_status(cudaGetLastError());
    if (rc == ZERO_OK && t_gather_log) {
        cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
        const cudaGraphNode_t* deps = nullptr;
        const cudaGraphEdgeData* edges = nullptr;
        size_t n_deps = 0;
        if (cudaStreamGetCaptureInfo(stream, &st, nullptr, nullptr, &deps, &edges, &n_deps) !=
                cudaSuccess ||
            st != cudaStreamCaptureStatusActive || n_deps != 1) {
            t_gather_log_failed = true;
        } else {
            try {
                t_gather_log->push_back(GatherNode{
                    deps[0], reinterpret_cast<uintptr_t>(full_unit),
                    static_cast<uintptr_t>(unit->n_padded) * sizeof(uint16_t)});
            } catch (...) {
                t_gather_log_failed = true;
            }
        }
    }
    return rc;
}
