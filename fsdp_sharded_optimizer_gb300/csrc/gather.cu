// gather.cu -- ZeRO-3 unit all-gather (zero3_gather_unit).
//
// Method: "Data parallelism, ZeRO and FSDP", "How FSDP implements ZeRO-3",
// steps 2-3 (a pre-forward hook, and again the backward pass, all-gathers the
// unit's bf16 parameters); "Data parallelism, collectives and ZeRO/FSDP",
// "Collectives" (every rank gets all shards).
//
// On one GPU the all-gather is a bit copy of the N_d rank shards of a unit
// into one full buffer: 2 bytes read + 2 bytes written per parameter.  The
// grid is two-dimensional -- y is the source rank, x strides over that rank's
// shard -- so no thread divides to find its owner, and each thread keeps
// kUnroll independent 16-byte loads in flight before it stores.
#include "device.cuh"
#include "zero_internal.h"

namespace zero {
namespace {

constexpr int kBlock = 256;
constexpr int kUnroll = 4;

struct Sources {
    const uint4* src[ZERO_MAX_RANKS]; // rank k's shard of this unit
};

__global__ void __launch_bounds__(kBlock)
gather_kernel(const __grid_constant__ Sources S, uint4* __restrict__ dst, int64_t shard_vec)
{
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
}

} // namespace

int preload_gather_kernel()
{
    return persistent_blocks(reinterpret_cast<const void*>(gather_kernel), kBlock, 0) > 0
               ? ZERO_OK
               : ZERO_ECUDA;
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
    const int max_blocks = persistent_blocks(reinterpret_cast<const void*>(gather_kernel),
                                             kBlock, 0);
    if (max_blocks <= 0) return ZERO_ECUDA;
    const int64_t tiles = (shard_vec + kBlock * kUnroll - 1) / (kBlock * kUnroll);
    int64_t gx = (max_blocks + n_ranks - 1) / n_ranks; // fill the GPU once across ranks
    if (gx > tiles) gx = tiles;
    if (gx < 1) gx = 1;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(n_ranks));
    gather_kernel<<<grid, kBlock, 0, stream>>>(S, reinterpret_cast<uint4*>(full_unit), shard_vec);
    return cuda_status(cudaGetLastError());
}
