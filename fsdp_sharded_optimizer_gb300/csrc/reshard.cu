// reshard.cu -- zero_reshard_f32: one unit's per-rank fp32 state re-laid from
// one rank count to another, for a run restarted on a different N_d.
//
// Method ("Data parallelism, ZeRO and FSDP", "6. Where it shows up",
// checkpoints: sharded optimizer state has to be resharded when a run
// restarts on another N_d).
//
// Element i of the unit's flat order sits at rank i / S_from, position
// i % S_from, and moves to rank i / S_to, position i % S_to; the new layout's
// padding is written +0 whatever the old padding held.  Both shard lengths
// are multiples of 8, so every aligned group of 8 elements lies inside one
// rank in both layouts: a thread moves one group with two 16-byte loads and
// two 16-byte stores.  The grid is two-dimensional, y = the destination rank
// and x = groups of its shard, grid-striding; 8 bytes per parameter, bound by
// HBM bandwidth.  Not on the training step's path: it runs once per restart.
#include "device.cuh"
#include "zero_internal.h"

namespace zero {
namespace {

constexpr int kBlock = 256;
constexpr int64_t kMaxBlocksX = 1 << 16;

struct ReshardTables {
    const float4* src[ZERO_MAX_RANKS]; // old rank r's storage at the unit's shard offset
    float4* dst[ZERO_MAX_RANKS];       // new rank k's storage at the unit's shard offset
};

__global__ void __launch_bounds__(kBlock)
reshard_kernel(const __grid_constant__ ReshardTables T, int64_t n_params, int64_t from_groups,
               int64_t to_groups)
{
    const int64_t k = blockIdx.y; // destination rank
    float4* __restrict__ out = T.dst[k];
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; j < to_groups;
         j += static_cast<int64_t>(gridDim.x) * kBlock) {
        const int64_t q = k * to_groups + j; // group index in the unit's flat order
        const int64_t i0 = 8 * q;            // its first element
        float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f), b = a;
        if (i0 < n_params) {
            const int64_t r = q / from_groups; // source rank
            const float4* p = T.src[r] + 2 * (q - r * from_groups);
            a = dev::ld_stream(p);
            b = dev::ld_stream(p + 1);
            if (i0 + 8 > n_params) { // the unit's last group: the rest is padding
                float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (i0 + e >= n_params) x[e] = 0.0f;
                a = make_float4(x[0], x[1], x[2], x[3]);
                b = make_float4(x[4], x[5], x[6], x[7]);
            }
        }
        dev::st_stream(out + 2 * j, a);
        dev::st_stream(out + 2 * j + 1, b);
    }
}

bool layout_ok(const zero_unit_t* u, int32_t n_ranks)
{
    return u && n_ranks >= 1 && n_ranks <= ZERO_MAX_RANKS && u->n_params > 0 &&
           u->n_padded >= u->n_params && u->shard_len > 0 && u->shard_len % 8 == 0 &&
           u->shard_len * n_ranks == u->n_padded && u->shard_offset >= 0 &&
           u->shard_offset % 8 == 0;
}

} // namespace
} // namespace zero

using namespace zero;

extern "C" int zero_reshard_f32(const zero_unit_t* from_unit, int32_t n_from,
                                const float* const* src, const zero_unit_t* to_unit,
                                int32_t n_to, float* const* dst, cudaStream_t stream)
{
    if (!layout_ok(from_unit, n_from) || !layout_ok(to_unit, n_to) ||
        from_unit->n_params != to_unit->n_params)
        return ZERO_EINVAL;
    int rc = check_table(src, n_from);
    if (rc != ZERO_OK) return rc;
    if ((rc = check_table(dst, n_to)) != ZERO_OK) return rc;
    ReshardTables T = {};
    for (int32_t r = 0; r < n_from; ++r)
        T.src[r] = reinterpret_cast<const float4*>(src[r] + from_unit->shard_offset);
    for (int32_t k = 0; k < n_to; ++k)
        T.dst[k] = reinterpret_cast<float4*>(dst[k] + to_unit->shard_offset);
    const int64_t to_groups = to_unit->shard_len / 8;
    const int64_t blocks = (to_groups + kBlock - 1) / kBlock;
    const dim3 grid(static_cast<unsigned>(blocks < kMaxBlocksX ? blocks : kMaxBlocksX),
                    static_cast<unsigned>(n_to));
    reshard_kernel<<<grid, kBlock, 0, stream>>>(T, from_unit->n_params, from_unit->shard_len / 8,
                                                to_groups);
    return cuda_status(cudaGetLastError());
}
