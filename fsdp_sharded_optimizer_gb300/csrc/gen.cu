// gen.cu -- harness kernels: seeded synthetic gradients and master weights,
// and the fp32 -> bf16 cast of initial weights.  None of this is the method;
// it fills device buffers with reproducible inputs without a host round trip.
//
// Generator: SplitMix64 (Steele, Lea and Flood, OOPSLA 2014; the constants
// of Vigna's public-domain splitmix64.c).  Output number i of a stream whose
// state starts at s is finalise(s + (i+1)*gamma), so every element is drawn
// independently.  A stream key is the first output of a stream seeded by the
// previous key xor the next field: seed, then stream id, step and rank.  A
// value sums the four 16-bit lanes of one output, centres the sum at 131070
// in integers and scales it by one fp32 constant sigma/sqrt((2^32-1)/3).
// With outliers on, a value whose own stream's next output is 0 mod 100 is
// multiplied by 100.
#include "device.cuh"
#include "zero_internal.h"

#include <cmath>

namespace zero {
namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr int kBlock = 256;

__host__ __device__ __forceinline__ uint64_t finalise(uint64_t z)
{
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t nth_output(uint64_t state, uint64_t i)
{
    return finalise(state + (i + 1) * kGamma);
}

uint64_t stream_key(uint64_t seed, uint64_t stream, uint64_t step, uint64_t rank)
{
    uint64_t key = nth_output(seed, 0);
    key = nth_output(key ^ stream, 0);
    key = nth_output(key ^ step, 0);
    return nth_output(key ^ rank, 0);
}

float value_scale(double sigma) { return static_cast<float>(sigma / std::sqrt(4294967295.0 / 3.0)); }

__device__ __forceinline__ float draw(uint64_t key, uint64_t index, float scale, bool outliers)
{
    const uint64_t h = nth_output(key, index);
    const int32_t lanes = static_cast<int32_t>(h & 0xFFFFu) + static_cast<int32_t>((h >> 16) & 0xFFFFu) +
                          static_cast<int32_t>((h >> 32) & 0xFFFFu) + static_cast<int32_t>(h >> 48);
    float z = __fmul_rn(__int2float_rn(lanes - 131070), scale);
    if (outliers && nth_output(h, 0) % 100u == 0u) z = __fmul_rn(z, 100.0f);
    return z;
}

struct GradArgs {
    uint4* dst[ZERO_MAX_RANKS];
    uint64_t key[ZERO_MAX_RANKS];
};

// y = rank; x strides over the unit's vectors of 8 elements.
__global__ void __launch_bounds__(kBlock)
gen_grads_kernel(const __grid_constant__ GradArgs A, int64_t n_vec, int64_t n_params,
                 int64_t param_offset, float scale, int outliers)
{
    const int r = blockIdx.y;
    const uint64_t key = A.key[r];
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; q < n_vec;
         q += static_cast<int64_t>(gridDim.x) * kBlock) {
        uint32_t b[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int64_t j = q * 8 + e;
            b[e] = j < n_params
                       ? dev::bf16_rne(draw(key, static_cast<uint64_t>(param_offset + j), scale,
                                            outliers != 0))
                       : 0u;
        }
        dev::st_stream(A.dst[r] + q, make_uint4(b[0] | (b[1] << 16), b[2] | (b[3] << 16),
                                                b[4] | (b[5] << 16), b[6] | (b[7] << 16)));
    }
}

struct GradArgsF32 {
    float4* dst[ZERO_MAX_RANKS];
    uint64_t key[ZERO_MAX_RANKS];
};

// The same draws kept in fp32 (no bf16 rounding): inputs of the fp32-gradient path.
__global__ void __launch_bounds__(kBlock)
gen_grads_f32_kernel(const __grid_constant__ GradArgsF32 A, int64_t n_vec, int64_t n_params,
                     int64_t param_offset, float scale, int outliers)
{
    const int r = blockIdx.y;
    const uint64_t key = A.key[r];
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; q < n_vec;
         q += static_cast<int64_t>(gridDim.x) * kBlock) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int64_t j = q * 8 + e;
            x[e] = j < n_params
                       ? draw(key, static_cast<uint64_t>(param_offset + j), scale, outliers != 0)
                       : 0.0f;
        }
        dev::st_stream(A.dst[r] + 2 * q, make_float4(x[0], x[1], x[2], x[3]));
        dev::st_stream(A.dst[r] + 2 * q + 1, make_float4(x[4], x[5], x[6], x[7]));
    }
}

struct MasterArgs {
    float4* dst[ZERO_MAX_RANKS]; // rank k's shard storage at this unit's offset
};

// y = owner rank k; x strides over the owner's shard in vectors of 8.
__global__ void __launch_bounds__(kBlock)
gen_master_kernel(const __grid_constant__ MasterArgs A, uint64_t key, int64_t shard_len,
                  int64_t n_params, int64_t param_offset, float scale)
{
    const int k = blockIdx.y;
    const int64_t shard_vec = shard_len / 8;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; q < shard_vec;
         q += static_cast<int64_t>(gridDim.x) * kBlock) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int64_t local = static_cast<int64_t>(k) * shard_len + q * 8 + e;
            x[e] = local < n_params ? draw(key, static_cast<uint64_t>(param_offset + local), scale, false)
                                    : 0.0f;
        }
        A.dst[k][2 * q] = make_float4(x[0], x[1], x[2], x[3]);
        A.dst[k][2 * q + 1] = make_float4(x[4], x[5], x[6], x[7]);
    }
}

__global__ void __launch_bounds__(kBlock)
cast_bf16_kernel(const float4* __restrict__ src, uint4* __restrict__ dst, int64_t n_vec)
{
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; q < n_vec;
         q += static_cast<int64_t>(gridDim.x) * kBlock) {
        const float4 a = src[2 * q], b = src[2 * q + 1];
        dst[q] = make_uint4(dev::pack_bf16x2(a.x, a.y), dev::pack_bf16x2(a.z, a.w),
                            dev::pack_bf16x2(b.x, b.y), dev::pack_bf16x2(b.z, b.w));
    }
}

unsigned grid_x(const void* kernel, int64_t work_vec, int rows)
{
    const int max_blocks = persistent_blocks(kernel, kBlock, 0);
    int64_t gx = (max_blocks + rows - 1) / rows;
    const int64_t need = (work_vec + kBlock - 1) / kBlock;
    if (gx > need) gx = need;
    return static_cast<unsigned>(gx < 1 ? 1 : gx);
}

bool unit_ok(const zero_unit_t* u, int32_t n_ranks)
{
    return u && n_ranks >= 1 && n_ranks <= ZERO_MAX_RANKS && u->n_params > 0 &&
           u->n_params <= u->n_padded && u->shard_len > 0 && u->shard_len % 8 == 0 &&
           u->shard_len * n_ranks == u->n_padded && u->shard_offset >= 0 &&
           u->shard_offset % 8 == 0 && u->param_offset >= 0;
}

} // namespace
} // namespace zero

using namespace zero;

extern "C" int zero_gen_grads_unit(uint64_t seed, int64_t step, double sigma, int32_t outliers,
                                   const zero_unit_t* unit, int32_t n_ranks,
                                   uint16_t* const* unit_grads, cudaStream_t stream)
{
    if (!unit_ok(unit, n_ranks) || step < 0 || !(sigma >= 0) || !std::isfinite(sigma))
        return ZERO_EINVAL;
    int rc = check_table(unit_grads, n_ranks);
    if (rc != ZERO_OK) return rc;
    GradArgs A = {};
    for (int32_t r = 0; r < n_ranks; ++r) {
        A.dst[r] = reinterpret_cast<uint4*>(unit_grads[r]);
        A.key[r] = stream_key(seed, 1, static_cast<uint64_t>(step), static_cast<uint64_t>(r));
    }
    const int64_t n_vec = unit->n_padded / 8;
    const dim3 grid(grid_x(reinterpret_cast<const void*>(gen_grads_kernel), n_vec, n_ranks),
                    static_cast<unsigned>(n_ranks));
    gen_grads_kernel<<<grid, kBlock, 0, stream>>>(A, n_vec, unit->n_params, unit->param_offset,
                                                  value_scale(sigma), outliers);
    return cuda_status(cudaGetLastError());
}

extern "C" int zero_gen_master(uint64_t seed, double sigma, const zero_unit_t* units,
                               int32_t n_units, int32_t n_ranks, float* const* master,
                               cudaStream_t stream)
{
    if (!units || n_units < 1 || !(sigma >= 0) || !std::isfinite(sigma)) return ZERO_EINVAL;
    for (int32_t u = 0; u < n_units; ++u)
        if (!unit_ok(&units[u], n_ranks)) return ZERO_EINVAL;
    int rc = check_table(master, n_ranks);
    if (rc != ZERO_OK) return rc;
    const uint64_t key = stream_key(seed, 0, 0, 0);
    const float scale = value_scale(sigma);
    for (int32_t u = 0; u < n_units; ++u) {
        MasterArgs A = {};
        for (int32_t k = 0; k < n_ranks; ++k)
            A.dst[k] = reinterpret_cast<float4*>(master[k] + units[u].shard_offset);
        const dim3 grid(grid_x(reinterpret_cast<const void*>(gen_master_kernel),
                               units[u].shard_len / 8, n_ranks),
                        static_cast<unsigned>(n_ranks));
        gen_master_kernel<<<grid, kBlock, 0, stream>>>(A, key, units[u].shard_len,
                                                       units[u].n_params, units[u].param_offset,
                                                       scale);
        if ((rc = cuda_status(cudaGetLastError())) != ZERO_OK) return rc;
    }
    return ZERO_OK;
}

extern "C" int zero_cast_bf16(const float* src, uint16_t* dst, int64_t n, cudaStream_t stream)
{
    if (!src || !dst || n < 0 || n % 8 != 0) return ZERO_EINVAL;
    if (!aligned16(src) || !aligned16(dst)) return ZERO_EALIGN;
    if (n == 0) return ZERO_OK;
    const int64_t n_vec = n / 8;
    cast_bf16_kernel<<<grid_x(reinterpret_cast<const void*>(cast_bf16_kernel), n_vec, 1), kBlock, 0,
                       stream>>>(reinterpret_cast<const float4*>(src), reinterpret_cast<uint4*>(dst),
                                 n_vec);
    return cuda_status(cudaGetLastError());
}

extern "C" int zero_gen_grads_unit_f32(uint64_t seed, int64_t step, double sigma, int32_t outliers,
                                       const zero_unit_t* unit, int32_t n_ranks,
                                       float* const* unit_grads, cudaStream_t stream)
{
    if (!unit_ok(unit, n_ranks) || step < 0 || !(sigma >= 0) || !std::isfinite(sigma))
        return ZERO_EINVAL;
    int rc = check_table(unit_grads, n_ranks);
    if (rc != ZERO_OK) return rc;
    GradArgsF32 A = {};
    for (int32_t r = 0; r < n_ranks; ++r) {
        A.dst[r] = reinterpret_cast<float4*>(unit_grads[r]);
        A.key[r] = stream_key(seed, 1, static_cast<uint64_t>(step), static_cast<uint64_t>(r));
    }
    const int64_t n_vec = unit->n_padded / 8;
    const dim3 grid(grid_x(reinterpret_cast<const void*>(gen_grads_f32_kernel), n_vec, n_ranks),
                    static_cast<unsigned>(n_ranks));
    gen_grads_f32_kernel<<<grid, kBlock, 0, stream>>>(A, n_vec, unit->n_params, unit->param_offset,
                                                      value_scale(sigma), outliers);
    return cuda_status(cudaGetLastError());
}
