// noalloc.cu -- zero_clip_coef_units_noalloc: the global-norm clip coefficient
// (and each unit's gradient norm) with no caller-provided scratch.
//
// Some callers cannot allocate device memory: code that runs inside another
// framework whose memory pool owns the GPU and forbids raw allocations, a
// watchdog or monitoring thread that must not disturb the allocator of the
// training loop it observes, or a runtime that works inside a fixed memory
// budget.  This entry point serves them: the norm pass's partial sums live in a
// fixed file-scope device array that every GPU loading the library holds until
// the process exits, and the caller passes only its inputs and outputs.
//
// The array is shared by all calls on a device and keeps the last call's
// contents.  Every slot a call reads is written earlier in the same call (the
// block partials are overwritten for each unit, each unit's sum is written,
// not added), so nothing has to start at zero.  Calls whose GPU work overlaps
// -- on two streams at once, or from two host threads -- race on the array;
// order them on one stream.
#include <mutex>

#include "device.cuh"
#include "zero_internal.h"

namespace zero {
namespace {

constexpr int kMaxUnits = ZERO_NOALLOC_MAX_UNITS;
constexpr int kThreads = 256;
constexpr int kMaxDevices = 64;

// [0, kNormBlocks): block partials of one unit; then one fp64 sum per unit.
static __device__ __align__(256) double g_noalloc_scratch[kNormBlocks + kMaxUnits];

// Host code must not use g_noalloc_scratch's name as an address: look up its
// device address once per device, with that device current, and keep it for
// the process (a cudaDeviceReset, which rebuilds the context, is not followed;
// the header says so).
std::mutex g_addr_mu;
double* g_addr[kMaxDevices] = {};

int scratch_address(double** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ZERO_ECUDA;
    std::lock_guard<std::mutex> lk(g_addr_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ZERO_ECUDA;
        g_addr[dev] = static_cast<double*>(p);
    }
    *out = g_addr[dev];
    return ZERO_OK;
}

__device__ __forceinline__ double block_sum(double d)
{
    __shared__ double warp_sums[kThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_down_sync(0xFFFFFFFFu, d, off);
    if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = d;
    __syncthreads();
    double total = 0.0;
    if (threadIdx.x == 0)
        for (int w = 0; w < kThreads / 32; ++w) total += warp_sums[w];
    return total; // valid in thread 0
}

// unit_sums[u] = the unit's block partials summed in a fixed order.
__global__ void __launch_bounds__(kThreads)
unit_sum_kernel(const double* __restrict__ partials, double* __restrict__ unit_sums, int u)
{
    double s = 0.0;
    for (int i = threadIdx.x; i < kNormBlocks; i += kThreads) s += partials[i];
    const double total = block_sum(s);
    if (threadIdx.x == 0) unit_sums[u] = total;
}

// The global norm over the units (summed in a fixed order), the clip coefficient, and
// optionally each unit's norm.
__global__ void __launch_bounds__(kThreads)
units_coef_kernel(const double* __restrict__ unit_sums, int n_units, double max_norm,
                  float* __restrict__ norm_coef, float* __restrict__ unit_norms)
{
    double s = 0.0;
    for (int u = threadIdx.x; u < n_units; u += kThreads) {
        s += unit_sums[u];
        if (unit_norms) unit_norms[u] = static_cast<float>(sqrt(unit_sums[u]));
    }
    const double total = block_sum(s);
    if (threadIdx.x == 0) {
        const double norm = sqrt(total);
        double c = max_norm / (norm + 1e-6);
        if (c > 1.0) c = 1.0;
        norm_coef[0] = static_cast<float>(norm);
        norm_coef[1] = static_cast<float>(c);
    }
}

} // namespace
} // namespace zero

using namespace zero;

extern "C" int zero_clip_coef_units_noalloc(const zero_unit_t* units, int32_t n_units,
                                            int32_t n_ranks, const uint16_t* const* grads,
                                            double max_norm, float* norm_coef, float* unit_norms,
                                            cudaStream_t stream)
{
    if (!units || n_units < 1 || n_ranks < 1 || n_ranks > ZERO_MAX_RANKS || !norm_coef ||
        !(max_norm > 0) || !std::isfinite(max_norm))
        return ZERO_EINVAL;
    if (n_units > kMaxUnits) return ZERO_EINVAL; // beyond the static array's capacity
    for (int32_t u = 0; u < n_units; ++u) {
        const zero_unit_t& U = units[u];
        if (U.n_padded <= 0 || U.n_padded % 8 != 0 || U.offset < 0 || U.offset % 8 != 0)
            return ZERO_EINVAL;
    }
    int rc = check_table(grads, n_ranks);
    if (rc != ZERO_OK) return rc;
    if (!aligned16(norm_coef) || (unit_norms && !aligned16(unit_norms))) return ZERO_EALIGN;

    double* scratch = nullptr;
    if ((rc = scratch_address(&scratch)) != ZERO_OK) return rc;
    double* partials = scratch;
    double* unit_sums = scratch + kNormBlocks;
    const uint16_t* unit_grads[ZERO_MAX_RANKS];
    for (int32_t u = 0; u < n_units; ++u) {
        for (int32_t r = 0; r < n_ranks; ++r) unit_grads[r] = grads[r] + units[u].offset;
        rc = grad_sqnorm(n_ranks, units[u].n_padded, unit_grads, 0, partials, kNormScratchBytes,
                         stream);
        if (rc != ZERO_OK) return rc;
        unit_sum_kernel<<<1, kThreads, 0, stream>>>(partials, unit_sums, u);
        if ((rc = cuda_status(cudaGetLastError())) != ZERO_OK) return rc;
    }
    units_coef_kernel<<<1, kThreads, 0, stream>>>(unit_sums, n_units, max_norm, norm_coef,
                                                  unit_norms);
    return cuda_status(cudaGetLastError());
}
