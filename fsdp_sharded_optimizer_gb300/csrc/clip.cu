// clip.cu -- global gradient-norm clipping across the shards: the squared norm
// of the averaged gradient (zero_grad_sqnorm) and the clip coefficient
// (zero_clip_coef).
//
// Method ("Data parallelism, ZeRO and FSDP", "7. Common mistakes", local
// gradient clipping): with sharded gradients the global norm needs an
// all-reduce of the squared shard norms.  The rule is that of the
// clip_grad_norm_ call in the DDP reference of "Distributed Training Basics --
// DDP and FSDP": coef = max_norm / (norm + 1e-6), at most 1.
//
// On one GPU the squared shard norms are per-block partial sums in a scratch
// array the caller provides; the "all-reduce" is one block summing them.  The
// norm pass reads the N_d bf16 gradients once (2 N_d bytes per parameter,
// HBM-bound) and rebuilds each mean gradient exactly as the fused step does.
// The grid is fixed (kNormBlocks), so the partials and their order -- and with
// them the result -- do not depend on the device's occupancy.  Accuracy: each
// thread sums 8 squares pairwise in fp32 and accumulates with Kahan
// compensation; the block and final sums run in fp64.  The relative error of
// the squared norm stays within about 6 fp32 roundings (< 4e-7), whatever the
// length.
//
// zero_grad_reduce_sqnorm is the same pass that also keeps what it computes:
// each element's mean gradient, stored to its owner's fp32 gradient shard
// (the reduce-scatter's output, FSDP's fp32 gradient shard).  The clipped
// update then reads 4 bytes per parameter of that shard instead of the 2N
// bytes of rank gradients: 2N + 34 bytes per parameter for the clipped step
// instead of 4N + 26.
#include "device.cuh"
#include "zero_internal.h"

namespace zero {
namespace {

constexpr int kNormThreads = 256;

struct GradTable {
    const uint4* g[ZERO_MAX_RANKS];
};

__device__ __forceinline__ double block_sum(double d)
{
    __shared__ double warp_sums[kNormThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_down_sync(0xFFFFFFFFu, d, off);
    if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = d;
    __syncthreads();
    double total = 0.0;
    if (threadIdx.x == 0)
        for (int w = 0; w < kNormThreads / 32; ++w) total += warp_sums[w];
    return total; // valid in thread 0
}

struct ReduceTable {
    const uint4* g[ZERO_MAX_RANKS];
    float4* out[ZERO_MAX_RANKS]; // the owners' fp32 gradient shards (kStore only)
};

// One vector's share of the squared norm: g = sum * (1/N) for its 8 elements,
// their squares summed pairwise, the result added to the thread's Kahan sum.
// Every path below calls it once per vector, in the vectors' order.
__device__ __forceinline__ void add_squares(const float (&acc)[8], float inv_n, float (&g)[8],
                                            float& sum, float& comp)
{
    float sq[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        g[e] = __fmul_rn(acc[e], inv_n);
        sq[e] = __fmul_rn(g[e], g[e]);
    }
    const float s8 = __fadd_rn(__fadd_rn(__fadd_rn(sq[0], sq[1]), __fadd_rn(sq[2], sq[3])),
                               __fadd_rn(__fadd_rn(sq[4], sq[5]), __fadd_rn(sq[6], sq[7])));
    const float y = __fsub_rn(s8, comp);
    const float t = __fadd_rn(sum, y);
    comp = __fsub_rn(__fsub_rn(t, sum), y);
    sum = t;
}

// The reduce-scatter's sum of one vector from loads already in registers:
// fp32 from +0 over ranks 0..kN-1 in order, as dev::sum_ranks.
template <int kN>
__device__ __forceinline__ void sum_loaded(const uint4 (&G)[kN], float (&acc)[8])
{
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
    for (int r = 0; r < kN; ++r) {
        acc[0] = __fadd_rn(acc[0], dev::bf16_lo(G[r].x));
        acc[1] = __fadd_rn(acc[1], dev::bf16_hi(G[r].x));
        acc[2] = __fadd_rn(acc[2], dev::bf16_lo(G[r].y));
        acc[3] = __fadd_rn(acc[3], dev::bf16_hi(G[r].y));
        acc[4] = __fadd_rn(acc[4], dev::bf16_lo(G[r].z));
        acc[5] = __fadd_rn(acc[5], dev::bf16_hi(G[r].z));
        acc[6] = __fadd_rn(acc[6], dev::bf16_lo(G[r].w));
        acc[7] = __fadd_rn(acc[7], dev::bf16_hi(G[r].w));
    }
}

// The norm pass.  Each thread takes the vectors q, q + stride, q + 2*stride,
// ... (stride = the fixed grid's threads) and adds their squares in that
// order; the block sums its threads in fp64.
// kStore: also store each element's mean gradient to its owner's fp32 shard
// (zero_grad_reduce_sqnorm); (owner, position) advance with the stride split
// into whole shards (step_k) and a remainder (step_j), as in the fused step.
// kN: the rank count (1, 2 or 4), known at compile time.  Then a loop trip
// issues the loads of kU = 8/kN consecutive vectors of the thread before it
// sums any, so a thread keeps 128 B in flight as at N_d = 8 (with 1 rank and
// one vector a trip it would keep 16 B).  The sums are the same operations in
// the same order as with kN = 0 (any count, one vector a trip): the bits do
// not change.
template <bool kStore, int kN>
__global__ void __launch_bounds__(kNormThreads)
grad_sqnorm_kernel(const __grid_constant__ ReduceTable T, int n_ranks, int64_t n_vec,
                   int64_t shard_vec, int64_t step_k, int64_t step_j, float inv_n, int accumulate,
                   double* __restrict__ partials)
{
    // A ZeRO-3 step's norm passes run one unit after another, each adding to
    // the partials the one before left.  Launched chained, a pass reads and
    // squares its own unit's gradients while the previous pass drains, and
    // waits for that pass to complete only before it adds to the partials.
    // Both instructions do nothing in a launch that is not chained.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float sum = 0.0f, comp = 0.0f; // Kahan: true sum ~ sum - comp
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kNormThreads;
    int64_t q = static_cast<int64_t>(blockIdx.x) * kNormThreads + threadIdx.x;
    int64_t k = 0, j = 0;
    if (kStore) {
        k = q / shard_vec;
        j = q - k * shard_vec;
    }
    auto finish = [&](const float (&acc)[8]) {
        float g[8];
        add_squares(acc, inv_n, g, sum, comp);
        if (kStore) {
            float4* o = T.out[k] + 2 * j;
            dev::st_stream(o, make_float4(g[0], g[1], g[2], g[3]));
            dev::st_stream(o + 1, make_float4(g[4], g[5], g[6], g[7]));
            k += step_k;
            j += step_j;
            if (j >= shard_vec) {
                j -= shard_vec;
                ++k;
            }
        }
    };
    if constexpr (kN == 0) {
        for (; q < n_vec; q += stride) {
            float acc[8];
            dev::sum_ranks<8>(T.g, n_ranks, q, acc);
            finish(acc);
        }
    } else {
        constexpr int kU = 8 / kN;
        for (; q < n_vec; q += kU * stride) {
            uint4 G[kU][kN];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t qu = q + u * stride;
                if (qu < n_vec) {
#pragma unroll
                    for (int r = 0; r < kN; ++r) G[u][r] = dev::ld_stream(T.g[r] + qu);
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (q + u * stride < n_vec) {
                    float acc[8];
                    sum_loaded<kN>(G[u], acc);
                    finish(acc);
                }
            }
        }
    }
    const double b = block_sum(static_cast<double>(sum) - static_cast<double>(comp));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) partials[blockIdx.x] = (accumulate ? partials[blockIdx.x] : 0.0) + b;
}

// The unrolled loop for 1, 2 or 4 ranks on the plain pass only.  Measured on
// GB300 (GPT-2-sized buffer, GB/s, old -> unrolled): N_d = 1 3,177 -> 5,894,
// N_d = 2 5,385 -> 6,675, N_d = 4 6,823 -> 6,945; N_d = 3 lost 3 % and the
// pass that stores the shard lost 6-10 % at every N_d <= 4 (its stores come
// in bursts after the loads), so those keep the one-vector loop.
// chained: launched with programmatic stream serialization (the previous
// kernel on the stream must be a norm pass over other gradients).
template <bool kStore>
cudaError_t launch_norm(const ReduceTable& T, int n_ranks, int64_t n_vec, int64_t shard_vec,
                        int64_t step_k, int64_t step_j, float inv_n, int accumulate,
                        double* partials, cudaStream_t stream, bool chained)
{
    const int kn = kStore ? 0 : (n_ranks == 1 || n_ranks == 2 || n_ranks == 4 ? n_ranks : 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kNormBlocks);
    cfg.blockDim = dim3(kNormThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = chained ? 1 : 0;
    auto go = [&](auto kernel) {
        return cudaLaunchKernelEx(&cfg, kernel, T, n_ranks, n_vec, shard_vec, step_k, step_j,
                                  inv_n, accumulate, partials);
    };
    switch (kn) {
    case 1: return go(grad_sqnorm_kernel<false, 1>);
    case 2: return go(grad_sqnorm_kernel<false, 2>);
    case 4: return go(grad_sqnorm_kernel<false, 4>);
    default: return go(grad_sqnorm_kernel<kStore, 0>);
    }
}

__global__ void __launch_bounds__(kNormThreads)
clip_coef_kernel(const double* __restrict__ partials, int n, double max_norm,
                 float* __restrict__ norm_coef)
{
    double s = 0.0;
    for (int i = threadIdx.x; i < n; i += kNormThreads) s += partials[i];
    const double total = block_sum(s);
    if (threadIdx.x == 0) {
        const double norm = sqrt(total);
        double c = max_norm / (norm + 1e-6);
        if (c > 1.0) c = 1.0;
        norm_coef[0] = static_cast<float>(norm);
        norm_coef[1] = static_cast<float>(c);
    }
}

// y = rank; each warp counts the rank's non-finite bf16 values (all exponent
// bits set) in its vectors and adds its count once.  Integer counts: the
// result does not depend on the order of the additions.
__global__ void __launch_bounds__(kNormThreads)
grad_nonfinite_kernel(const __grid_constant__ GradTable T, int64_t n_vec,
                      unsigned int* __restrict__ counts)
{
    const int r = blockIdx.y;
    unsigned int c = 0;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kNormThreads + threadIdx.x; q < n_vec;
         q += static_cast<int64_t>(gridDim.x) * kNormThreads) {
        const uint4 x = dev::ld_stream(T.g[r] + q);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            c += (w[i] & 0x7F80u) == 0x7F80u;
            c += (w[i] & 0x7F800000u) == 0x7F800000u;
        }
    }
    c = __reduce_add_sync(0xFFFFFFFFu, c);
    if ((threadIdx.x & 31) == 0 && c) atomicAdd(&counts[r], c);
}

} // namespace

int grad_sqnorm(int32_t n_ranks, int64_t n_elems, const uint16_t* const* grads, int32_t accumulate,
                double* scratch, int64_t scratch_bytes, cudaStream_t stream, bool chained)
{
    if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS || n_elems <= 0 || n_elems % 8 != 0 || !scratch ||
        scratch_bytes < kNormScratchBytes)
        return ZERO_EINVAL;
    int rc = check_table(grads, n_ranks);
    if (rc != ZERO_OK) return rc;
    if (!aligned16(scratch)) return ZERO_EALIGN;
    ReduceTable T = {};
    for (int32_t r = 0; r < n_ranks; ++r) T.g[r] = reinterpret_cast<const uint4*>(grads[r]);
    const float inv_n = static_cast<float>(1.0 / static_cast<double>(n_ranks));
    return cuda_status(launch_norm<false>(T, n_ranks, n_elems / 8, 1, 0, 0, inv_n,
                                          accumulate ? 1 : 0, scratch, stream, chained));
}

int grad_reduce_sqnorm(int32_t n_ranks, int64_t n_elems, const uint16_t* const* grads,
                       float* const* grad_shard, int32_t accumulate, double* scratch,
                       int64_t scratch_bytes, cudaStream_t stream, bool chained)
{
    if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS || n_elems <= 0 ||
        n_elems % (8 * static_cast<int64_t>(n_ranks)) != 0 || !scratch ||
        scratch_bytes < kNormScratchBytes)
        return ZERO_EINVAL;
    int rc = check_table(grads, n_ranks);
    if (rc != ZERO_OK) return rc;
    if ((rc = check_table(grad_shard, n_ranks)) != ZERO_OK) return rc;
    if (!aligned16(scratch)) return ZERO_EALIGN;
    ReduceTable T = {};
    for (int32_t r = 0; r < n_ranks; ++r) {
        T.g[r] = reinterpret_cast<const uint4*>(grads[r]);
        T.out[r] = reinterpret_cast<float4*>(grad_shard[r]);
    }
    const int64_t shard_vec = n_elems / n_ranks / 8;
    const StrideSplit sp = split_stride(static_cast<int64_t>(kNormBlocks) * kNormThreads, shard_vec);
    const float inv_n = static_cast<float>(1.0 / static_cast<double>(n_ranks));
    return cuda_status(launch_norm<true>(T, n_ranks, n_elems / 8, shard_vec, sp.k, sp.j, inv_n,
                                         accumulate ? 1 : 0, scratch, stream, chained));
}

int clip_coef(const double* scratch, int64_t scratch_bytes, double max_norm, float* norm_coef,
              cudaStream_t stream)
{
    if (!scratch || scratch_bytes < kNormScratchBytes || !norm_coef || !(max_norm > 0) ||
        !std::isfinite(max_norm))
        return ZERO_EINVAL;
    if (!aligned16(scratch) || !aligned16(norm_coef)) return ZERO_EALIGN;
    clip_coef_kernel<<<1, kNormThreads, 0, stream>>>(scratch, kNormBlocks, max_norm, norm_coef);
    return cuda_status(cudaGetLastError());
}

int preload_clip_kernels()
{
    cudaFuncAttributes a;
    const void* kernels[] = {
        reinterpret_cast<const void*>(grad_sqnorm_kernel<false, 0>),
        reinterpret_cast<const void*>(grad_sqnorm_kernel<false, 1>),
        reinterpret_cast<const void*>(grad_sqnorm_kernel<false, 2>),
        reinterpret_cast<const void*>(grad_sqnorm_kernel<false, 4>),
        reinterpret_cast<const void*>(grad_sqnorm_kernel<true, 0>),
        reinterpret_cast<const void*>(clip_coef_kernel),
    };
    for (const void* k : kernels)
        if (cudaFuncGetAttributes(&a, k) != cudaSuccess) return ZERO_ECUDA;
    return ZERO_OK;
}

} // namespace zero

using namespace zero;

extern "C" int64_t zero_clip_scratch_bytes(void) { return kNormScratchBytes; }

extern "C" int zero_grad_sqnorm(int32_t n_ranks, int64_t n_elems, const uint16_t* const* grads,
                                int32_t accumulate, double* scratch, int64_t scratch_bytes,
                                cudaStream_t stream)
{
    return grad_sqnorm(n_ranks, n_elems, grads, accumulate, scratch, scratch_bytes, stream);
}

extern "C" int zero_grad_reduce_sqnorm(int32_t n_ranks, int64_t n_elems,
                                       const uint16_t* const* grads, float* const* grad_shard,
                                       int32_t accumulate, double* scratch, int64_t scratch_bytes,
                                       cudaStream_t stream)
{
    return grad_reduce_sqnorm(n_ranks, n_elems, grads, grad_shard, accumulate, scratch,
                              scratch_bytes, stream);
}

extern "C" int zero_clip_coef(const double* scratch, int64_t scratch_bytes, double max_norm,
                              float* norm_coef, cudaStream_t stream)
{
    return clip_coef(scratch, scratch_bytes, max_norm, norm_coef, stream);
}

extern "C" int zero_grad_nonfinite(int32_t n_ranks, int64_t n_elems, const uint16_t* const* grads,
                                   uint32_t* counts, int32_t reset, cudaStream_t stream)
{
    if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS || n_elems <= 0 || n_elems % 8 != 0 || !counts)
        return ZERO_EINVAL;
    int rc = check_table(grads, n_ranks);
    if (rc != ZERO_OK) return rc;
    if (!aligned16(counts)) return ZERO_EALIGN;
    if (reset && (rc = cuda_status(cudaMemsetAsync(counts, 0, sizeof(uint32_t) * n_ranks,
                                                   stream))) != ZERO_OK)
        return rc;
    GradTable T = {};
    for (int32_t r = 0; r < n_ranks; ++r) T.g[r] = reinterpret_cast<const uint4*>(grads[r]);
    const int64_t n_vec = n_elems / 8;
    int64_t gx = (kNormBlocks + n_ranks - 1) / n_ranks;
    const int64_t need = (n_vec + kNormThreads - 1) / kNormThreads;
    if (gx > need) gx = need;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(n_ranks));
    grad_nonfinite_kernel<<<grid, kNormThreads, 0, stream>>>(T, n_vec,
                                                             reinterpret_cast<unsigned int*>(counts));
    return cuda_status(cudaGetLastError());
}
