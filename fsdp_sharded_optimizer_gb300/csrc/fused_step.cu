// fused_step.cu -- the fused reduce-scatter + AdamW + bf16 all-gather kernel
// and its two entry points, zero_step_stage12 and zero3_reduce_scatter_unit.
//
// Method ("Data parallelism, ZeRO and FSDP", lesson 8): "The communication is
// already there" puts the optimizer step between the two halves of the
// all-reduce; the Theorem's proof steps 2, 3 and 6 (ZeRO-1/2) and 7 (ZeRO-3);
// the AdamW update of "5. In code", first block.
//
// One pass over HBM per element: read the N_d bf16 gradients and the owner's
// fp32 master/m/v, write master/m/v and one bf16 weight -- 26 + 2*N_d bytes
// per parameter.  The reduce-scatter is the owner's in-register fp32 sum in
// rank order; the all-gather is the bf16 store.  The path is bound by HBM
// bandwidth (about 0.5 flop per byte), so the kernel is a persistent
// grid-stride stream of 16-byte vector accesses: each thread handles 8
// consecutive elements (one 16-byte bf16 vector per rank, two 16-byte fp32
// vectors per state array) and keeps all of a batch's loads in flight before
// it sums.  A call is issued as chained launches over 25 MiB chunks (see
// launch()).  The update from an already reduced fp32 gradient shard has its
// own kernel with 32-byte accesses (fused_step_wide_kernel).  No tensor
// cores: this is not a contraction.
#include <new>
#include <vector>

#include "device.cuh"
#include "zero_internal.h"

namespace zero {
namespace {

constexpr int kBlock = 256;
constexpr int kRankBatch = 8; // gradient loads issued together before summing (three-block shape)
// Two launch shapes.  The three-block one: three resident blocks per SM (an
// 80-register cap) instead of the two that the unconstrained 94-102 registers
// allow, with 8-rank load batches (+12 % at N_d = 8 over two blocks per SM on
// one unchunked launch).  It now serves only the update from the fp32
// gradient shard (fused_step_wide_kernel and its 16-byte fallback), which
// reads no rank gradients.
constexpr int kMinBlocksPerSM = 3;
// The four-block one: four resident blocks per SM (a 64-register cap) and
// loads in batches of 4 ranks.  It first won up to 4 ranks, where a thread
// has few gradient vectors to hold and the bytes in flight per thread fall
// (112 B at N_d = 1 against 224 B at 8; GB300, GPT-2 buffer: N_d = 1 5,719 ->
// 6,478 GB/s, N_d = 2 5,876 -> 6,507, N_d = 4 6,260 -> 6,477), and on chained
// chunks it also wins at N_d = 8 (0.748 -> 0.745 ms a step).  Since the
// kernel loads the gradients before the state (no register spill), every
// kernel that reads rank gradients -- the plain, clipped and accumulated
// steps, the fp32-gradient step and the accumulation of micro-batches
// 1..m-1 -- takes it at every rank count.
constexpr int kMinBlocksPerSMSmall = 4;
constexpr int kRankBatchSmall = 4;

// Per-rank device pointers, passed by value in the kernel's parameter space
// (5 x 64 x 8 B = 2.5 KB).  o[k] points at rank k's output slice: the
// replicated buffer at k*S for ZeRO-1/2, the rank's shard for ZeRO-3.
struct Tables {
    const uint4* g[ZERO_MAX_RANKS];
    float4* w[ZERO_MAX_RANKS];
    float4* m[ZERO_MAX_RANKS];
    float4* v[ZERO_MAX_RANKS];
    uint4* o[ZERO_MAX_RANKS];
    float4* a[ZERO_MAX_RANKS]; // ZeRO-2 accumulation: rank k's fp32 gradient accumulator
};

// The vectors [q0, q1) this launch covers (a vector = 8 elements), the shard
// length in vectors, and the grid stride split into whole shards + remainder.
struct Range {
    int64_t q0, q1;
    int64_t shard_vec;
    int64_t step_k, step_j;
    int32_t n_ranks;
    float inv_m; // ZeRO-2 accumulation: 1/micro-batches
    // kCheck: device uint32[2]; bit r is set when rank r's gradient holds an
    // infinity or a NaN
    uint32_t* nonfinite;
};

__device__ __forceinline__ void adamw(float g, float& w, float& m, float& v,
                                      const StepScalars& s)
{
    // The page's operand order; each operation is one rounded fp32 op.
    const float m1 = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
    const float v1 = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(__fmul_rn(s.omb2, g), g));
    // With m1 = v1 = 0 (a zero gradient on a zero state: padding, parameters
    // that have not had a gradient yet) each quotient below is m1 itself:
    // 0 / bc1, 0 / bc2 and 0 / (sqrt(0) + eps) are zeros of m1's sign, as
    // bc1, bc2 and eps are finite and positive.  Skipping them keeps the bits
    // and avoids the IEEE division's slow path for zero operands (GB300,
    // GPT-2 buffer, N_d = 8: all-zero gradients 0.989 -> 0.752 ms, half of
    // them zero 0.864 -> 0.749; random gradients 0.7420 -> 0.7444).
    float q = m1;
    if (m1 != 0.0f || v1 != 0.0f) {
        const float mh = __fdiv_rn(m1, s.bc1);
        const float vh = __fdiv_rn(v1, s.bc2);
        q = __fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), s.eps));
    }
    const float upd = __fadd_rn(q, __fmul_rn(s.wd, w));
    w = __fsub_rn(w, __fmul_rn(s.lr, upd));
    m = m1;
    v = v1;
}

// The clip coefficient clip[1], read in each loop trip where it is used (an
// L1 hit) instead of being held in a register across the loop.  It was
// written by an earlier kernel on the stream, so the read-only path is safe.
__device__ __forceinline__ float ld_coef(const float* clip)
{
    float c;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(c) : "l"(clip + 1));
    return c;
}

// kClip: the mean gradient is multiplied by clip[1], the coefficient of the
// global-norm clipping computed on the device by zero_clip_coef.
// kAcc: the last micro-batch of ZeRO-2 gradient accumulation; the gradient is
// (a[k] + this micro-batch's mean) * (1/m), a[k] holding the earlier ones.
// kF32: the rank gradients are fp32 (T.g holds float4 pointers).
// kG32: the mean gradient is already reduced: read g from the owner's fp32
// gradient shard T.a[k] (written by zero_grad_reduce_sqnorm) instead of the
// N rank gradients.  Used when a pointer is only 16-byte aligned;
// fused_step_wide_kernel does the same with 32-byte accesses otherwise.
// kSmall: the four-block launch shape (every step that reads rank gradients);
// without it the three-block shape of the 16-byte update from the gradient
// shard.
// kCheck: the pre-reduction finite check of each rank's bf16 gradient, on the
// values the reduction loads anyway: bit r of R.nonfinite is set when rank r
// contributed an infinity or a NaN.  The results are unchanged.
template <bool kClip, bool kAcc, bool kF32 = false, bool kG32 = false, bool kSmall = false,
          bool kCheck = false>
__global__ void __launch_bounds__(kBlock, kSmall ? kMinBlocksPerSMSmall : kMinBlocksPerSM)
fused_step_kernel(const __grid_constant__ Tables T, const StepScalars s, const Range R,
                  const float* __restrict__ clip)
{
    static_assert(!(kAcc && (kF32 || kG32)), "accumulation reads bf16 rank gradients");
    static_assert(!(kCheck && (kF32 || kG32)), "the finite check reads bf16 rank gradients");
    // Chained launches (programmatic dependent launch): the next chunk's grid
    // may start as soon as every block of this one is running, so its blocks
    // fill the SMs this grid's tail leaves idle.  Chunks touch disjoint
    // elements; the wait at the end keeps "this grid completes after its
    // predecessor" for everything later on the stream.  Threads without work
    // leave at once; thread 0 of block 0 always has work (q0 < q1) and waits,
    // which is enough to hold the grid's completion.  Both instructions do
    // nothing for a launch without the attribute.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
    int64_t q = R.q0 + static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (q >= R.q1) return;
    int64_t k = q / R.shard_vec;     // owner
    int64_t j = q - k * R.shard_vec; // vector position inside the owner's shard
    const int N = R.n_ranks;
    uint64_t bad = 0; // kCheck: ranks seen with a non-finite gradient

    for (; q < R.q1; q += stride) {
        // The gradient of the 8 elements is loaded, summed and scaled before
        // the owner's state is loaded, so the 24 state values are not live
        // while a rank batch is in flight.  Loading the state first needed
        // more than the 64 registers of the four-block shape (16-32 B of
        // spill a thread); this order spills nothing in any variant and is
        // faster throughout (GB300, GPT-2 buffer, same data, ms a step: N_d = 8
        // 0.7800 -> 0.7558, N_d = 1 0.531 -> 0.518, N_d = 64 2.846 -> 2.785;
        // last micro-batch of an accumulation at N_d = 8 0.851 -> 0.806; fp32
        // rank gradients at N_d = 8 1.070 -> 1.025).  The results are the same
        // operations on the same values.
        //
        // reduce-scatter: fp32 sum from +0 over ranks 0..N-1, in order
        float acc[8];
        if (kG32) {
            const float4 g0 = dev::ld_stream(T.a[k] + 2 * j), g1 = dev::ld_stream(T.a[k] + 2 * j + 1);
            acc[0] = g0.x; acc[1] = g0.y; acc[2] = g0.z; acc[3] = g0.w;
            acc[4] = g1.x; acc[5] = g1.y; acc[6] = g1.z; acc[7] = g1.w;
        } else if (kF32)
            dev::sum_ranks_f32<kSmall ? kRankBatchSmall / 2 : kRankBatch / 2>(
                reinterpret_cast<const float4* const*>(T.g), N, q, acc);
        else
            dev::sum_ranks<kSmall ? kRankBatchSmall : kRankBatch, kCheck>(T.g, N, q, acc, &bad);
        // g = mean (the shard already holds it), then for the last micro-batch
        // (earlier micro-batches + this mean) / m, then times the clip coefficient
        if (kAcc) {
            const float4 a0 = dev::ld_stream(T.a[k] + 2 * j), a1 = dev::ld_stream(T.a[k] + 2 * j + 1);
            const float prior[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[e] = __fmul_rn(__fadd_rn(prior[e], __fmul_rn(acc[e], s.inv_n)), R.inv_m);
        } else if (!kG32) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = __fmul_rn(acc[e], s.inv_n);
        }
        if (kClip) {
            const float coef = ld_coef(clip);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = __fmul_rn(acc[e], coef);
        }

        // AdamW on the owner's fp32 state
        float4* wp = T.w[k] + 2 * j;
        float4* mp = T.m[k] + 2 * j;
        float4* vp = T.v[k] + 2 * j;
        const float4 w0 = dev::ld_stream(wp), w1 = dev::ld_stream(wp + 1);
        const float4 m0 = dev::ld_stream(mp), m1 = dev::ld_stream(mp + 1);
        const float4 v0 = dev::ld_stream(vp), v1 = dev::ld_stream(vp + 1);
        float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) adamw(acc[e], w[e], m[e], v[e], s);

        dev::st_stream(wp, make_float4(w[0], w[1], w[2], w[3]));
        dev::st_stream(wp + 1, make_float4(w[4], w[5], w[6], w[7]));
        dev::st_stream(mp, make_float4(m[0], m[1], m[2], m[3]));
        dev::st_stream(mp + 1, make_float4(m[4], m[5], m[6], m[7]));
        dev::st_stream(vp, make_float4(v[0], v[1], v[2], v[3]));
        dev::st_stream(vp + 1, make_float4(v[4], v[5], v[6], v[7]));
        // all-gather: the owner's new bf16 slice
        dev::st_stream(T.o[k] + j,
                       make_uint4(dev::pack_bf16x2(w[0], w[1]), dev::pack_bf16x2(w[2], w[3]),
                                  dev::pack_bf16x2(w[4], w[5]), dev::pack_bf16x2(w[6], w[7])));

        k += R.step_k;
        j += R.step_j;
        if (j >= R.shard_vec) {
            j -= R.shard_vec;
            ++k;
        }
    }
    if (kCheck && bad != 0) { // rare: only threads that met a non-finite value
        if (static_cast<uint32_t>(bad) != 0) atomicOr(R.nonfinite, static_cast<uint32_t>(bad));
        if ((bad >> 32) != 0) atomicOr(R.nonfinite + 1, static_cast<uint32_t>(bad >> 32));
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The update from the reduced fp32 gradient shard (what kG32 selects in
// fused_step_kernel) with 32-byte accesses: each thread's 8 fp32 values of g,
// master, m and v move in one 256-bit load or store instead of two 16-byte
// ones; the arithmetic is fused_step_kernel's, element for element.
// Measured on GB300 (GPT-2 buffer, 16 B read + 14 B written per parameter):
// 6,364 -> 6,658 GB/s.  The same change slowed the bf16-gradient step (6,974
// -> 6,747), the ZeRO-2 accumulation and the norm pass's shard store, which
// keep their 16-byte accesses.  Every fp32 table entry must be 32-byte
// aligned; launch_range falls back to fused_step_kernel otherwise.
template <bool kClip>
__global__ void __launch_bounds__(kBlock, kMinBlocksPerSM)
fused_step_wide_kernel(const __grid_constant__ Tables T, const StepScalars s, const Range R,
                       const float* __restrict__ clip)
{
    // chained like fused_step_kernel (the same two instructions, the same reasons)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
    int64_t q = R.q0 + static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (q >= R.q1) return;
    int64_t k = q / R.shard_vec;
    int64_t j = q - k * R.shard_vec;
    const float coef = kClip ? clip[1] : 1.0f;

    for (; q < R.q1; q += stride) {
        float4* wp = T.w[k] + 2 * j;
        float4* mp = T.m[k] + 2 * j;
        float4* vp = T.v[k] + 2 * j;
        float w[8], m[8], v[8], g[8];
        dev::ld8_stream(wp, w);
        dev::ld8_stream(mp, m);
        dev::ld8_stream(vp, v);
        dev::ld8_stream(T.a[k] + 2 * j, g);
#pragma unroll
        for (int e = 0; e < 8; ++e) adamw(kClip ? __fmul_rn(g[e], coef) : g[e], w[e], m[e], v[e], s);
        dev::st8_stream(wp, w);
        dev::st8_stream(mp, m);
        dev::st8_stream(vp, v);
        dev::st_stream(T.o[k] + j,
                       make_uint4(dev::pack_bf16x2(w[0], w[1]), dev::pack_bf16x2(w[2], w[3]),
                                  dev::pack_bf16x2(w[4], w[5]), dev::pack_bf16x2(w[6], w[7])));
        k += R.step_k;
        j += R.step_j;
        if (j >= R.shard_vec) {
            j -= R.shard_vec;
            ++k;
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ZeRO-2 accumulation of micro-batches 1..m-1: a[k] = (first ? +0 : a[k]) + mean,
// in the fused step's four-block launch shape.
template <bool kFirst>
__global__ void __launch_bounds__(kBlock, kMinBlocksPerSMSmall)
accumulate_kernel(const __grid_constant__ Tables T, const float inv_n, const Range R)
{
    // chained like fused_step_kernel (the same two instructions, the same reasons)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
    int64_t q = R.q0 + static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    if (q >= R.q1) return;
    int64_t k = q / R.shard_vec;
    int64_t j = q - k * R.shard_vec;
    for (; q < R.q1; q += stride) {
        float acc[8];
        dev::sum_ranks<kRankBatchSmall>(T.g, R.n_ranks, q, acc);
        float4* ap = T.a[k] + 2 * j;
        float prior[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (!kFirst) {
            const float4 a0 = dev::ld_stream(ap), a1 = dev::ld_stream(ap + 1);
            prior[0] = a0.x; prior[1] = a0.y; prior[2] = a0.z; prior[3] = a0.w;
            prior[4] = a1.x; prior[5] = a1.y; prior[6] = a1.z; prior[7] = a1.w;
        }
        float out[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = __fadd_rn(prior[e], __fmul_rn(acc[e], inv_n));
        dev::st_stream(ap, make_float4(out[0], out[1], out[2], out[3]));
        dev::st_stream(ap + 1, make_float4(out[4], out[5], out[6], out[7]));
        k += R.step_k;
        j += R.step_j;
        if (j >= R.shard_vec) {
            j -= R.shard_vec;
            ++k;
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

Range make_range(const void* kernel, int64_t q0, int64_t q1, int64_t shard_vec, int32_t n_ranks,
                 int* blocks_out)
{
    const int max_blocks = persistent_blocks(kernel, kBlock, 0);
    const int64_t need = (q1 - q0 + kBlock - 1) / kBlock;
    const int blocks = max_blocks <= 0 ? 0 : static_cast<int>(need < max_blocks ? need : max_blocks);
    const int64_t stride = static_cast<int64_t>(blocks > 0 ? blocks : 1) * kBlock;
    const StrideSplit sp = split_stride(stride, shard_vec);
    *blocks_out = blocks;
    return Range{q0, q1, shard_vec, sp.k, sp.j, n_ranks, 1.0f};
}

constexpr int64_t kChunkVec = ZERO_CHUNK_ELEMS / 8;

} // namespace

int64_t chunk_count(int64_t n_vec) { return n_vec <= 0 ? 0 : (n_vec + kChunkVec - 1) / kChunkVec; }

namespace {

// A fused-step launch recorded while a CUDA-graph capture is running: the
// kernel node it added and a copy of its arguments.
struct LoggedLaunch {
    cudaGraphNode_t node;
    const void* func;
    unsigned blocks;
    Tables T;
    StepScalars s;
    Range R;
    const float* clip;
};

} // namespace

// The fused-step launches of one capture (zero3_graph_create), in issue order.
struct StepNodeList {
    std::vector<LoggedLaunch> launches;
    bool failed = false;
};

namespace {

thread_local StepNodeList* t_capture_log = nullptr;

// While a capture log is installed on this thread, a fused-step launch asks
// the capture which node it just added (the stream's only dependency right
// after a kernel launch) and keeps it with the arguments, so the graph's step
// scalars can be rewritten before each replay.
void log_capture(const void* func, int blocks, const Tables& T, const StepScalars& s,
                 const Range& R, const float* clip, cudaStream_t stream)
{
    StepNodeList* log = t_capture_log;
    if (!log) return;
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    const cudaGraphNode_t* deps = nullptr;
    const cudaGraphEdgeData* edges = nullptr; // asked for, so that non-default edges are no error
    size_t n_deps = 0;
    if (cudaStreamGetCaptureInfo(stream, &st, nullptr, nullptr, &deps, &edges, &n_deps) !=
            cudaSuccess ||
        st != cudaStreamCaptureStatusActive || n_deps != 1) {
        log->failed = true;
        return;
    }
    try {
        log->launches.push_back(
            LoggedLaunch{deps[0], func, static_cast<unsigned>(blocks), T, s, R, clip});
    } catch (...) {
        log->failed = true;
    }
}

// One fused-step launch.  chained: launched with programmatic stream
// serialization, so it may begin while the previous kernel on the stream (the
// previous chunk or bucket of the same call, which touches other elements)
// finishes.
template <bool kClip, bool kAcc, bool kF32, bool kG32 = false, bool kSmall = false,
          bool kCheck = false>
cudaError_t launch_fused(int blocks, cudaStream_t stream, bool chained, const Tables& T,
                         const StepScalars& s, const Range& R, const float* clip)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = chained ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, fused_step_kernel<kClip, kAcc, kF32, kG32, kSmall, kCheck>, T, s, R, clip);
    if (e == cudaSuccess)
        log_capture(reinterpret_cast<const void*>(
                        fused_step_kernel<kClip, kAcc, kF32, kG32, kSmall, kCheck>),
                    blocks, T, s, R, clip, stream);
    return e;
}

// One launch of fused_step_wide_kernel<kClip> (same arguments, same logging).
template <bool kClip>
cudaError_t launch_wide(int blocks, cudaStream_t stream, bool chained, const Tables& T,
                        const StepScalars& s, const Range& R, const float* clip)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = chained ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, fused_step_wide_kernel<kClip>, T, s, R, clip);
    if (e == cudaSuccess)
        log_capture(reinterpret_cast<const void*>(fused_step_wide_kernel<kClip>), blocks, T, s, R,
                    clip, stream);
    return e;
}

// Whether every fp32 pointer the update from the gradient shard touches (the
// first n entries of w, m, v and a) is 32-byte aligned.
bool wide_aligned(const Tables& T, int32_t n)
{
    uintptr_t bits = 0;
    for (int32_t r = 0; r < n; ++r)
        bits |= reinterpret_cast<uintptr_t>(T.w[r]) | reinterpret_cast<uintptr_t>(T.m[r]) |
                reinterpret_cast<uintptr_t>(T.v[r]) | reinterpret_cast<uintptr_t>(T.a[r]);
    return (bits & 31u) == 0;
}

// One launch of a bf16-gradient variant (plain, clipped, last micro-batch of an
// accumulation, plain with the finite check), in the four-block shape.
int launch_bf16(const Tables& T, const StepScalars& s, int64_t q0, int64_t q1, int64_t shard_vec,
                int32_t n_ranks, const float* clip, cudaStream_t stream, float inv_m, bool chained,
                uint32_t* nonfinite)
{
    const bool acc = inv_m != 0.0f;
    if (nonfinite) { // the plain step with the finite check
        if (clip || acc) return ZERO_EINVAL;
        const void* k =
            reinterpret_cast<const void*>(fused_step_kernel<false, false, false, false, true, true>);
        int blocks = 0;
        Range R = make_range(k, q0, q1, shard_vec, n_ranks, &blocks);
        if (blocks <= 0) return ZERO_ECUDA;
        R.nonfinite = nonfinite;
        return cuda_status(launch_fused<false, false, false, false, true, true>(
            blocks, stream, chained, T, s, R, nullptr));
    }
    const void* kernel =
        clip ? (acc ? reinterpret_cast<const void*>(fused_step_kernel<true, true, false, false, true>)
                    : reinterpret_cast<const void*>(fused_step_kernel<true, false, false, false, true>))
             : (acc ? reinterpret_cast<const void*>(fused_step_kernel<false, true, false, false, true>)
                    : reinterpret_cast<const void*>(fused_step_kernel<false, false, false, false, true>));
    int blocks = 0;
    Range R = make_range(kernel, q0, q1, shard_vec, n_ranks, &blocks);
    if (blocks <= 0) return ZERO_ECUDA;
    R.inv_m = acc ? inv_m : 1.0f;
    cudaError_t e;
    if (clip && acc)
        e = launch_fused<true, true, false, false, true>(blocks, stream, chained, T, s, R, clip);
    else if (clip)
        e = launch_fused<true, false, false, false, true>(blocks, stream, chained, T, s, R, clip);
    else if (acc)
        e = launch_fused<false, true, false, false, true>(blocks, stream, chained, T, s, R, nullptr);
    else
        e = launch_fused<false, false, false, false, true>(blocks, stream, chained, T, s, R, nullptr);
    return cuda_status(e);
}

// One launch over the vectors [q0, q1).
int launch_range(const Tables& T, const StepScalars& s, int64_t q0, int64_t q1, int64_t shard_vec,
                 int32_t n_ranks, const float* clip, cudaStream_t stream, float inv_m, bool f32,
                 bool chained, bool g32, uint32_t* nonfinite)
{
    if (nonfinite && (f32 || g32)) return ZERO_EINVAL; // the check reads bf16 rank gradients
    if (g32 && wide_aligned(T, n_ranks)) { // the reduced fp32 gradient shard, 32-byte accesses
        const void* k = clip ? reinterpret_cast<const void*>(fused_step_wide_kernel<true>)
                             : reinterpret_cast<const void*>(fused_step_wide_kernel<false>);
        int blocks = 0;
        const Range R = make_range(k, q0, q1, shard_vec, n_ranks, &blocks);
        if (blocks <= 0) return ZERO_ECUDA;
        return cuda_status(clip ? launch_wide<true>(blocks, stream, chained, T, s, R, clip)
                                : launch_wide<false>(blocks, stream, chained, T, s, R, nullptr));
    }
    if (g32) { // the same with 16-byte accesses (a pointer only 16-byte aligned)
        const void* k = clip ? reinterpret_cast<const void*>(fused_step_kernel<true, false, false, true>)
                             : reinterpret_cast<const void*>(fused_step_kernel<false, false, false, true>);
        int blocks = 0;
        const Range R = make_range(k, q0, q1, shard_vec, n_ranks, &blocks);
        if (blocks <= 0) return ZERO_ECUDA;
        return cuda_status(clip ? launch_fused<true, false, false, true>(blocks, stream, chained, T,
                                                                         s, R, clip)
                                : launch_fused<false, false, false, true>(blocks, stream, chained,
                                                                          T, s, R, nullptr));
    }
    if (f32) { // fp32 gradients: no clipping or accumulation variant
        // The four-block shape at every rank count: with 32 B of gradient per
        // rank and vector, more threads with 2-rank batches win throughout
        // (GB300, GPT-2 buffer, GB/s: N_d = 8 6,860 -> 6,907, 16 6,867 ->
        // 6,905, 32 6,887 -> 7,035, 64 6,887 -> 7,090; up to 4 it already was).
        const void* k = reinterpret_cast<const void*>(fused_step_kernel<false, false, true, false, true>);
        int blocks = 0;
        const Range R = make_range(k, q0, q1, shard_vec, n_ranks, &blocks);
        if (blocks <= 0) return ZERO_ECUDA;
        return cuda_status(launch_fused<false, false, true, false, true>(blocks, stream, chained, T,
                                                                         s, R, nullptr));
    }
    // The plain, clipped and accumulated steps: the four-block shape at every
    // rank count.  Measured on GB300, GPT-2 buffer, random gradients, ms: the
    // plain step at N_d = 8 0.7482 -> 0.7403 and 0.7767 -> 0.7750 on two
    // boxes, N_d = 12 0.9366 -> 0.9243, N_d = 16 1.0676 -> 1.0740; the last
    // micro-batch of an accumulation, once it no longer spilled, N_d = 5
    // 0.7272 -> 0.7036, 8 0.8053 -> 0.8016, 12 0.9548 -> 0.9290, 16 1.0795 ->
    // 1.0694, 24 1.3547 -> 1.3485.  Elements whose gradient, m and v are all
    // zero take a slower path through the IEEE division, which more resident
    // warps hide better: all-zero gradients 1.098 -> 0.989 ms, half of them
    // zero 0.921 -> 0.864.
    return launch_bf16(T, s, q0, q1, shard_vec, n_ranks, clip, stream, inv_m, chained, nonfinite);
}

// The fused step over the vectors [q0, q1), issued as chunk_count() chained
// launches: consecutive chunks of kChunkVec vectors, the last one shorter.
// One persistent launch over a long range gives every block the same share of
// it, so the step ends when the slowest SM's share does; with chained chunks a
// block that finishes early hands its SM to the next chunk's blocks.  Chunk
// starts stay on kChunkVec boundaries from q0 (25 MiB of bf16 per rank): an
// equal split at odd vector offsets made every warp's loads straddle one more
// cache line and cost 0.8 %.  Measured on GB300, GPT-2 flat buffer at
// N_d = 8: one launch 0.765 ms; chunks of 100 MiB of gradient 0.755 ms,
// 25 MiB 0.748-0.750 ms; 12.5 MiB and below lose again.  The chunks touch
// disjoint elements, and every element is computed exactly as in one launch.
// The first chunk is chained only if the caller asks (a later bucket of the
// same step).
int launch(const Tables& T, const StepScalars& s, int64_t q0, int64_t q1, int64_t shard_vec,
           int32_t n_ranks, const float* clip, cudaStream_t stream, float inv_m = 0.0f,
           bool f32 = false, bool chained = false, bool g32 = false, uint32_t* nonfinite = nullptr)
{
    for (int64_t a = q0; a < q1; a += kChunkVec) {
        const int64_t b = q1 - a > kChunkVec ? a + kChunkVec : q1;
        const int rc = launch_range(T, s, a, b, shard_vec, n_ranks, clip, stream, inv_m, f32,
                                    chained || a > q0, g32, nonfinite);
        if (rc != ZERO_OK) return rc;
    }
    return ZERO_OK;
}

int check_state_tables(int32_t n, const uint16_t* const* grads, float* const* master,
                       float* const* m, float* const* v)
{
    int rc;
    if ((rc = check_table(grads, n)) != ZERO_OK) return rc;
    if ((rc = check_table(master, n)) != ZERO_OK) return rc;
    if ((rc = check_table(m, n)) != ZERO_OK) return rc;
    return check_table(v, n);
}

// The two entry points with an optional device clip coefficient (nullptr = none).
int step_stage12(int32_t stage, int32_t n_ranks, int64_t n_padded, const void* const* grads,
                 float* const* master, float* const* m, float* const* v, uint16_t* params_bf16,
                 const zero_hparams_t* hp, int64_t bucket_elems, const float* clip,
                 cudaStream_t stream, bool f32 = false, bool g32 = false,
                 uint32_t* nonfinite = nullptr)
{
    // g32: `grads` holds the n_ranks fp32 gradient shards (S each) of the
    // reduced mean gradient instead of the rank gradients.
    if ((stage != 1 && stage != 2) || n_ranks < 1 || n_ranks > ZERO_MAX_RANKS ||
        n_padded <= 0 || n_padded % (8 * static_cast<int64_t>(n_ranks)) != 0 ||
        bucket_elems < 0 || bucket_elems % 8 != 0 || !valid_hparams(hp) || !params_bf16)
        return ZERO_EINVAL;
    int rc = check_state_tables(n_ranks, reinterpret_cast<const uint16_t* const*>(grads), master, m, v);
    if (rc != ZERO_OK) return rc;
    if (!aligned16(params_bf16)) return ZERO_EALIGN;

    const int64_t S = n_padded / n_ranks;
    Tables T = {};
    for (int32_t r = 0; r < n_ranks; ++r) {
        if (g32)
            T.a[r] = reinterpret_cast<float4*>(const_cast<void*>(grads[r]));
        else
            T.g[r] = reinterpret_cast<const uint4*>(grads[r]);
        T.w[r] = reinterpret_cast<float4*>(master[r]);
        T.m[r] = reinterpret_cast<float4*>(m[r]);
        T.v[r] = reinterpret_cast<float4*>(v[r]);
        T.o[r] = reinterpret_cast<uint4*>(params_bf16 + r * S);
    }
    const StepScalars s = make_scalars(hp, n_ranks);
    const int64_t nvec = n_padded / 8, shard_vec = S / 8;
    // ZeRO-2 reduces the gradient bucket by bucket as it becomes ready; the
    // per-element arithmetic is the same, so stage 1 and 2 give equal bits.
    const int64_t bucket_vec = (stage == 2 && bucket_elems > 0) ? bucket_elems / 8 : nvec;
    // Buckets after the first are chained to the one before (disjoint elements).
    for (int64_t q0 = 0; q0 < nvec; q0 += bucket_vec) {
        const int64_t q1 = q0 + bucket_vec < nvec ? q0 + bucket_vec : nvec;
        if ((rc = launch(T, s, q0, q1, shard_vec, n_ranks, clip, stream, 0.0f, f32, q0 > 0,
                         g32, nonfinite)) != ZERO_OK)
            return rc;
    }
    return ZERO_OK;
}

// g32: unit_grads holds each rank's fp32 gradient-shard storage of all units
// (laid out like master; this unit at shard_offset) instead of the unit's
// rank gradients.
// A unit layout a ZeRO-3 call can use with n_ranks ranks.
bool unit_valid(const zero_unit_t* unit, int32_t n_ranks)
{
    return unit && n_ranks >= 1 && n_ranks <= ZERO_MAX_RANKS && unit->n_padded > 0 &&
           unit->shard_len > 0 && unit->shard_len % 8 == 0 &&
           unit->shard_len * n_ranks == unit->n_padded && unit->shard_offset >= 0 &&
           unit->shard_offset % 8 == 0;
}

int rs_unit(const zero_unit_t* unit, int32_t n_ranks, const void* const* unit_grads,
            float* const* master, float* const* m, float* const* v, uint16_t* const* shard_bf16,
            const zero_hparams_t* hp, const float* clip, cudaStream_t stream, bool f32 = false,
            bool g32 = false, bool chain_first = false, uint32_t* nonfinite = nullptr)
{
    if (!unit_valid(unit, n_ranks) || !valid_hparams(hp)) return ZERO_EINVAL;
    int rc = check_state_tables(n_ranks, reinterpret_cast<const uint16_t* const*>(unit_grads), master, m,
                                v);
    if (rc != ZERO_OK) return rc;
    if ((rc = check_table(shard_bf16, n_ranks)) != ZERO_OK) return rc;

    const int64_t off = unit->shard_offset;
    Tables T = {};
    for (int32_t r = 0; r < n_ranks; ++r) {
        if (g32)
            T.a[r] = reinterpret_cast<float4*>(
                const_cast<float*>(static_cast<const float*>(unit_grads[r])) + off);
        else
            T.g[r] = reinterpret_cast<const uint4*>(unit_grads[r]);
        T.w[r] = reinterpret_cast<float4*>(master[r] + off);
        T.m[r] = reinterpret_cast<float4*>(m[r] + off);
        T.v[r] = reinterpret_cast<float4*>(v[r] + off);
        T.o[r] = reinterpret_cast<uint4*>(shard_bf16[r] + off);
    }
    const StepScalars s = make_scalars(hp, n_ranks);
    return launch(T, s, 0, unit->n_padded / 8, unit->shard_len / 8, n_ranks, clip, stream, 0.0f,
                  f32, chain_first, g32, nonfinite);
}

int check_clip(const float* norm_coef)
{
    if (!norm_coef) return ZERO_EINVAL;
    return aligned16(norm_coef) ? ZERO_OK : ZERO_EALIGN;
}

// The finite check's output: a device uint32[2], 8-byte aligned.
int check_flags(const uint32_t* nonfinite)
{
    if (!nonfinite) return ZERO_EINVAL;
    return reinterpret_cast<uintptr_t>(nonfinite) % 8 == 0 ? ZERO_OK : ZERO_EALIGN;
}

} // namespace

int unit_update(const zero_unit_t* unit, int32_t n_ranks, const void* const* grads,
                float* const* master, float* const* m, float* const* v,
                uint16_t* const* shard_bf16, const zero_hparams_t* hp, const float* clip,
                cudaStream_t stream, bool f32, bool g32, bool chain_first, uint32_t* nonfinite)
{
    if (clip) {
        const int rc = check_clip(clip);
        if (rc != ZERO_OK) return rc;
    }
    if (nonfinite) {
        const int rc = check_flags(nonfinite);
        if (rc != ZERO_OK) return rc;
    }
    return rs_unit(unit, n_ranks, grads, master, m, v, shard_bf16, hp, clip, stream, f32, g32,
                   chain_first, nonfinite);
}

StepNodeList* step_nodes_begin()
{
    StepNodeList* log = new (std::nothrow) StepNodeList;
    t_capture_log = log;
    return log;
}

void step_nodes_end() { t_capture_log = nullptr; }

bool step_nodes_ok(const StepNodeList* log, size_t expected)
{
    return log && !log->failed && log->launches.size() == expected;
}

int step_nodes_set_scalars(StepNodeList* log, cudaGraphExec_t exec, const StepScalars& s)
{
    for (LoggedLaunch& x : log->launches) {
        x.s = s;
        void* args[4] = {&x.T, &x.s, &x.R, &x.clip};
        cudaKernelNodeParams p = {};
        p.func = const_cast<void*>(x.func);
        p.gridDim = dim3(x.blocks);
        p.blockDim = dim3(kBlock);
        p.sharedMemBytes = 0;
        p.kernelParams = args;
        p.extra = nullptr;
        const int rc = cuda_status(cudaGraphExecKernelNodeSetParams(exec, x.node, &p));
        if (rc != ZERO_OK) return rc;
    }
    return ZERO_OK;
}

void step_nodes_free(StepNodeList* log) { delete log; }

cudaGraphNode_t step_node_at(const StepNodeList* log, size_t i)
{
    return log && i < log->launches.size() ? log->launches[i].node : nullptr;
}

int preload_fused_kernels()
{
    const void* kernels[] = {
        reinterpret_cast<const void*>(fused_step_kernel<true, false, false, true>),
        reinterpret_cast<const void*>(fused_step_kernel<false, false, false, true>),
        reinterpret_cast<const void*>(fused_step_kernel<false, false, false, false, true>),
        reinterpret_cast<const void*>(fused_step_kernel<true, false, false, false, true>),
        reinterpret_cast<const void*>(fused_step_kernel<false, true, false, false, true>),
        reinterpret_cast<const void*>(fused_step_kernel<true, true, false, false, true>),
        reinterpret_cast<const void*>(fused_step_kernel<false, false, true, false, true>),
        reinterpret_cast<const void*>(fused_step_wide_kernel<false>),
        reinterpret_cast<const void*>(fused_step_wide_kernel<true>),
    };
    for (const void* k : kernels)
        if (persistent_blocks(k, kBlock, 0) <= 0) return ZERO_ECUDA;
    return ZERO_OK;
}

} // namespace zero

using namespace zero;

extern "C" int zero_step_stage12(int32_t stage, int32_t n_ranks, int64_t n_padded,
                                 const uint16_t* const* grads, float* const* master,
                                 float* const* m, float* const* v, uint16_t* params_bf16,
                                 const zero_hparams_t* hp, int64_t bucket_elems,
                                 cudaStream_t stream)
{
    return step_stage12(stage, n_ranks, n_padded, reinterpret_cast<const void* const*>(grads),
                        master, m, v, params_bf16, hp, bucket_elems, nullptr, stream);
}

extern "C" int zero_step_stage12_checked(int32_t stage, int32_t n_ranks, int64_t n_padded,
                                         const uint16_t* const* grads, float* const* master,
                                         float* const* m, float* const* v,
                                         uint16_t* params_bf16, const zero_hparams_t* hp,
                                         int64_t bucket_elems, uint32_t* nonfinite_ranks,
                                         cudaStream_t stream)
{
    const int rc = check_flags(nonfinite_ranks);
    if (rc != ZERO_OK) return rc;
    return step_stage12(stage, n_ranks, n_padded, reinterpret_cast<const void* const*>(grads),
                        master, m, v, params_bf16, hp, bucket_elems, nullptr, stream, false, false,
                        nonfinite_ranks);
}

extern "C" int zero_step_stage12_clip(int32_t stage, int32_t n_ranks, int64_t n_padded,
                                      const uint16_t* const* grads, float* const* master,
                                      float* const* m, float* const* v, uint16_t* params_bf16,
                                      const zero_hparams_t* hp, int64_t bucket_elems,
                                      const float* norm_coef, cudaStream_t stream)
{
    const int rc = check_clip(norm_coef);
    if (rc != ZERO_OK) return rc;
    return step_stage12(stage, n_ranks, n_padded, reinterpret_cast<const void* const*>(grads),
                        master, m, v, params_bf16, hp, bucket_elems, norm_coef, stream);
}

extern "C" int zero_step_stage12_reduced(int32_t stage, int32_t n_ranks, int64_t n_padded,
                                         const float* const* grad_shard, float* const* master,
                                         float* const* m, float* const* v,
                                         uint16_t* params_bf16, const zero_hparams_t* hp,
                                         int64_t bucket_elems, const float* norm_coef,
                                         cudaStream_t stream)
{
    if (norm_coef) {
        const int rc = check_clip(norm_coef);
        if (rc != ZERO_OK) return rc;
    }
    return step_stage12(stage, n_ranks, n_padded, reinterpret_cast<const void* const*>(grad_shard),
                        master, m, v, params_bf16, hp, bucket_elems, norm_coef, stream, false, true);
}

extern "C" int zero3_update_unit_reduced(const zero_unit_t* unit, int32_t n_ranks,
                                         const float* const* grad_shard, float* const* master,
                                         float* const* m, float* const* v,
                                         uint16_t* const* shard_bf16, const zero_hparams_t* hp,
                                         const float* norm_coef, cudaStream_t stream)
{
    if (norm_coef) {
        const int rc = check_clip(norm_coef);
        if (rc != ZERO_OK) return rc;
    }
    return rs_unit(unit, n_ranks, reinterpret_cast<const void* const*>(grad_shard), master, m, v,
                   shard_bf16, hp, norm_coef, stream, false, true);
}

extern "C" int zero3_reduce_scatter_unit(const zero_unit_t* unit, int32_t n_ranks,
                                         const uint16_t* const* unit_grads,
                                         float* const* master, float* const* m,
                                         float* const* v, uint16_t* const* shard_bf16,
                                         const zero_hparams_t* hp, cudaStream_t stream)
{
    return rs_unit(unit, n_ranks, reinterpret_cast<const void* const*>(unit_grads), master, m, v,
                   shard_bf16, hp, nullptr, stream);
}

extern "C" int zero3_reduce_scatter_unit_checked(const zero_unit_t* unit, int32_t n_ranks,
                                                 const uint16_t* const* unit_grads,
                                                 float* const* master, float* const* m,
                                                 float* const* v, uint16_t* const* shard_bf16,
                                                 const zero_hparams_t* hp,
                                                 uint32_t* nonfinite_ranks, cudaStream_t stream)
{
    const int rc = check_flags(nonfinite_ranks);
    if (rc != ZERO_OK) return rc;
    return rs_unit(unit, n_ranks, reinterpret_cast<const void* const*>(unit_grads), master, m, v,
                   shard_bf16, hp, nullptr, stream, false, false, false, nonfinite_ranks);
}

extern "C" int zero3_reduce_scatter_unit_clip(const zero_unit_t* unit, int32_t n_ranks,
                                              const uint16_t* const* unit_grads,
                                              float* const* master, float* const* m,
                                              float* const* v, uint16_t* const* shard_bf16,
                                              const zero_hparams_t* hp, const float* norm_coef,
                                              cudaStream_t stream)
{
    const int rc = check_clip(norm_coef);
    if (rc != ZERO_OK) return rc;
    return rs_unit(unit, n_ranks, reinterpret_cast<const void* const*>(unit_grads), master, m, v,
                   shard_bf16, hp, norm_coef, stream);
}

extern "C" int zero2_accumulate(int32_t n_ranks, int64_t n_padded, const uint16_t* const* grads,
                                float* const* grad_acc, int32_t first, cudaStream_t stream)
{
    if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS || n_padded <= 0 ||
        n_padded % (8 * static_cast<int64_t>(n_ranks)) != 0)
        return ZERO_EINVAL;
    int rc;
    if ((rc = check_table(grads, n_ranks)) != ZERO_OK) return rc;
    if ((rc = check_table(grad_acc, n_ranks)) != ZERO_OK) return rc;
    Tables T = {};
    for (int32_t r = 0; r < n_ranks; ++r) {
        T.g[r] = reinterpret_cast<const uint4*>(grads[r]);
        T.a[r] = reinterpret_cast<float4*>(grad_acc[r]);
    }
    const int64_t S = n_padded / n_ranks;
    // The four-block launch shape at every rank count (GB300, GPT-2 buffer, a
    // later micro-batch, ms: N_d = 5 0.335 -> 0.320, 8 0.425 -> 0.413, 12 0.573
    // -> 0.554, 16 0.701 -> 0.688, 24 0.981 -> 0.965 against the three-block
    // one; N_d = 32 7,116 -> 7,216 GB/s, 64 7,135 -> 7,212).
    const void* kernel = first ? reinterpret_cast<const void*>(accumulate_kernel<true>)
                               : reinterpret_cast<const void*>(accumulate_kernel<false>);
    const float inv_n = static_cast<float>(1.0 / static_cast<double>(n_ranks));
    // chained chunks of kChunkVec vectors, as the fused step's launch()
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    const int64_t nvec = n_padded / 8;
    for (int64_t a = 0; a < nvec; a += kChunkVec) {
        const int64_t b = nvec - a > kChunkVec ? a + kChunkVec : nvec;
        int blocks = 0;
        const Range R = make_range(kernel, a, b, S / 8, n_ranks, &blocks);
        if (blocks <= 0) return ZERO_ECUDA;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(blocks));
        cfg.blockDim = dim3(kBlock);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = a > 0 ? 1 : 0;
        const cudaError_t e = first ? cudaLaunchKernelEx(&cfg, accumulate_kernel<true>, T, inv_n, R)
                                    : cudaLaunchKernelEx(&cfg, accumulate_kernel<false>, T, inv_n, R);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return ZERO_OK;
}

extern "C" int zero2_step_accumulated(int32_t n_ranks, int64_t n_padded,
                                      const uint16_t* const* grads, float* const* grad_acc,
                                      int32_t micro_batches, float* const* master,
                                      float* const* m, float* const* v, uint16_t* params_bf16,
                                      const zero_hparams_t* hp, cudaStream_t stream)
{
    if (micro_batches < 1) return ZERO_EINVAL;
    if (micro_batches == 1)  // nothing accumulated: the plain ZeRO-2 step
        return step_stage12(2, n_ranks, n_padded, reinterpret_cast<const void* const*>(grads),
                            master, m, v, params_bf16, hp, 0, nullptr, stream);
    if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS || n_padded <= 0 ||
        n_padded % (8 * static_cast<int64_t>(n_ranks)) != 0 || !valid_hparams(hp) || !params_bf16)
        return ZERO_EINVAL;
    int rc = check_state_tables(n_ranks, grads, master, m, v);
    if (rc != ZERO_OK) return rc;
    if ((rc = check_table(grad_acc, n_ranks)) != ZERO_OK) return rc;
    if (!aligned16(params_bf16)) return ZERO_EALIGN;
    const int64_t S = n_padded / n_ranks;
    Tables T = {};
    for (int32_t r = 0; r < n_ranks; ++r) {
        T.g[r] = reinterpret_cast<const uint4*>(grads[r]);
        T.w[r] = reinterpret_cast<float4*>(master[r]);
        T.m[r] = reinterpret_cast<float4*>(m[r]);
        T.v[r] = reinterpret_cast<float4*>(v[r]);
        T.o[r] = reinterpret_cast<uint4*>(params_bf16 + r * S);
        T.a[r] = reinterpret_cast<float4*>(grad_acc[r]);
    }
    const StepScalars s = make_scalars(hp, n_ranks);
    const float inv_m = static_cast<float>(1.0 / static_cast<double>(micro_batches));
    return launch(T, s, 0, n_padded / 8, S / 8, n_ranks, nullptr, stream, inv_m);
}

extern "C" int zero3_accumulate_unit(const zero_unit_t* unit, int32_t n_ranks,
                                     const uint16_t* const* unit_grads, float* const* grad_acc,
                                     int32_t first, cudaStream_t stream)
{
    if (!unit_valid(unit, n_ranks)) return ZERO_EINVAL;
    const int rc = check_table(grad_acc, n_ranks);
    if (rc != ZERO_OK) return rc;
    float* acc[ZERO_MAX_RANKS];
    for (int32_t r = 0; r < n_ranks; ++r) acc[r] = grad_acc[r] + unit->shard_offset;
    return zero2_accumulate(n_ranks, unit->n_padded, unit_grads, acc, first, stream);
}

extern "C" int zero3_reduce_scatter_unit_accumulated(const zero_unit_t* unit, int32_t n_ranks,
                                                     const uint16_t* const* unit_grads,
                                                     float* const* grad_acc,
                                                     int32_t micro_batches, float* const* master,
                                                     float* const* m, float* const* v,
                                                     uint16_t* const* shard_bf16,
                                                     const zero_hparams_t* hp,
                                                     cudaStream_t stream)
{
    if (micro_batches < 1) return ZERO_EINVAL;
    if (micro_batches == 1) // nothing accumulated: the plain unit step
        return zero3_reduce_scatter_unit(unit, n_ranks, unit_grads, master, m, v, shard_bf16, hp,
                                         stream);
    if (!unit_valid(unit, n_ranks) || !valid_hparams(hp)) return ZERO_EINVAL;
    int rc = check_state_tables(n_ranks, unit_grads, master, m, v);
    if (rc != ZERO_OK) return rc;
    if ((rc = check_table(shard_bf16, n_ranks)) != ZERO_OK) return rc;
    if ((rc = check_table(grad_acc, n_ranks)) != ZERO_OK) return rc;
    const int64_t off = unit->shard_offset;
    Tables T = {};
    for (int32_t r = 0; r < n_ranks; ++r) {
        T.g[r] = reinterpret_cast<const uint4*>(unit_grads[r]);
        T.w[r] = reinterpret_cast<float4*>(master[r] + off);
        T.m[r] = reinterpret_cast<float4*>(m[r] + off);
        T.v[r] = reinterpret_cast<float4*>(v[r] + off);
        T.o[r] = reinterpret_cast<uint4*>(shard_bf16[r] + off);
        T.a[r] = reinterpret_cast<float4*>(grad_acc[r] + off);
    }
    const StepScalars s = make_scalars(hp, n_ranks);
    const float inv_m = static_cast<float>(1.0 / static_cast<double>(micro_batches));
    return launch(T, s, 0, unit->n_padded / 8, unit->shard_len / 8, n_ranks, nullptr, stream,
                  inv_m);
}

extern "C" int zero_step_stage12_f32grads(int32_t stage, int32_t n_ranks, int64_t n_padded,
                                          const float* const* grads, float* const* master,
                                          float* const* m, float* const* v,
                                          uint16_t* params_bf16, const zero_hparams_t* hp,
                                          int64_t bucket_elems, cudaStream_t stream)
{
    return step_stage12(stage, n_ranks, n_padded, reinterpret_cast<const void* const*>(grads),
                        master, m, v, params_bf16, hp, bucket_elems, nullptr, stream, true);
}

extern "C" int zero3_reduce_scatter_unit_f32grads(const zero_unit_t* unit, int32_t n_ranks,
                                                  const float* const* unit_grads,
                                                  float* const* master, float* const* m,
                                                  float* const* v, uint16_t* const* shard_bf16,
                                                  const zero_hparams_t* hp, cudaStream_t stream)
{
    return rs_unit(unit, n_ranks, reinterpret_cast<const void* const*>(unit_grads), master, m, v,
                   shard_bf16, hp, nullptr, stream, true);
}
