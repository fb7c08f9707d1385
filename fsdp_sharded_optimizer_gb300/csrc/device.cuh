// device.cuh -- small device helpers shared by the library's kernels:
// bf16 unpacking and nearest-even packing, streaming vector loads/stores.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace zero {
namespace dev {

// A uint32 word holds two bf16 values, element 2w in the low half.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 -> bf16 bits, round to nearest with ties to even: adding 0x7FFF plus
// the lowest kept bit carries into the kept half exactly when the discarded
// half is above one half, or equal to it with an odd kept part.  NaN maps to
// the canonical quiet NaN 0x7FC0; overflow rounds to infinity.
__device__ __forceinline__ uint32_t bf16_rne(float x)
{
    const uint32_t u = __float_as_uint(x);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    return bf16_rne(lo) | (bf16_rne(hi) << 16);
}

// Streaming accesses: every byte of these buffers is touched once per call,
// so they are loaded and stored with the evict-first (".cs") policy.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, uint4 x) { __stcs(p, x); }
__device__ __forceinline__ void st_stream(float4* p, float4 x) { __stcs(p, x); }

// Streaming 32-byte (256-bit) load and store of 8 consecutive fp32 values, one
// instruction each (sm_100 and later); p must be 32-byte aligned.
__device__ __forceinline__ void ld8_stream(const float4* p, float (&x)[8])
{
    asm volatile("ld.global.cs.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]), "=f"(x[4]), "=f"(x[5]),
                   "=f"(x[6]), "=f"(x[7])
                 : "l"(p));
}
__device__ __forceinline__ void st8_stream(float4* p, const float (&x)[8])
{
    asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
                 "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
                 "f"(x[7])
                 : "memory");
}

// Whether any of the 8 bf16 values in v is infinite or NaN (exponent all
// ones).  Per 16-bit half, (h & 0x7F80) + 0x0080 reaches 0x8000 exactly when
// the exponent field is all ones; a half's sum never carries into the other
// half.
__device__ __forceinline__ bool nonfinite_bf16x8(uint4 v)
{
    constexpr uint32_t kExp = 0x7F807F80u, kOne = 0x00800080u;
    const uint32_t x = ((v.x & kExp) + kOne) | ((v.y & kExp) + kOne) | ((v.z & kExp) + kOne) |
                       ((v.w & kExp) + kOne);
    return (x & 0x80008000u) != 0;
}

// The reduce-scatter's sum for 8 consecutive elements of vector q: fp32 from
// +0 over ranks 0..n_ranks-1 in order.  All loads of a batch of `kBatch`
// ranks are issued before any of them is summed.  kCheck: also set bit r of
// *bad when rank r's 8 values hold an infinity or a NaN (the sums are the
// same).
template <int kBatch, bool kCheck = false>
__device__ __forceinline__ void sum_ranks(const uint4* const* g, int n_ranks, int64_t q,
                                          float (&acc)[8], uint64_t* bad = nullptr)
{
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    for (int r0 = 0; r0 < n_ranks; r0 += kBatch) {
        uint4 G[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            if (r0 + i < n_ranks) G[i] = ld_stream(g[r0 + i] + q);
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (r0 + i < n_ranks) {
                if (kCheck && nonfinite_bf16x8(G[i])) *bad |= 1ull << (r0 + i);
                acc[0] = __fadd_rn(acc[0], bf16_lo(G[i].x));
                acc[1] = __fadd_rn(acc[1], bf16_hi(G[i].x));
                acc[2] = __fadd_rn(acc[2], bf16_lo(G[i].y));
                acc[3] = __fadd_rn(acc[3], bf16_hi(G[i].y));
                acc[4] = __fadd_rn(acc[4], bf16_lo(G[i].z));
                acc[5] = __fadd_rn(acc[5], bf16_hi(G[i].z));
                acc[6] = __fadd_rn(acc[6], bf16_lo(G[i].w));
                acc[7] = __fadd_rn(acc[7], bf16_hi(G[i].w));
            }
        }
    }
}

// The same sum for fp32 gradients: two 16-byte vectors per rank for the 8
// elements of vector q.
template <int kBatch>
__device__ __forceinline__ void sum_ranks_f32(const float4* const* g, int n_ranks, int64_t q,
                                              float (&acc)[8])
{
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    for (int r0 = 0; r0 < n_ranks; r0 += kBatch) {
        float4 G0[kBatch], G1[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            if (r0 + i < n_ranks) {
                G0[i] = ld_stream(g[r0 + i] + 2 * q);
                G1[i] = ld_stream(g[r0 + i] + 2 * q + 1);
            }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (r0 + i < n_ranks) {
                acc[0] = __fadd_rn(acc[0], G0[i].x);
                acc[1] = __fadd_rn(acc[1], G0[i].y);
                acc[2] = __fadd_rn(acc[2], G0[i].z);
                acc[3] = __fadd_rn(acc[3], G0[i].w);
                acc[4] = __fadd_rn(acc[4], G1[i].x);
                acc[5] = __fadd_rn(acc[5], G1[i].y);
                acc[6] = __fadd_rn(acc[6], G1[i].z);
                acc[7] = __fadd_rn(acc[7], G1[i].w);
            }
        }
    }
}

} // namespace dev
} // namespace zero
