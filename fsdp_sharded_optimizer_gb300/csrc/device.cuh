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

} // namespace dev
} // namespace zero
