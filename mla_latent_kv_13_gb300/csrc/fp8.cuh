// fp8.cuh -- e4m3 conversions of the FP8 latent cache (hardware cvt instructions).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"

namespace mla {

// 2^e as a float for e in [-126, 127] (exact).
__device__ __forceinline__ float exp2_int(int e) {
    return __int_as_float(static_cast<uint32_t>(127 + e) << 23);
}

// Two e4m3 codes (low byte = first value) to two f16 values (low half = first value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
    return r;
}

// The pair of codes dequantised with the power-of-two scale s and packed as bf16 (low
// half = first value). Every step is exact: e4m3 -> f16 (3-bit mantissas), f16 -> f32,
// the multiplication by a power of two, and the final bf16 rounding of a value that has
// at most four significant bits.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_scaled(uint16_t two, float s) {
    const uint32_t h = e4m3x2_to_f16x2(two);
    const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
    const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
    return pack_bf16x2(lo * s, hi * s);
}

// The same widening in five instructions, for the decode kernel's converter warps: every
// e4m3 value is a normal f16 (or zero) with only the top three of its ten mantissa bits
// set, so shifting the f16 pair right by 3 (the high half's low mantissa bits are zero, so
// nothing crosses the halves) and keeping the signs turns each half into the bf16 pattern
// of value * 2^-112 (exponent field 1..30, zero stays zero); one bf16 multiplication by
// s2 = 2^(112 + e) (a bf16 pair) then gives code * 2^e, exactly (normal results, products
// of at most four significant bits).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_mul(uint16_t two, uint32_t s2) {
    const uint32_t h = e4m3x2_to_f16x2(two);
    const uint32_t t = ((h >> 3) & 0x0FFF0FFFu) | (h & 0x80008000u);
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(s2));
    return r;
}
// bf16 pair (2^k, 2^k) for k in [-126, 127]
__device__ __forceinline__ uint32_t bf16x2_pow2(int k) {
    const uint32_t b = static_cast<uint32_t>(127 + k) << 7;
    return b | (b << 16);
}

// Two floats to two e4m3 codes, round to nearest even, saturating at +-448. The result's
// high byte is `hi`, its low byte `lo` (so a little-endian 16-bit store puts lo first).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace mla
