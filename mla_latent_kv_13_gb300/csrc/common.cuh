// common.cuh -- small device helpers shared by the libmla kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla.h"

namespace mla {

constexpr int D_C = MLA_D_C;
constexpr int D_ROPE = MLA_D_ROPE;
constexpr int D_QK = MLA_D_QK;
constexpr int BLOCK = MLA_BLOCK;
constexpr int D_NOPE = MLA_D_NOPE;
constexpr int D_V = MLA_D_V;

// Workspace header: the sticky device error word sits at offset 0.
struct WsHeader {
    uint32_t error;       // first mla_status_t recorded by a kernel (0 = none)
    uint32_t detail;      // kernel-specific detail of that error (e.g. sequence index)
    uint32_t pad[62];
};
static_assert(sizeof(WsHeader) == MLA_WS_HEADER_BYTES, "header size");

__device__ __forceinline__ void flag_error(uint32_t *err, uint32_t code, uint32_t detail) {
    if (atomicCAS(err, 0u, code) == 0u) err[1] = detail;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// RoPE rotation of one pair (x0, x1) for pair index i of a 64-wide vector at
// position pos. The angle is formed in double so that large positions keep
// their fractional part; the rotation itself is done in fp32.
__device__ __forceinline__ void rope_pair(float &x0, float &x1, int i, int pos, float theta) {
    double freq = pow(static_cast<double>(theta), -2.0 * i / static_cast<double>(D_ROPE));
    double s, c;
    sincos(static_cast<double>(pos) * freq, &s, &c);
    float cf = static_cast<float>(c), sf = static_cast<float>(s);
    float y0 = x0 * cf - x1 * sf;
    float y1 = x0 * sf + x1 * cf;
    x0 = y0;
    x1 = y1;
}

}  // namespace mla
