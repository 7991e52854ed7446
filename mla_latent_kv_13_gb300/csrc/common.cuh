// common.cuh -- small device helpers shared by the libmla kernels (sm_103a).
#pragma once

#include <utility>

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

// Programmatic dependent launch. Every kernel of the library is launched with
// launch_pdl, so it may start while its predecessor in the stream is still running: its
// prologue (barriers, TMEM, tensor-map and weight prefetch) overlaps the predecessor's tail.
// It calls grid_dependency_wait() before it reads anything a predecessor wrote (or writes
// anything a predecessor may still read), and grid_launch_dependents() once its successor may
// start -- in kernels that allocate TMEM only after the allocation, so that a successor CTA
// can never hold columns a not yet started CTA of this kernel needs.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// RoPE rotation frequencies theta^(-2i/64), i = 0..31, computed on the host in double
// and passed by value (a pow per element on the device costs far more than the
// rotation itself: fp64 throughput on this part is small).
struct RopeFreqs {
    double f[D_ROPE / 2];
};

// cos / sin of pos * freq. The product is formed in double and reduced to [-pi, pi]
// with a double fma (both exact enough for positions in the millions); the reduced
// angle is then evaluated in fp32.
__device__ __forceinline__ void rope_cos_sin(int pos, double freq, float &c, float &s) {
    const double a = static_cast<double>(pos) * freq;
    const double two_pi = 6.283185307179586476925286766559;
    const double k = rint(a * (1.0 / two_pi));
    const float r = static_cast<float>(fma(-k, two_pi, a));
    sincosf(r, &s, &c);
}

// Rotate the pair (x0, x1) by the angle pos * freq.
__device__ __forceinline__ void rope_pair(float &x0, float &x1, int pos, double freq) {
    float c, s;
    rope_cos_sin(pos, freq, c, s);
    const float y0 = x0 * c - x1 * s;
    const float y1 = x0 * s + x1 * c;
    x0 = y0;
    x1 = y1;
}

}  // namespace mla
