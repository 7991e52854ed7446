// fp8.cu -- the FP8 (e4m3) latent cache: quantisation of cache rows (one power-of-two
// scale per row), dequantisation, and the epilogue of the FP8 append.
//
// Format ("LLM inference: from the memory wall to the compute wall" §5 names a mixed-
// precision FP8/FP16 KV cache; the pages fix no format): e4m3 codes (bias 7, largest
// finite 448, no infinities), round to nearest with ties to even and saturation at 448
// (the hardware's cvt.rn.satfinite), and per cached row the exponent e of a power-of-two
// scale, the smallest with max|x| * 2^-e <= 448. A dequantised value code * 2^e has at
// most four significant bits, so it is exactly a bf16 value.
#include "common.cuh"
#include "fp8.cuh"
#include "kernels.h"

namespace mla {

namespace {

// Exponent of a row's scale from its largest magnitude (0 for an all-zero row), computed
// exactly from the bits of mx: the smallest e with mx * 2^-e <= 448.
__device__ __forceinline__ int row_scale_exp(float mx) {
    if (!(mx > 0.f)) return 0;
    // mx = f * 2^k with f in [1, 2): mx * 2^-e <= 448 = 1.75 * 2^8  <=>
    // e >= k - 8 when f <= 1.75, else e >= k - 7
    int k;
    const float f = 2.f * frexpf(mx, &k);  // frexpf: mx = (f / 2) * 2^k
    k -= 1;
    const int e = f <= 1.75f ? k - 8 : k - 7;
    return e < -126 ? -126 : e;  // the scale 2^-e must stay a normal float (rows < 2^-117)
}

// One warp per row of D (= 576) bf16 values: codes and the row's exponent.
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint16_t *src, long rows,
                                                            uint8_t *codes, int8_t *exps) {
    grid_launch_dependents();
    grid_dependency_wait();
    const long r = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const uint16_t *x = src + r * D_QK;
    float v[18];  // 576 / 32 values per lane: columns 2 * (lane + 32 j) + {0, 1}
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < 9; ++j) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(x + 2 * (lane + 32 * j));
        v[2 * j] = bf16_to_f32(static_cast<uint16_t>(w & 0xFFFFu));
        v[2 * j + 1] = bf16_to_f32(static_cast<uint16_t>(w >> 16));
        mx = fmaxf(mx, fmaxf(fabsf(v[2 * j]), fabsf(v[2 * j + 1])));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const int e = row_scale_exp(mx);
    const float s = exp2_int(-e);  // exact power of two
#pragma unroll
    for (int j = 0; j < 9; ++j)
        *reinterpret_cast<uint16_t *>(codes + r * D_QK + 2 * (lane + 32 * j)) =
            f32x2_to_e4m3x2(v[2 * j + 1] * s, v[2 * j] * s);
    if (lane == 0) exps[r] = static_cast<int8_t>(e);
}

// Codes and exponents back to bf16 rows (exact). One warp per row.
__global__ void __launch_bounds__(256) dequantize_rows_kernel(const uint8_t *codes,
                                                              const int8_t *exps, long rows,
                                                              uint16_t *dst) {
    grid_launch_dependents();
    grid_dependency_wait();
    const long r = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const float s = exp2_int(exps[r]);
#pragma unroll
    for (int j = 0; j < 9; ++j) {
        const int c = 2 * (lane + 32 * j);
        const uint16_t two = *reinterpret_cast<const uint16_t *>(codes + r * D_QK + c);
        *reinterpret_cast<uint32_t *>(dst + r * D_QK + c) = e4m3x2_to_bf16x2_scaled(two, s);
    }
}

// FP8 append epilogue: as append_finalize, but the rotated fp32 row is quantised (row
// max over its 576 values, the row's exponent, e4m3 codes) instead of rounded to bf16.
// One CTA of 288 threads per sequence: thread t owns columns (2t, 2t+1).
__global__ void __launch_bounds__(288) append_finalize_fp8_kernel(
    const float *part, int S, int B, const int32_t *pos, const int32_t *block_table,
    int max_blocks, uint8_t *codes, int8_t *exps, int num_blocks, RopeFreqs freqs,
    uint32_t *err) {
    __shared__ float wmax[9];
    grid_launch_dependents();
    grid_dependency_wait();
    const int b = blockIdx.x, t = threadIdx.x;
    const int p = pos[b];
    if (p < 0 || p >= max_blocks * BLOCK) {
        if (t == 0) flag_error(err, MLA_ERR_OUT_OF_RANGE, b);
        return;
    }
    const int blk = block_table[(size_t)b * max_blocks + p / BLOCK];
    if (blk < 0 || blk >= num_blocks) {
        if (t == 0) flag_error(err, MLA_ERR_OUT_OF_RANGE, b);
        return;
    }
    const int col = 2 * t;
    float x0 = 0.f, x1 = 0.f;
#pragma unroll 8
    for (int s = 0; s < S; ++s) {  // split order, as in the bf16 epilogue
        float2 v = *reinterpret_cast<const float2 *>(part + ((size_t)s * B + b) * D_QK + col);
        x0 += v.x;
        x1 += v.y;
    }
    if (col >= D_C) rope_pair(x0, x1, p, freqs.f[(col - D_C) / 2]);
    float mx = fmaxf(fabsf(x0), fabsf(x1));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((t & 31) == 0) wmax[t >> 5] = mx;
    __syncthreads();
    mx = wmax[0];
#pragma unroll
    for (int w = 1; w < 9; ++w) mx = fmaxf(mx, wmax[w]);
    const int e = row_scale_exp(mx);
    const float s = exp2_int(-e);
    const size_t slot = (size_t)blk * BLOCK + (p % BLOCK);
    *reinterpret_cast<uint16_t *>(codes + slot * D_QK + col) = f32x2_to_e4m3x2(x1 * s, x0 * s);
    if (t == 0) exps[slot] = static_cast<int8_t>(e);
}

RopeFreqs make_freqs_fp8(float theta) {
    RopeFreqs r;
    for (int i = 0; i < D_ROPE / 2; ++i)
        r.f[i] = pow(static_cast<double>(theta), -2.0 * i / static_cast<double>(D_ROPE));
    return r;
}

}  // namespace

cudaError_t launch_quantize_rows(const uint16_t *src, long rows, uint8_t *codes, int8_t *exps,
                                 cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    return launch_pdl(quantize_rows_kernel, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0,
                      stream, src, rows, codes, exps);
}

cudaError_t launch_dequantize_rows(const uint8_t *codes, const int8_t *exps, long rows,
                                   uint16_t *dst, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    return launch_pdl(dequantize_rows_kernel, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0,
                      stream, codes, exps, rows, dst);
}

cudaError_t launch_append_finalize_fp8(const float *part, int S, int B, const int32_t *pos,
                                       const int32_t *block_table, int max_blocks,
                                       uint8_t *codes, int8_t *exps, int num_blocks,
                                       float theta, uint32_t *err, cudaStream_t stream) {
    return launch_pdl(append_finalize_fp8_kernel, dim3(B), dim3(288), 0, stream, part, S, B, pos,
                      block_table, max_blocks, codes, exps, num_blocks, make_freqs_fp8(theta),
                      err);
}

}  // namespace mla
