// finalize.cu -- epilogues of the projection products: split-K reduction, RoPE on the
// decoupled position branch, bf16 rounding, and the paged-cache scatter of append.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace mla {

namespace {

// One CTA per sequence: threads 0..255 own latent columns (2t, 2t+1); threads
// 256..287 own RoPE pair t-256 (columns 512 + 2i, 513 + 2i).
__global__ void __launch_bounds__(288) append_finalize_kernel(
    const float *part, int S, int B, const int32_t *pos, const int32_t *block_table,
    int max_blocks, uint16_t *cache, int num_blocks, RopeFreqs freqs, uint32_t *err) {
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
    const int col = 2 * t;  // 0..574
    float x0 = 0.f, x1 = 0.f;
    // the split partials are summed in split order; unrolled so the loads overlap
#pragma unroll 8
    for (int s = 0; s < S; ++s) {
        float2 v = *reinterpret_cast<const float2 *>(part + ((size_t)s * B + b) * D_QK + col);
        x0 += v.x;
        x1 += v.y;
    }
    if (col >= D_C) rope_pair(x0, x1, p, freqs.f[(col - D_C) / 2]);
    uint16_t *dst = cache + ((size_t)blk * BLOCK + (p % BLOCK)) * D_QK + col;
    *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(x0, x1);
}

// CTA (b, y): 256 of the H x 32 (head, pair) entries of sequence b. The 32 rotations of
// its position are formed first; each thread reduces one pair of c_q W_QR^T over the
// k-splits (in split order), rotates it and stores it bf16.
__global__ void __launch_bounds__(256) qrope_finalize_kernel(const float *part, int S, int B,
                                                             int H, const int32_t *pos,
                                                             RopeFreqs freqs, uint16_t *q_rope) {
    __shared__ float cs[D_ROPE / 2], sn[D_ROPE / 2];
    grid_launch_dependents();
    grid_dependency_wait();
    const int b = blockIdx.x;
    if (threadIdx.x < D_ROPE / 2)
        rope_cos_sin(pos[b], freqs.f[threadIdx.x], cs[threadIdx.x], sn[threadIdx.x]);
    __syncthreads();
    const int e = blockIdx.y * blockDim.x + threadIdx.x;
    if (e >= H * (D_ROPE / 2)) return;
    const long row_len = (long)H * D_ROPE;
    const int h = e / (D_ROPE / 2), pair = e % (D_ROPE / 2);
    const long off = (long)b * row_len + (long)h * D_ROPE + 2 * pair;
    float x0 = 0.f, x1 = 0.f;
#pragma unroll 8
    for (int s = 0; s < S; ++s) {
        float2 v = *reinterpret_cast<const float2 *>(part + (long)s * B * row_len + off);
        x0 += v.x;
        x1 += v.y;
    }
    const float y0 = x0 * cs[pair] - x1 * sn[pair];
    const float y1 = x0 * sn[pair] + x1 * cs[pair];
    *reinterpret_cast<uint32_t *>(q_rope + off) = pack_bf16x2(y0, y1);
}

RopeFreqs make_freqs(float theta) {
    RopeFreqs r;
    for (int i = 0; i < D_ROPE / 2; ++i)
        r.f[i] = std::pow(static_cast<double>(theta), -2.0 * i / static_cast<double>(D_ROPE));
    return r;
}

}  // namespace

cudaError_t launch_append_finalize(const float *part, int S, int B, const int32_t *pos,
                                   const int32_t *block_table, int max_blocks, uint16_t *cache,
                                   int num_blocks, float theta, uint32_t *err,
                                   cudaStream_t stream) {
    return launch_pdl(append_finalize_kernel, dim3(B), dim3(288), 0, stream, part, S, B, pos,
                      block_table, max_blocks, cache, num_blocks, make_freqs(theta), err);
}

cudaError_t launch_qrope_finalize(const float *part, int S, int B, int H, const int32_t *pos,
                                  float theta, uint16_t *q_rope, cudaStream_t stream) {
    const dim3 grid(B, (H * (D_ROPE / 2) + 255) / 256);
    return launch_pdl(qrope_finalize_kernel, grid, dim3(256), 0, stream, part, S, B, H, pos,
                      make_freqs(theta), q_rope);
}

}  // namespace mla
