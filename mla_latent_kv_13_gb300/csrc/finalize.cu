// finalize.cu -- epilogues of the projection products: split-K reduction, RoPE on the
// decoupled position branch, bf16 rounding, and the paged-cache scatter of append.
#include "common.cuh"
#include "kernels.h"

namespace mla {

namespace {

// One CTA per sequence: threads 0..255 own latent columns (2t, 2t+1); threads
// 256..287 own RoPE pair t-256 (columns 512 + 2i, 513 + 2i).
__global__ void __launch_bounds__(288) append_finalize_kernel(
    const float *part, int S, int B, const int32_t *pos, const int32_t *block_table,
    int max_blocks, uint16_t *cache, int num_blocks, float theta, uint32_t *err) {
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
    for (int s = 0; s < S; ++s) {
        float2 v = *reinterpret_cast<const float2 *>(part + ((size_t)s * B + b) * D_QK + col);
        x0 += v.x;
        x1 += v.y;
    }
    if (col >= D_C) rope_pair(x0, x1, (col - D_C) / 2, p, theta);
    uint16_t *dst = cache + ((size_t)blk * BLOCK + (p % BLOCK)) * D_QK + col;
    *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(x0, x1);
}

// Grid-stride over (b, h, pair): sum the partials of c_q W_QR^T, rotate, store bf16.
__global__ void qrope_finalize_kernel(const float *part, int S, int B, int H, const int32_t *pos,
                                      float theta, uint16_t *q_rope) {
    const long n = (long)B * H * (D_ROPE / 2);
    const long row_len = (long)H * D_ROPE;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n;
         i += (long)gridDim.x * blockDim.x) {
        int pair = i % (D_ROPE / 2);
        long bh = i / (D_ROPE / 2);
        int b = bh / H;
        long off = (long)b * row_len + (bh % H) * D_ROPE + 2 * pair;
        float x0 = 0.f, x1 = 0.f;
        for (int s = 0; s < S; ++s) {
            float2 v = *reinterpret_cast<const float2 *>(part + (long)s * B * row_len + off);
            x0 += v.x;
            x1 += v.y;
        }
        rope_pair(x0, x1, pair, pos[b], theta);
        *reinterpret_cast<uint32_t *>(q_rope + bh * D_ROPE + 2 * pair) = pack_bf16x2(x0, x1);
    }
}

}  // namespace

cudaError_t launch_append_finalize(const float *part, int S, int B, const int32_t *pos,
                                   const int32_t *block_table, int max_blocks, uint16_t *cache,
                                   int num_blocks, float theta, uint32_t *err,
                                   cudaStream_t stream) {
    append_finalize_kernel<<<B, 288, 0, stream>>>(part, S, B, pos, block_table, max_blocks, cache,
                                                  num_blocks, theta, err);
    return cudaGetLastError();
}

cudaError_t launch_qrope_finalize(const float *part, int S, int B, int H, const int32_t *pos,
                                  float theta, uint16_t *q_rope, cudaStream_t stream) {
    long n = (long)B * H * (D_ROPE / 2);
    long nb = (n + 255) / 256;
    int blocks = (int)(nb < 4096 ? nb : 4096);
    qrope_finalize_kernel<<<blocks, 256, 0, stream>>>(part, S, B, H, pos, theta, q_rope);
    return cudaGetLastError();
}

}  // namespace mla
