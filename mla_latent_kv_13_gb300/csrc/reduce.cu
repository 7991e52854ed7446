// reduce.cu -- the two reductions of the path: the split-KV merge of decode partials
// (exact log-sum-exp weighting) and the sum of split-K GEMM partials into bf16.
#include "common.cuh"
#include "kernels.h"

namespace mla {

namespace {

// One CTA per (h, b); 128 threads x 4 latent columns.
__global__ void __launch_bounds__(128) combine_kernel(const float *o_part, const float *lse_part,
                                                      int S, int H, uint16_t *out, float *lse) {
    const int h = blockIdx.x, b = blockIdx.y;
    float m = -INFINITY;
    for (int s = 0; s < S; ++s) m = fmaxf(m, lse_part[((size_t)b * S + s) * H + h]);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float tot = -INFINITY;
    if (m != -INFINITY) {
        float den = 0.f;
        for (int s = 0; s < S; ++s) {
            float l = lse_part[((size_t)b * S + s) * H + h];
            if (l != -INFINITY) den += __expf(l - m);
        }
        tot = m + __logf(den);
        for (int s = 0; s < S; ++s) {
            float l = lse_part[((size_t)b * S + s) * H + h];
            if (l == -INFINITY) continue;
            float w = __expf(l - tot);
            float4 v = *reinterpret_cast<const float4 *>(
                o_part + (((size_t)b * S + s) * H + h) * D_C + threadIdx.x * 4);
            acc[0] += w * v.x;
            acc[1] += w * v.y;
            acc[2] += w * v.z;
            acc[3] += w * v.w;
        }
    }
    uint2 pk = make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
    *reinterpret_cast<uint2 *>(out + ((size_t)b * H + h) * D_C + threadIdx.x * 4) = pk;
    if (threadIdx.x == 0) lse[(size_t)b * H + h] = tot;
}

// Sum k-split partials [S][batch][M][N] into bf16 C (batch stride c_bstride, row ldc).
__global__ void reduce_partials_bf16(const float *part, int S, int batch, int M, int N,
                                     uint16_t *C, long ldc, long c_bstride) {
    long total = (long)batch * M * N / 2;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
         i += (long)gridDim.x * blockDim.x) {
        long e = i * 2;
        int n = e % N;
        long bm = e / N;
        int m = bm % M, bt = bm / M;
        float v0 = 0.f, v1 = 0.f;
        for (int s = 0; s < S; ++s) {
            float2 t = *reinterpret_cast<const float2 *>(part + ((long)s * batch * M * N) + e);
            v0 += t.x;
            v1 += t.y;
        }
        *reinterpret_cast<uint32_t *>(C + bt * c_bstride + (long)m * ldc + n) = pack_bf16x2(v0, v1);
    }
}

}  // namespace

cudaError_t launch_combine(const float *o_part, const float *lse_part, int B, int S, int H,
                           uint16_t *out, float *lse, cudaStream_t stream) {
    dim3 grid(H, B);
    combine_kernel<<<grid, 128, 0, stream>>>(o_part, lse_part, S, H, out, lse);
    return cudaGetLastError();
}

cudaError_t launch_reduce_bf16(const float *part, int S, int batch, int M, int N, uint16_t *C,
                               long ldc, long c_bstride, cudaStream_t stream) {
    long pairs = (long)batch * M * N / 2;
    long nb = (pairs + 255) / 256;
    int blocks = (int)(nb < 4096 ? nb : 4096);
    reduce_partials_bf16<<<blocks, 256, 0, stream>>>(part, S, batch, M, N, C, ldc, c_bstride);
    return cudaGetLastError();
}

}  // namespace mla
