// gemm_mma.cu -- skinny bf16 GEMM for the absorbed projections (batch rows x weights).
//
// C[m][n] = sum_k A[m][k] * B(k, n), fp32 accumulation, where B is either
//   "TN": stored [N][K] (row n is an output feature; the [out, in] weight layout), or
//   "NN": stored [K][N] (used for W_UK, whose rows are per-head key dims).
// A is [M][K] row-major with leading dimension lda. A batch index (grid.z / k_splits)
// offsets A, B and C by their batch strides (one batch per head for the per-head
// products). K is cut into k_splits ranges; each range writes an fp32 partial that
// a finalize kernel reduces, so that weight-bound products with few output
// columns still spread over every SM.
//
// Tiles: 64 (m) x 64 (n) x 64 (k), 4 warps of 32 x 32, three cp.async stages,
// XOR-swizzled 128-byte smem rows read with ldmatrix, mma.sync m16n8k16.
#include "common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr int GBM = 64, GBN = 64, GBK = 64, GSTAGES = 3;
constexpr int GTHREADS = 128;
constexpr int TILE_BYTES = GBM * GBK * 2;  // 8 KB (also GBK x GBN for NN)

template <bool NN>
__global__ void __launch_bounds__(GTHREADS) gemm_bf16_kernel(GemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n0 = blockIdx.x * GBN, m0 = blockIdx.y * GBM;
    const int batch = blockIdx.z / p.k_splits, split = blockIdx.z % p.k_splits;
    const int k_begin = split * p.k_per_split;
    const int k_end = min(p.K, k_begin + p.k_per_split);
    const int nk = (k_end - k_begin + GBK - 1) / GBK;

    const uint16_t *A = p.A + batch * p.a_bstride;
    const uint16_t *B = p.B + batch * p.b_bstride;

    uint8_t *sA = smem;
    uint8_t *sB = smem + GSTAGES * TILE_BYTES;

    auto load_stage = [&](int stage, int kt) {
        const int k0 = k_begin + kt * GBK;
        // A tile: 64 rows x 8 chunks of 16 B
        for (int i = tid; i < GBM * 8; i += GTHREADS) {
            int r = i >> 3, c = i & 7;
            int m = m0 + r, k = k0 + c * 8;
            bool ok = (m < p.M) && (k < k_end);
            const uint16_t *src = A + (ok ? (size_t)m * p.lda + k : 0);
            cp_async16(smem_u32(sA + stage * TILE_BYTES) + swz128(r, c), src, ok ? 16 : 0);
        }
        for (int i = tid; i < 64 * 8; i += GTHREADS) {
            int r = i >> 3, c = i & 7;
            const uint16_t *src;
            bool ok;
            if (!NN) {  // rows = n, chunks along k
                int n = n0 + r, k = k0 + c * 8;
                ok = (n < p.N) && (k < k_end);
                src = B + (ok ? (size_t)n * p.ldb + k : 0);
            } else {    // rows = k, chunks along n
                int k = k0 + r, n = n0 + c * 8;
                ok = (k < k_end) && (n < p.N);
                src = B + (ok ? (size_t)k * p.ldb + n : 0);
            }
            cp_async16(smem_u32(sB + stage * TILE_BYTES) + swz128(r, c), src, ok ? 16 : 0);
        }
    };

    float acc[2][4][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;

    const int wm = (warp >> 1) * 32, wn = (warp & 1) * 32;

#pragma unroll
    for (int s = 0; s < GSTAGES - 1; ++s) {
        if (s < nk) load_stage(s, s);
        cp_async_commit();
    }

    for (int kt = 0; kt < nk; ++kt) {
        cp_async_wait<GSTAGES - 2>();
        __syncthreads();
        {
            int nt = kt + GSTAGES - 1;
            if (nt < nk) load_stage(nt % GSTAGES, nt);
            cp_async_commit();
        }
        const uint32_t aBase = smem_u32(sA + (kt % GSTAGES) * TILE_BYTES);
        const uint32_t bBase = smem_u32(sB + (kt % GSTAGES) * TILE_BYTES);
#pragma unroll
        for (int ks = 0; ks < GBK / 16; ++ks) {
            uint32_t af[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                int row = wm + i * 16 + (lane & 15);
                int chunk = ks * 2 + (lane >> 4);
                ldsm_x4(aBase + swz128(row, chunk), af[i][0], af[i][1], af[i][2], af[i][3]);
            }
            uint32_t bf[4][2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                uint32_t r0, r1, r2, r3;
                if (!NN) {
                    // rows n: lanes 0-7 n0-7/k-lo, 8-15 n0-7/k-hi, 16-23 n8-15/k-lo, 24-31 n8-15/k-hi
                    int row = wn + j * 16 + (lane & 7) + ((lane >> 4) << 3);
                    int chunk = ks * 2 + ((lane >> 3) & 1);
                    ldsm_x4(bBase + swz128(row, chunk), r0, r1, r2, r3);
                } else {
                    // rows k: lanes 0-7 k0-7/n-lo, 8-15 k8-15/n-lo, 16-23 k0-7/n-hi, 24-31 k8-15/n-hi
                    int row = ks * 16 + (lane & 15);
                    int chunk = (wn + j * 16) / 8 + (lane >> 4);
                    ldsm_x4_t(bBase + swz128(row, chunk), r0, r1, r2, r3);
                }
                bf[j * 2][0] = r0;
                bf[j * 2][1] = r1;
                bf[j * 2 + 1][0] = r2;
                bf[j * 2 + 1][1] = r3;
            }
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) mma_bf16_16816(acc[i][j], af[i], bf[j][0], bf[j][1]);
        }
    }
    cp_async_wait<0>();

    // epilogue
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int hrow = 0; hrow < 2; ++hrow) {
                int m = m0 + wm + i * 16 + (lane >> 2) + hrow * 8;
                int n = n0 + wn + j * 8 + (lane & 3) * 2;
                if (m >= p.M || n >= p.N) continue;
                float v0 = acc[i][j][hrow * 2], v1 = acc[i][j][hrow * 2 + 1];
                if (p.c_part) {
                    float *dst = p.c_part +
                                 (((size_t)split * p.batch + batch) * p.M + m) * (size_t)p.N + n;
                    *reinterpret_cast<float2 *>(dst) = make_float2(v0, v1);
                } else {
                    uint16_t *dst = p.c_bf16 + batch * p.c_bstride + (size_t)m * p.ldc + n;
                    *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(v0, v1);
                }
            }
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

cudaError_t launch_gemm(const GemmParams &p, bool nn, cudaStream_t stream) {
    dim3 grid((p.N + GBN - 1) / GBN, (p.M + GBM - 1) / GBM, p.batch * p.k_splits);
    size_t smem = 2 * GSTAGES * TILE_BYTES;
    if (nn) {
        cudaFuncSetAttribute(gemm_bf16_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        gemm_bf16_kernel<true><<<grid, GTHREADS, smem, stream>>>(p);
    } else {
        cudaFuncSetAttribute(gemm_bf16_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        gemm_bf16_kernel<false><<<grid, GTHREADS, smem, stream>>>(p);
    }
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
