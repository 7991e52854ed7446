// decode_mma.cu -- absorbed MLA decode attention with mma.sync (portable tensor path),
// and the split-KV combine.
//
// One CTA owns (token range s, sequence b, group of 64 heads). All heads of the
// group score the same 64-token latent tiles, so a tile is staged once in shared
// memory (cp.async, double buffered) and feeds both products:
//   S = Q [64 x 576] . K^T [576 x 64]   (K = [c_kv | k_rope] rows of the tile)
//   O += P [64 x 64] . V [64 x 512]     (V = the c_kv part of the same rows)
// with an online softmax in the exp2 domain between them. Eight warps: for S
// each warp owns 16 heads x 32 tokens; for PV each warp owns 32 heads x 128
// latent columns, whose fp32 accumulators stay in registers across tiles.
#include "common.cuh"
#include "kernels.h"

namespace mla {

namespace {

constexpr int HPC = 64;            // heads per CTA
constexpr int TOK = 64;            // tokens per tile (= cache block)
constexpr int NTHR = 256;
constexpr int SEG = 9;             // 576 = 9 segments of 64 bf16 (128 B)
constexpr int SEG_BYTES = 64 * 128;
constexpr int Q_BYTES = SEG * SEG_BYTES;   // 72 KB
constexpr int KV_BYTES = SEG * SEG_BYTES;  // 72 KB per stage
constexpr int P_BYTES = SEG_BYTES;         // 64 heads x 64 tokens bf16
constexpr int SMEM_BYTES = Q_BYTES + 2 * KV_BYTES + P_BYTES + 6 * 64 * 4 + 64 * 4;

__device__ __forceinline__ uint32_t seg_addr(uint32_t base, int row, int col_chunk) {
    // col_chunk counts 16-byte chunks across the 576-wide row (0..71)
    return base + (col_chunk >> 3) * SEG_BYTES + swz128(row, col_chunk & 7);
}

__global__ void __launch_bounds__(NTHR, 1) decode_mma_kernel(DecodeParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *sQ = smem;
    uint8_t *sKV = smem + Q_BYTES;
    uint8_t *sP = sKV + 2 * KV_BYTES;
    float *sRed = reinterpret_cast<float *>(sP + P_BYTES);  // [2][64] tile row max halves
    float *sL = sRed + 128;                                  // [2][64] row sums halves
    float *sLe = sL + 128;                                   // [2][64] exact sums halves
    float *sAlpha = sLe + 128;                               // [64]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, b = blockIdx.y, h0 = blockIdx.z * HPC;
    const int H = p.H;

    int L = p.seqlens[b];
    if (L < 0 || L > p.max_blocks * TOK) {
        if (tid == 0) flag_error(p.err, MLA_ERR_OUT_OF_RANGE, b);
        L = L < 0 ? 0 : p.max_blocks * TOK;
    }
    const int ntiles = (L + TOK - 1) / TOK;
    const int t_begin = split * p.tiles_per_split;
    const int t_end = min(ntiles, t_begin + p.tiles_per_split);
    const int32_t *btab = p.block_table + (size_t)b * p.max_blocks;

    const uint32_t qBase = smem_u32(sQ);
    const uint32_t kvBase = smem_u32(sKV);
    const uint32_t pBase = smem_u32(sP);

    // ---- Q: 64 rows x 72 chunks (rows >= H zero-filled)
    for (int i = tid; i < HPC * 72; i += NTHR) {
        int r = i / 72, c = i % 72;
        int h = h0 + r;
        bool ok = h < H;
        const uint16_t *src;
        if (c < 64)
            src = p.q_lat + ((size_t)b * H + (ok ? h : 0)) * D_C + c * 8;
        else
            src = p.q_rope + ((size_t)b * H + (ok ? h : 0)) * D_ROPE + (c - 64) * 8;
        cp_async16(seg_addr(qBase, r, c), src, ok ? 16 : 0);
    }

    auto load_tile = [&](int stage, int tile) {
        int blk = btab[tile];
        bool ok = blk >= 0 && blk < p.num_blocks;
        if (!ok && tid == 0) flag_error(p.err, MLA_ERR_OUT_OF_RANGE, b);
        const uint16_t *base = p.cache + (size_t)(ok ? blk : 0) * TOK * D_QK;
        uint32_t dst = kvBase + stage * KV_BYTES;
        // rows past the sequence end are zero-filled: their probabilities are 0, and
        // 0 * (stale NaN/Inf) would otherwise poison the P.V product
        const int valid_rows = min(TOK, L - tile * TOK);
        for (int i = tid; i < TOK * 72; i += NTHR) {
            int r = i / 72, c = i % 72;
            bool rok = ok && r < valid_rows;
            cp_async16(seg_addr(dst, r, c), base + (size_t)(rok ? r : 0) * D_QK + c * 8,
                       rok ? 16 : 0);
        }
    };

    if (t_begin < t_end) load_tile(0, t_begin);
    cp_async_commit();

    // S-phase role
    const int hm = warp & 3, th = warp >> 2;
    // PV-phase role
    const int hg = warp >> 2, lq = warp & 3;

    float o[2][16][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 16; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[i][j][e] = 0.f;

    float m_run[2] = {-INFINITY, -INFINITY};  // rows g and g+8 of the S-role head tile
    float l_run[2] = {0.f, 0.f};   // sums of the bf16-rounded p this warp feeds to P.V
    float le_run[2] = {0.f, 0.f};  // sums of the unrounded p (for lse)

    for (int tile = t_begin; tile < t_end; ++tile) {
        const int stage = (tile - t_begin) & 1;
        if (tile + 1 < t_end) load_tile(stage ^ 1, tile + 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const int blk = btab[tile];
        const bool blk_ok = blk >= 0 && blk < p.num_blocks;
        const uint32_t kv = kvBase + stage * KV_BYTES;

        // ---------------- S = Q K^T for 16 heads x 32 tokens
        float s[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
#pragma unroll 4
        for (int ks = 0; ks < 36; ++ks) {
            uint32_t a[4];
            ldsm_x4(seg_addr(qBase, hm * 16 + (lane & 15), ks * 2 + (lane >> 4)), a[0], a[1],
                    a[2], a[3]);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                uint32_t r0, r1, r2, r3;
                int row = th * 32 + j * 16 + (lane & 7) + ((lane >> 4) << 3);
                ldsm_x4(seg_addr(kv, row, ks * 2 + ((lane >> 3) & 1)), r0, r1, r2, r3);
                mma_bf16_16816(s[2 * j], a, r0, r1);
                mma_bf16_16816(s[2 * j + 1], a, r2, r3);
            }
        }

        // ---------------- online softmax (exp2 domain)
        const int tok0 = tile * TOK;
        float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int t = tok0 + th * 32 + j * 8 + (lane & 3) * 2 + (e & 1);
                bool valid = blk_ok && t < L;
                float x = valid ? s[j][e] * p.scale_log2 : -INFINITY;
                s[j][e] = x;
                tmax[e >> 1] = fmaxf(tmax[e >> 1], x);
            }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
            tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
        }
        if ((lane & 3) == 0) {
            sRed[th * 64 + hm * 16 + (lane >> 2)] = tmax[0];
            sRed[th * 64 + hm * 16 + (lane >> 2) + 8] = tmax[1];
        }
        __syncthreads();
        float alpha[2], m_new[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            int row = hm * 16 + (lane >> 2) + r * 8;
            float mt = fmaxf(sRed[row], sRed[64 + row]);
            m_new[r] = fmaxf(m_run[r], mt);
            alpha[r] = (m_new[r] == -INFINITY) ? 1.f : fast_exp2(m_run[r] - m_new[r]);
        }
        float rsum[2] = {0.f, 0.f}, esum[2] = {0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float p0 = (m_new[r] == -INFINITY) ? 0.f : fast_exp2(s[j][2 * r] - m_new[r]);
                float p1 = (m_new[r] == -INFINITY) ? 0.f : fast_exp2(s[j][2 * r + 1] - m_new[r]);
                uint32_t pk = pack_bf16x2(p0, p1);
                // the output is normalised by the sum of the values the P.V product
                // actually uses (bf16-rounded); lse uses the unrounded sum
                rsum[r] += bf16_to_f32(pk & 0xffff) + bf16_to_f32(pk >> 16);
                esum[r] += p0 + p1;
                int row = hm * 16 + (lane >> 2) + r * 8;
                int col = th * 32 + j * 8 + (lane & 3) * 2;  // token within tile
                uint32_t addr = pBase + swz128(row, col >> 3) + (col & 7) * 2;
                asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(addr), "r"(pk));
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            rsum[r] += __shfl_xor_sync(0xffffffffu, rsum[r], 1);
            rsum[r] += __shfl_xor_sync(0xffffffffu, rsum[r], 2);
            esum[r] += __shfl_xor_sync(0xffffffffu, esum[r], 1);
            esum[r] += __shfl_xor_sync(0xffffffffu, esum[r], 2);
            l_run[r] = l_run[r] * alpha[r] + rsum[r];
            le_run[r] = le_run[r] * alpha[r] + esum[r];
            m_run[r] = m_new[r];
        }
        if (th == 0 && (lane & 3) == 0) {
            sAlpha[hm * 16 + (lane >> 2)] = alpha[0];
            sAlpha[hm * 16 + (lane >> 2) + 8] = alpha[1];
        }
        __syncthreads();

        // ---------------- O = O * alpha + P V for 32 heads x 128 latent columns
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float a0 = sAlpha[hg * 32 + i * 16 + (lane >> 2)];
            float a1 = sAlpha[hg * 32 + i * 16 + (lane >> 2) + 8];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                o[i][j][0] *= a0;
                o[i][j][1] *= a0;
                o[i][j][2] *= a1;
                o[i][j][3] *= a1;
            }
        }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t a[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i)
                ldsm_x4(pBase + swz128(hg * 32 + i * 16 + (lane & 15), ks * 2 + (lane >> 4)),
                        a[i][0], a[i][1], a[i][2], a[i][3]);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                int c0 = lq * 128 + jj * 16;  // latent column of this n-tile pair
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(seg_addr(kv, ks * 16 + (lane & 15), (c0 >> 3) + (lane >> 4)), r0, r1,
                          r2, r3);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    mma_bf16_16816(o[i][2 * jj], a[i], r0, r1);
                    mma_bf16_16816(o[i][2 * jj + 1], a[i], r2, r3);
                }
            }
        }
        __syncthreads();  // P and this KV stage are free again
    }
    cp_async_wait<0>();

    // ---- final row sums and maxima
    if ((lane & 3) == 0) {
        sL[th * 64 + hm * 16 + (lane >> 2)] = l_run[0];
        sL[th * 64 + hm * 16 + (lane >> 2) + 8] = l_run[1];
        sLe[th * 64 + hm * 16 + (lane >> 2)] = le_run[0];
        sLe[th * 64 + hm * 16 + (lane >> 2) + 8] = le_run[1];
        if (th == 0) {
            sRed[hm * 16 + (lane >> 2)] = m_run[0];
            sRed[hm * 16 + (lane >> 2) + 8] = m_run[1];
        }
    }
    __syncthreads();

    const bool direct = p.num_splits == 1;
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            int row = hg * 32 + i * 16 + (lane >> 2) + r * 8;
            int h = h0 + row;
            if (h >= H) continue;
            float l = sL[row] + sL[64 + row];
            float inv = l > 0.f ? 1.f / l : 0.f;
            size_t obase = direct ? ((size_t)b * H + h) * D_C
                                  : (((size_t)b * p.num_splits + split) * H + h) * D_C;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                int c = lq * 128 + j * 8 + (lane & 3) * 2;
                float v0 = o[i][j][2 * r] * inv, v1 = o[i][j][2 * r + 1] * inv;
                if (direct)
                    *reinterpret_cast<uint32_t *>(p.out + obase + c) = pack_bf16x2(v0, v1);
                else
                    *reinterpret_cast<float2 *>(p.o_part + obase + c) = make_float2(v0, v1);
            }
            if (lq == 0 && (lane & 3) == 0) {
                float m2 = sRed[row];
                float le = sLe[row] + sLe[64 + row];
                float lse = le > 0.f ? (m2 + log2f(le)) * 0.69314718055994531f : -INFINITY;
                if (direct)
                    p.lse[(size_t)b * H + h] = lse;
                else
                    p.lse_part[((size_t)b * p.num_splits + split) * H + h] = lse;
            }
        }
}

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

}  // namespace

cudaError_t launch_decode_mma(const DecodeParams &p, cudaStream_t stream) {
    dim3 grid(p.num_splits, p.B, (p.H + HPC - 1) / HPC);
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    decode_mma_kernel<<<grid, NTHR, SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float *o_part, const float *lse_part, int B, int S, int H,
                           uint16_t *out, float *lse, cudaStream_t stream) {
    dim3 grid(H, B);
    combine_kernel<<<grid, 128, 0, stream>>>(o_part, lse_part, S, H, out, lse);
    return cudaGetLastError();
}

}  // namespace mla
