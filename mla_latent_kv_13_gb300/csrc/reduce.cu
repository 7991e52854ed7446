// reduce.cu -- the two reductions of the path: the split-KV merge of decode partials
// (exact log-sum-exp weighting) and the sum of split-K GEMM partials into bf16; and the
// balanced decode schedule's device-side offsets, weights and part counts.
#include "common.cuh"
#include "kernels.h"

namespace mla {

namespace {

// Merge np partial rows (fp32 [512], each with its log-sum-exp) into one bf16 row and its
// log-sum-exp, with one warp: lane l holds columns 4l + 128k (k < 4), so every part row is
// read as four coalesced 512-byte segments. Every lane reads every part's log-sum-exp (one
// broadcast load each). The rows of the first two parts are loaded together with the
// log-sum-exps, before the weights are known, so that merging two parts (a sequence cut
// once) takes one memory round trip; further parts follow two at a time. Parts are
// accumulated in order. A part with lse = -inf (an empty range) contributes nothing.
__device__ __forceinline__ void merge_row_warp(const float *o0, size_t ostride, const float *l0,
                                               size_t lstride, int np, uint16_t *orow,
                                               float *orow32, float *lse_out, int lane) {
    auto load_row = [&](int s, float4 (&v)[4]) {
        const float *row = o0 + (size_t)s * ostride + lane * 4;
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = __ldcs(reinterpret_cast<const float4 *>(row + 128 * k));
    };
    float4 va[4], vb[4];
    const float la = np > 0 ? l0[0] : -INFINITY;
    const float lb = np > 1 ? l0[lstride] : -INFINITY;
    if (np > 0) load_row(0, va);
    if (np > 1) load_row(1, vb);
    float m = fmaxf(la, lb);
    for (int s = 2; s < np; ++s) m = fmaxf(m, l0[s * lstride]);
    float tot = -INFINITY;
    if (m != -INFINITY) {
        float den = 0.f;
        if (la != -INFINITY) den += __expf(la - m);
        if (lb != -INFINITY) den += __expf(lb - m);
        for (int s = 2; s < np; ++s) {
            const float l = l0[s * lstride];
            if (l != -INFINITY) den += __expf(l - m);
        }
        tot = m + __logf(den);
    }
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    auto add_row = [&](float l, const float4 (&v)[4]) {
        const float w = l != -INFINITY ? __expf(l - tot) : 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc[4 * k] += w * v[k].x;
            acc[4 * k + 1] += w * v[k].y;
            acc[4 * k + 2] += w * v[k].z;
            acc[4 * k + 3] += w * v[k].w;
        }
    };
    if (tot != -INFINITY) {
        if (np > 0) add_row(la, va);
        if (np > 1) add_row(lb, vb);
        for (int s = 2; s < np; s += 2) {
            const float l2 = l0[s * lstride];
            const float l3 = s + 1 < np ? l0[(s + 1) * lstride] : -INFINITY;
            load_row(s, va);
            if (s + 1 < np) load_row(s + 1, vb);
            add_row(l2, va);
            if (s + 1 < np) add_row(l3, vb);
        }
    }
    if (orow32) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            *reinterpret_cast<float4 *>(orow32 + lane * 4 + 128 * k) =
                make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint2 *>(orow + lane * 4 + 128 * k) =
                make_uint2(pack_bf16x2(acc[4 * k], acc[4 * k + 1]),
                           pack_bf16x2(acc[4 * k + 2], acc[4 * k + 3]));
    }
    if (lane == 0) *lse_out = tot;
}

constexpr int MERGE_ROWS = 8;  // head rows (one warp each) per CTA of the merge kernels

// Rows (b, h) of S parts each (token ranges of one sequence, or one range per rank), part s
// of row (b, h) at o_part + b * o_bstride + s * o_pstride + h * 512 (lse likewise).
// Grid (ceil(H / 8), B), 256 threads.
__global__ void __launch_bounds__(32 * MERGE_ROWS)
    combine_kernel(const float *o_part, const float *lse_part, int S, int H, long o_bstride,
                   long o_pstride, long l_bstride, long l_pstride, uint16_t *out,
                   float *out_f32, float *lse) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int h = blockIdx.x * MERGE_ROWS + (threadIdx.x >> 5), b = blockIdx.y;
    if (h >= H) return;
    const size_t row = (size_t)b * H + h;
    merge_row_warp(o_part + b * o_bstride + (size_t)h * D_C, o_pstride,
                   lse_part + b * l_bstride + h, l_pstride, S,
                   out_f32 ? nullptr : out + row * D_C, out_f32 ? out_f32 + row * D_C : nullptr,
                   lse + row, threadIdx.x & 31);
}

// Sum k-split partials [S][batch][M][N] into bf16 C (batch stride c_bstride, row ldc).
__global__ void reduce_partials_bf16(const float *part, int S, int batch, int M, int N,
                                     uint16_t *C, long ldc, long c_bstride) {
    grid_launch_dependents();
    grid_dependency_wait();
    long total = (long)batch * M * N / 2;
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total;
         i += (long)gridDim.x * blockDim.x) {
        long e = i * 2;
        int n = e % N;
        long bm = e / N;
        int m = bm % M, bt = bm / M;
        float v0 = 0.f, v1 = 0.f;
#pragma unroll 8
        for (int s = 0; s < S; ++s) {  // split order; unrolled so the loads overlap
            float2 t = *reinterpret_cast<const float2 *>(part + ((long)s * batch * M * N) + e);
            v0 += t.x;
            v1 += t.y;
        }
        *reinterpret_cast<uint32_t *>(C + bt * c_bstride + (long)m * ldc + n) = pack_bf16x2(v0, v1);
    }
}

// Block-wide exclusive scan of v over n <= 4 * blockDim.x elements (1024 threads).
__device__ int block_exclusive_scan4(const int *v, int n, int *out, int *warp_tot) {
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    int a[4], sum = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = 4 * t + k;
        a[k] = i < n ? v[i] : 0;
        sum += a[k];
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) warp_tot[w] = inc;
    __syncthreads();
    if (w == 0) {
        const int x = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
        int xi = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, xi, o);
            if (lane >= o) xi += y;
        }
        warp_tot[lane] = xi - x;  // exclusive prefix of the warp totals
        if (lane == 31) warp_tot[32] = xi;
    }
    __syncthreads();
    int run = warp_tot[w] + inc - sum;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = 4 * t + k;
        if (i < n) out[i] = run;
        run += a[k];
    }
    const int total = warp_tot[32];
    __syncthreads();
    return total;
}

// One CTA of 1024 threads (B <= 4096): tiles per sequence -> tile_start; weighted positions
// (SEG_COST + tiles per sequence with tiles) -> wpos; parts of the sequences that the equal
// split of the total weight cuts between clusters -> nparts, part_begin; and the merge jobs:
// the sequence cut at the end of cluster c's range (its first tile in that range) is job c,
// jobs[c] = (b, first part, parts), else (-1, 0, 0). Reads only seqlens, so it may run once
// for several attention calls over the same lengths. Everything is computed in shared memory
// before the dependency wait, which comes only before the first store: the lengths are the
// caller's input, so the kernel may run beside its predecessor (the last query projection of
// a decode step), while its outputs may still be read by the previous attention call's merge.
__global__ void __launch_bounds__(1024) decode_schedule_kernel(
    const int32_t *seqlens, int B, int max_len, int P, int32_t *tile_start, int32_t *wpos,
    int32_t *part_begin, int32_t *nparts, int4 *jobs, uint32_t *err) {
    // dynamic shared memory, four arrays of B: v = tiles per sequence, later parts per
    // sequence; ts = the tiles' exclusive scan (tile_start); wp = the weights' exclusive
    // scan, then the weighted positions (wpos); pb = the parts' exclusive scan (part_begin)
    extern __shared__ int sched_smem[];
    int *const v = sched_smem, *const ts = v + B, *const wp = ts + B, *const pb = wp + B;
    __shared__ int warp_tot[33];
    __shared__ int bad;
    grid_launch_dependents();
    if (threadIdx.x == 0) bad = -1;
    __syncthreads();
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        int L = seqlens[b];
        if (L < 0 || L > max_len) {  // the attention kernel clamps the same way
            atomicMax(&bad, b);
            L = L < 0 ? 0 : max_len;
        }
        v[b] = (L + BLOCK - 1) / BLOCK;
    }
    __syncthreads();
    const int T = block_exclusive_scan4(v, B, ts, warp_tot);
    for (int b = threadIdx.x; b < B; b += blockDim.x) wp[b] = v[b] > 0 ? v[b] + SEG_COST : 0;
    __syncthreads();
    const int W = block_exclusive_scan4(wp, B, wp, warp_tot);  // in place
    // never more ranges than weight positions, so that every range is non-empty and a
    // sequence cut between clusters c0..c1 gets exactly one part from each of them
    const int Pe = W < P ? W : P;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int w0 = wp[b] + (v[b] > 0 ? SEG_COST : 0);
        int np = 0;
        if (v[b] > 0) {
            const int c0 = cluster_of_tile(w0, W, Pe);
            const int c1 = cluster_of_tile(w0 + v[b] - 1, W, Pe);
            np = c1 > c0 ? c1 - c0 + 1 : 0;
        }
        wp[b] = w0;
        v[b] = np;  // the tile counts are in ts from here on
    }
    __syncthreads();
    block_exclusive_scan4(v, B, pb, warp_tot);
    // every output below may still be read by the attention call before this one
    grid_dependency_wait();
    if (threadIdx.x == 0 && bad >= 0) flag_error(err, MLA_ERR_OUT_OF_RANGE, bad);
    for (int c = threadIdx.x; c < P; c += blockDim.x) jobs[c] = make_int4(-1, 0, 0, 0);
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        tile_start[b] = ts[b];
        wpos[b] = wp[b];
        nparts[b] = v[b];
        part_begin[b] = pb[b];
    }
    if (threadIdx.x == 0) {
        tile_start[B] = T;
        wpos[B] = W;
    }
    __syncthreads();  // the job list is cleared before the jobs go in
    for (int b = threadIdx.x; b < B; b += blockDim.x)
        if (v[b] > 0) jobs[cluster_of_tile(wp[b], W, Pe)] = make_int4(b, pb[b], v[b], 0);
}

constexpr int EMPTY_CTAS = 32;  // rows of CTAs of the merge kernel writing empty sequences

// Balanced schedule, after the attention kernel. Grid (ceil(H / 8), P + EMPTY_CTAS), one warp
// per head row. CTA (x, c < P) merges rows 8x .. 8x+7 of job c, the sequence cut at the end
// of cluster c's range. CTA (x, P + j) writes rows 8x .. 8x+7 of the sequences without tiles
// among b = j (mod EMPTY_CTAS), which no cluster's range holds: out = 0 (or out_f32 = 0),
// lse = -inf. The job list comes from the schedule kernel, which had finished before the
// attention kernel let this grid start, so it is read before the dependency wait. CTA (0, 0)
// waits even without a job: a grid that completes counts as done for its successors only
// once one of its CTAs has waited for the attention kernel.
__global__ void __launch_bounds__(32 * MERGE_ROWS) combine_sched_kernel(
    const float *o_part, const float *lse_part, const int4 *jobs, const int32_t *tile_start,
    int B, int P, int H, uint16_t *out, float *out_f32, float *lse) {
    const int h = blockIdx.x * MERGE_ROWS + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    grid_launch_dependents();
    if (blockIdx.y >= P) {  // empty sequences
        grid_dependency_wait();
        if (h >= H) return;
        const int j = blockIdx.y - P;
        for (int base = j; base < B; base += 32 * EMPTY_CTAS) {
            const int bq = base + EMPTY_CTAS * lane;
            const bool e = bq < B && tile_start[bq + 1] == tile_start[bq];
            for (unsigned m = __ballot_sync(0xffffffffu, e); m; m &= m - 1) {
                const size_t row = (size_t)(base + EMPTY_CTAS * (__ffs(m) - 1)) * H + h;
                if (out_f32) {
                    float4 *d = reinterpret_cast<float4 *>(out_f32 + row * D_C);
#pragma unroll
                    for (int k = 0; k < 4; ++k) d[lane + 32 * k] = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
                    uint4 *d = reinterpret_cast<uint4 *>(out + row * D_C);
                    d[lane] = d[lane + 32] = make_uint4(0u, 0u, 0u, 0u);
                }
                if (lane == 0) lse[row] = -INFINITY;
            }
        }
        return;
    }
    const int4 job = __ldcg(jobs + blockIdx.y);
    if ((job.x < 0 || h >= H) && (blockIdx.x | blockIdx.y) != 0) return;
    grid_dependency_wait();
    if (job.x < 0 || h >= H) return;
    const size_t row = (size_t)job.x * H + h;
    merge_row_warp(o_part + ((size_t)job.y * H + h) * D_C, (size_t)H * D_C,
                   lse_part + (size_t)job.y * H + h, H, job.z,
                   out_f32 ? nullptr : out + row * D_C, out_f32 ? out_f32 + row * D_C : nullptr,
                   lse + row, lane);
}

}  // namespace

cudaError_t launch_decode_schedule(const int32_t *seqlens, int B, int max_len, int P,
                                   int32_t *tile_start, int32_t *wpos, int32_t *part_begin,
                                   int32_t *nparts, int4 *jobs, uint32_t *err,
                                   cudaStream_t stream) {
    const size_t smem = 4 * sizeof(int) * (size_t)B;  // B <= 4096: at most 64 KB
    cudaError_t e = cudaFuncSetAttribute(decode_schedule_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 4 * 4 * 4096);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_schedule_kernel, dim3(1), dim3(1024), smem, stream, seqlens, B,
                      max_len, P, tile_start, wpos, part_begin, nparts, jobs, err);
}

cudaError_t launch_combine_sched(const float *o_part, const float *lse_part, const int4 *jobs,
                                 const int32_t *tile_start, int B, int P, int H, uint16_t *out,
                                 float *out_f32, float *lse, cudaStream_t stream) {
    dim3 grid((H + MERGE_ROWS - 1) / MERGE_ROWS, P + EMPTY_CTAS);
    return launch_pdl(combine_sched_kernel, grid, dim3(32 * MERGE_ROWS), 0, stream, o_part,
                      lse_part, jobs, tile_start, B, P, H, out, out_f32, lse);
}

cudaError_t launch_combine(const float *o_part, const float *lse_part, int B, int S, int H,
                           long o_bstride, long o_pstride, long l_bstride, long l_pstride,
                           uint16_t *out, float *out_f32, float *lse, cudaStream_t stream) {
    dim3 grid((H + MERGE_ROWS - 1) / MERGE_ROWS, B);
    return launch_pdl(combine_kernel, grid, dim3(32 * MERGE_ROWS), 0, stream, o_part, lse_part, S,
                      H, o_bstride, o_pstride, l_bstride, l_pstride, out, out_f32, lse);
}

cudaError_t launch_reduce_bf16(const float *part, int S, int batch, int M, int N, uint16_t *C,
                               long ldc, long c_bstride, cudaStream_t stream) {
    long pairs = (long)batch * M * N / 2;
    long nb = (pairs + 255) / 256;
    int blocks = (int)(nb < 4096 ? nb : 4096);
    return launch_pdl(reduce_partials_bf16, dim3(blocks), dim3(256), 0, stream, part, S, batch, M,
                      N, C, ldc, c_bstride);
}

}  // namespace mla
