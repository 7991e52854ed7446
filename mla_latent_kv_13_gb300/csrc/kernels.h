// kernels.h -- internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mla.h"

namespace mla {

struct GemmParams {
    const uint16_t *A;  // [batch][M][K] via a_bstride / lda
    long lda, a_bstride;
    const uint16_t *B;  // TN: [N][K]; NN: [K][N]
    long ldb, b_bstride;
    int M, N, K, batch;
    int k_splits, k_per_split;  // k_per_split a multiple of 64
    float *c_part;              // if non-null: fp32 partials [k_splits][batch][M][N]
    uint16_t *c_bf16;           // else: bf16 C with ldc / c_bstride
    long ldc, c_bstride;
};

// tcgen05/TMA GEMM (one 128 x gemm_block_n(N, K) tile per CTA); err = workspace error word
cudaError_t launch_gemm_tc(const GemmParams &p, bool nn, cudaStream_t stream, uint32_t *err);
// Split-K whose k-splits of an output tile run as one thread-block cluster and reduce
// through its shared memory into bf16 C (TN, batch 1): gemm_cluster_plan gives the splits
// (and the K per split) for this shape on this device, 0 when none fits every tile in one
// wave, and the output-tile width (128, 224 or 256); launch_gemm_tc_cluster takes them in
// p.k_splits / p.k_per_split and block_n, p.c_part null.
// With `ap`, the product is append's h W_DKR^T (N = 576): row b is sequence b's new latent
// row, its k_rope pairs rotated at pos[b], written into the paged cache (C unused).
struct ClusterAppend {
    const int32_t *pos, *block_table;
    int max_blocks, num_blocks;
    uint16_t *cache;
    float theta;
};
int gemm_cluster_plan(int M, int N, int K, int *k_per_split, int *block_n);
// whether launch_gemm_tc_cluster_dq_append finds a cluster split for these shapes
bool gemm_cluster_fits_dq_append(int M, int N1, int K);
// c_q = A W_DQ^T (bf16 [M][N1]) and append's rows from A W_DKR^T in one cluster-reduced
// launch; cudaErrorNotSupported when no cluster split fits (run them separately then).
cudaError_t launch_gemm_tc_cluster_dq_append(const uint16_t *A, int M, int K, const uint16_t *B1,
                                            int N1, uint16_t *C1, const uint16_t *B2,
                                            const ClusterAppend &ap, cudaStream_t stream,
                                            uint32_t *err);
cudaError_t launch_gemm_tc_cluster(const GemmParams &p, int block_n, const ClusterAppend *ap,
                                   cudaStream_t stream, uint32_t *err);
// C1 = A B1^T and C2 = RoPE(A B2^T) (64-column heads rotated pairwise at pos[row]) in one
// launch; bf16 everywhere, N1 and N2 multiples of 64, M <= 128
cudaError_t launch_gemm_tc_rope(const uint16_t *A, int M, int K, const uint16_t *B1, int N1,
                                uint16_t *C1, const uint16_t *B2, int N2, uint16_t *C2,
                                const int32_t *pos, float theta, cudaStream_t stream,
                                uint32_t *err);
int gemm_block_n(int N, int K);  // output-tile width the GEMM uses (128 or 256)
int gemm_block_n(int M, int N, int K);
cudaError_t launch_reduce_bf16(const float *part, int S, int batch, int M, int N, uint16_t *C,
                               long ldc, long c_bstride, cudaStream_t stream);

// Append: reduce split partials of x = h W_DKR^T, RoPE the last 64, round, scatter.
cudaError_t launch_append_finalize(const float *part, int S, int B, const int32_t *pos,
                                   const int32_t *block_table, int max_blocks, uint16_t *cache,
                                   int num_blocks, float theta, uint32_t *err,
                                   cudaStream_t stream);

// Query side: reduce partials of c_q W_QR^T, RoPE per head, write bf16 q_rope.
cudaError_t launch_qrope_finalize(const float *part, int S, int B, int H, const int32_t *pos,
                                  float theta, uint16_t *q_rope, cudaStream_t stream);

struct DecodeParams {
    const uint16_t *q_lat;     // [B][H][512]
    const uint16_t *q_rope;    // [B][H][64]
    const uint16_t *cache;     // [num_blocks][64][576] bf16 (when codes is null)
    const uint8_t *codes;      // FP8 cache: e4m3 codes [num_blocks][64][576], or null
    const int8_t *exps;        // FP8 cache: row exponents [num_blocks][64] (scale 2^e)
    const int32_t *block_table;
    const int32_t *seqlens;
    int num_blocks, max_blocks, B, H;  // H = query rows per sequence (s_q x hq)
    int max_seqlen;            // caller's bound on seqlens (<= 64 * max_blocks)
    int s_q, hq;  // query tokens per sequence (draft tokens, causal among them), heads each
    int num_splits, tiles_per_split;
    float scale_log2;          // scale * log2(e)
    uint16_t *out;             // [B][H][512]  (written when num_splits == 1)
    float *out_f32;            // if non-null: the output as fp32 [B][H][512] instead of out
    float *lse;                // [B][H]       (written when num_splits == 1)
    float *o_part;             // [B][S][H][512] (num_splits > 1); [2P][H][512] if scheduled
    float *lse_part;           // [B][S][H]      (num_splits > 1); [2P][H]      if scheduled
    uint32_t *err;
    // Balanced schedule (num_splits == 0): P clusters each take an equal contiguous range
    // of the weighted tile list; sequences cut between clusters become parts.
    const int32_t *tile_start;  // [B+1] exclusive prefix of tiles per sequence
    const int32_t *wpos;        // [B+1] weight position of each sequence's first tile; [B] = W
    const int32_t *part_begin;  // [B]   first part index of a sequence that is cut
    const int32_t *nparts;      // [B]   number of parts (0 = whole in one cluster)
};

// Balanced schedule. A sequence with v > 0 tiles weighs SEG_COST + v: a segment (the
// piece of one sequence that one cluster processes) costs about as much to start and to
// finish -- Q rows loaded, rings filled, the output rows written -- as SEG_COST tiles of
// the steady loop. With the weights laid end to end, sequence b owns the weight range
// [wpos[b] - SEG_COST, wpos[b] + v): its start-up first, then one position per tile.
// Cluster c of P takes the weight range [c*W/P, (c+1)*W/P) (W = total weight) and
// processes the tiles that fall inside it, so a cluster that starts many short sequences
// gets fewer tiles than one that streams a long one.
constexpr int SEG_COST = 12;

// The cluster (of P) whose range [c*W/P, (c+1)*W/P) holds weight position t.
__host__ __device__ inline int cluster_of_tile(long t, long W, int P) {
    long c = (t * P) / W;
    while (c + 1 < P && ((c + 1) * W) / P <= t) ++c;
    while (c > 0 && (c * W) / P > t) --c;
    return static_cast<int>(c);
}

// One segment of a cluster's share: tiles [t_begin, t_end) of sequence b, written straight
// to the output (direct) or as fp32 part `part` of a sequence cut between clusters.
struct SchedSegment {
    int b, t_begin, t_end, part;
    bool direct;
};

// Largest b with wpos[b] <= r0 (the first sequence that may have tiles in [r0, r1)).
__host__ __device__ inline int sched_first(const int32_t *wpos, int B, long r0) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (wpos[mid] <= r0) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The next segment of cluster cl (range [r0, r1) of W, P ranges) at or after sequence
// *cursor, which advances past it; false when the share has no further tiles.
__host__ __device__ inline bool sched_next(const int32_t *tile_start, const int32_t *wpos,
                                           const int32_t *part_begin, int B, long r0, long r1,
                                           long W, int P, int cl, int *cursor,
                                           SchedSegment *s) {
    int b = *cursor;
    while (b < B) {  // skip empty sequences and one whose tiles end before the range
        const int v = tile_start[b + 1] - tile_start[b];
        if (v > 0 && wpos[b] + v > r0) break;
        ++b;
    }
    if (b >= B || wpos[b] >= r1 || r0 >= r1) {
        *cursor = b;
        return false;
    }
    *cursor = b + 1;
    const long ws = wpos[b], we = ws + (tile_start[b + 1] - tile_start[b]);
    s->b = b;
    s->t_begin = static_cast<int>((r0 > ws ? r0 : ws) - ws);
    s->t_end = static_cast<int>((r1 < we ? r1 : we) - ws);
    s->direct = ws >= r0 && we <= r1;
    s->part = s->direct ? 0 : part_begin[b] + (cl - cluster_of_tile(ws, W, P));
    return true;
}

// The first sequence at or after b with tiles, if its first tile lies before r1; else -1.
__host__ __device__ inline int sched_peek(const int32_t *tile_start, const int32_t *wpos, int B,
                                          long r1, int b) {
    while (b < B && tile_start[b + 1] == tile_start[b]) ++b;
    return b < B && wpos[b] < r1 ? b : -1;
}

// seqlens outside [0, max_len] are recorded as MLA_ERR_OUT_OF_RANGE and clamped to it.
// Also lists the merge jobs (jobs [P]: (sequence, first part, parts) of the sequence cut at
// the end of cluster c's range, or (-1, 0, 0)).
cudaError_t launch_decode_schedule(const int32_t *seqlens, int B, int max_len, int P,
                                   int32_t *tile_start, int32_t *wpos, int32_t *part_begin,
                                   int32_t *nparts, int4 *jobs, uint32_t *err,
                                   cudaStream_t stream);
// Merges the jobs' parts and writes the sequences without tiles (out = 0, lse = -inf);
// out_f32 (if non-null) receives the rows as fp32 instead of out
cudaError_t launch_combine_sched(const float *o_part, const float *lse_part, const int4 *jobs,
                                 const int32_t *tile_start, int B, int P, int H, uint16_t *out,
                                 float *out_f32, float *lse, cudaStream_t stream);

// grid = `clusters` two-CTA clusters (one per work item, or P with the schedule)
cudaError_t launch_decode_tc(const DecodeParams &p, int clusters, cudaStream_t stream);
int decode_tc_cluster_slots();
// Merge S parts per (b, h) row: part s of row (b, h) at o_part + b*o_bstride + s*o_pstride
// + h*512 (lse_part likewise with l_bstride, l_pstride, + h); out / out_f32 as above.
cudaError_t launch_combine(const float *o_part, const float *lse_part, int B, int S, int H,
                           long o_bstride, long o_pstride, long l_bstride, long l_pstride,
                           uint16_t *out, float *out_f32, float *lse, cudaStream_t stream);

int device_sm_count();

// FP8 (e4m3) cache rows of 576 values, one power-of-two scale per row.
cudaError_t launch_quantize_rows(const uint16_t *src, long rows, uint8_t *codes, int8_t *exps,
                                 cudaStream_t stream);
cudaError_t launch_dequantize_rows(const uint8_t *codes, const int8_t *exps, long rows,
                                   uint16_t *dst, cudaStream_t stream);
cudaError_t launch_append_finalize_fp8(const float *part, int S, int B, const int32_t *pos,
                                       const int32_t *block_table, int max_blocks,
                                       uint8_t *codes, int8_t *exps, int num_blocks,
                                       float theta, uint32_t *err, cudaStream_t stream);

// Host-side argument checks of a decode call (all but the workspace): MLA_OK or the
// status the entry point returns. Launches nothing.
mla_status_t decode_validate(const void *q_lat, const void *q_rope, const void *kv_cache,
                             int num_blocks, const int32_t *block_table, int max_blocks,
                             const int32_t *seqlens, int B, int s_q, int hq, int max_seqlen,
                             float scale, int num_splits, const void *out, const float *lse);

// Chunked prefill: gather one sequence's first T cache rows contiguous (c_kv, k_rope), then
// causal attention of the C chunk queries in the expanded form.
cudaError_t launch_gather_rows(const uint16_t *cache, int num_blocks, const int32_t *block_table,
                               int max_blocks, int T, uint16_t *ckv, uint16_t *kr, uint32_t *err,
                               cudaStream_t stream);
cudaError_t launch_prefill_tc(const uint16_t *q_nope, const uint16_t *q_rope,
                              const uint16_t *k_nope, const uint16_t *k_rope, const uint16_t *v,
                              int C, int T, int H, int prefix, float scale, uint16_t *out,
                              float *lse, uint32_t *err, cudaStream_t stream);

// One CTA waits on a barrier nothing completes; records MLA_ERR_TIMEOUT after limit_ns.
cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, uint32_t *err, cudaStream_t stream);

}  // namespace mla
