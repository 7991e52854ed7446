// kernels.h -- internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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
    const uint16_t *cache;     // [num_blocks][64][576]
    const int32_t *block_table;
    const int32_t *seqlens;
    int num_blocks, max_blocks, B, H;  // H = query rows per sequence (s_q x hq)
    int s_q, hq;  // query tokens per sequence (draft tokens, causal among them), heads each
    int num_splits, tiles_per_split;
    float scale_log2;          // scale * log2(e)
    uint16_t *out;             // [B][H][512]  (written when num_splits == 1)
    float *lse;                // [B][H]       (written when num_splits == 1)
    float *o_part;             // [B][S][H][512] (num_splits > 1); [2P][H][512] if scheduled
    float *lse_part;           // [B][S][H]      (num_splits > 1); [2P][H]      if scheduled
    uint32_t *err;
    // Balanced schedule (num_splits == 0): P clusters each take an equal contiguous range
    // of the concatenated tile list; sequences cut between clusters become parts.
    const int32_t *tile_start;  // [B+1] exclusive prefix of tiles per sequence
    const int32_t *part_begin;  // [B]   first part index of a sequence that is cut
    const int32_t *nparts;      // [B]   number of parts (0 = whole in one cluster)
};

// The cluster (of P) whose tile range [c*T/P, (c+1)*T/P) holds global tile t.
__host__ __device__ inline int cluster_of_tile(long t, long T, int P) {
    long c = (t * P) / T;
    while (c + 1 < P && ((c + 1) * T) / P <= t) ++c;
    while (c > 0 && (c * T) / P > t) --c;
    return static_cast<int>(c);
}

cudaError_t launch_decode_schedule(const int32_t *seqlens, int B, int max_blocks, int P,
                                   int32_t *tile_start, int32_t *part_begin, int32_t *nparts,
                                   uint32_t *err, cudaStream_t stream);
cudaError_t launch_combine_sched(const float *o_part, const float *lse_part,
                                 const int32_t *tile_start, const int32_t *part_begin,
                                 const int32_t *nparts, int B, int H, uint16_t *out, float *lse,
                                 cudaStream_t stream);

// grid = `clusters` two-CTA clusters (one per work item, or P with the schedule)
cudaError_t launch_decode_tc(const DecodeParams &p, int clusters, cudaStream_t stream);
int decode_tc_cluster_slots();
cudaError_t launch_combine(const float *o_part, const float *lse_part, int B, int S, int H,
                           uint16_t *out, float *lse, cudaStream_t stream);

int device_sm_count();

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
