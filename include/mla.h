/*
 * mla.h -- C ABI of libmla: Multi-head Latent Attention (MLA) decode over a
 * paged, compressed latent KV cache, with the up-projections absorbed.
 *
 * Sources (web pages, cited by address and section):
 *   [V2] sheratonhq.com/news/191949 "DeepSeek-V2 teardown: how MLA and MoE cut
 *        the KV cache by 93.3%", section 2.1 -- only the low-rank latent c_t is
 *        cached; W_UK is absorbed into the query projection and W_UV into the
 *        output projection; queries are low-rank compressed too; a separate
 *        decoupled-RoPE branch carries position.
 *   [MW] zskr.cn/news/1409628 "from the memory wall to the compute wall",
 *        section 2.1 (hidden 7168 -> latent 512; scores = (Q W_DK^T) CKV^T;
 *        decoupled RoPE), 2.2 (reorder the products by associativity), 2.3 (all
 *        heads share the compressed cache), 4.2 (fuse Q generation with W_DK).
 *   [V3] fsdata.site/2026/11/deepseek-v3-mla-optimization, section 1 (paged
 *        storage of the latent; on-the-fly back projection).
 *
 * Conventions shared by every call:
 *   - bf16 values are passed as uint16_t bit patterns (mla_bf16_t).
 *   - Every tensor argument is a DEVICE pointer to caller-owned, contiguous,
 *     row-major memory, unless stated otherwise. The library never allocates,
 *     frees or retains device memory; it keeps no state between calls.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream), on the device current for the calling thread.
 *   - Arguments are validated on the host first: a bad argument returns an error
 *     code and launches nothing.
 *   - Conditions only the GPU can see (a block-table entry outside the pool for
 *     a token that is read or written, a position beyond the block table) set a
 *     sticky error word in the caller's workspace; the affected token is skipped
 *     (reads are treated as masked, writes are dropped), nothing traps. Read the
 *     word with mla_check_device_status().
 *   - A workspace is caller-owned device memory of at least the size the
 *     matching *_workspace_size() call reports, aligned to 256 bytes. Its first
 *     256 bytes hold the error word; clear it once with mla_clear_device_status()
 *     before first use. One workspace may serve consecutive calls on one stream;
 *     calls that overlap on the GPU must not share one.
 *
 * Fixed dimensions (the only ones the kernels are built for):
 *   d_c = 512 latent, d_rope = 64 decoupled-RoPE key, 576 cached values per
 *   token, 64 tokens per cache block, d_nope = d_v = 128 per head.
 * Cache layout: kv_cache[num_blocks][64][576] bf16; row = [c_kv (512) | k_rope (64)],
 *   k_rope stored already rotated to the token's position.
 * Block table: block_table[B][max_blocks] int32; token t of sequence b lives in
 *   block block_table[b][t / 64], slot t % 64. Entries past a sequence's last
 *   block are never read and may hold any value.
 * RoPE: pairs (2i, 2i+1) of a 64-vector turn by pos * rope_theta^(-2i/64)
 *   radians; pos is the 0-based token index within its sequence.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t mla_bf16_t;
typedef void *mla_stream_t; /* cudaStream_t */

#define MLA_D_C 512
#define MLA_D_ROPE 64
#define MLA_D_QK 576
#define MLA_BLOCK 64
#define MLA_D_NOPE 128
#define MLA_D_V 128
#define MLA_WS_HEADER_BYTES 256

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer         */
    MLA_ERR_UNSUPPORTED = 2,  /* shape outside what the kernels are built for       */
    MLA_ERR_WORKSPACE = 3,    /* workspace smaller than the *_workspace_size figure */
    MLA_ERR_OUT_OF_RANGE = 4, /* device-detected: block id or position out of range */
    MLA_ERR_TIMEOUT = 5,      /* device-detected: a bounded wait gave up            */
    MLA_ERR_CUDA = 6          /* a CUDA runtime call failed (launch, sync)          */
} mla_status_t;

/* Human-readable name of a status code (static storage). */
const char *mla_status_string(mla_status_t status);

/* ---------------------------------------------------------------- append */

/*
 * [V2] 2.1, [MW] 2.1: write one new token per sequence into the latent cache.
 *   x = h[b] . W_DKR^T                (d_model -> 576, fp32 accumulation)
 *   c_kv = x[0:512]; k_rope = RoPE(x[512:576], pos[b])
 *   kv_cache[block_table[b][pos[b]/64]][pos[b]%64] = bf16([c_kv | k_rope])  (nearest-even)
 *
 * h       [B][d_model] bf16            w_dkr [576][d_model] bf16 (rows 0..511 = W_DKV,
 * pos     [B] int32 (slot to write)                                rows 512..575 = W_KR)
 * The caller advances its own sequence lengths after the append (pos is usually
 * the length before it). Requires 1 <= B <= 4096, d_model a multiple of 64.
 * Workspace: mla_append_kv_workspace_size(B, d_model).
 */
mla_status_t mla_append_kv_workspace_size(int B, int d_model, size_t *bytes);
mla_status_t mla_append_kv(const mla_bf16_t *h, int B, int d_model, const mla_bf16_t *w_dkr,
                           const int32_t *pos, const int32_t *block_table, int max_blocks,
                           mla_bf16_t *kv_cache, int num_blocks, float rope_theta,
                           void *workspace, size_t ws_bytes, mla_stream_t stream);

/* ------------------------------------------------------- decode attention */

/*
 * [V2] 2.1, [MW] 2.1-2.3: absorbed decode attention. For every sequence b and
 * head h, over the tokens j < seqlens[b] of the paged cache:
 *   s_j   = scale * (q_lat[b][h] . c_kv_j + q_rope[b][h] . k_rope_j)
 *   out   = sum_j softmax(s)_j c_kv_j     (the latent output; W_UV is applied later)
 *   lse   = ln sum_j exp(s_j)             (natural log, fp32)
 * seqlens[b] = 0 gives out = 0 and lse = -inf.
 *
 * q_lat [B][H][512] bf16, q_rope [B][H][64] bf16 (already rotated),
 * seqlens [B] int32 with 0 <= seqlens[b] <= max_seqlen (checked on the device: a length
 * outside that range is recorded as MLA_ERR_OUT_OF_RANGE and clamped into it, by every
 * work distribution alike),
 * out [B][H][512] bf16 (32-byte aligned: its rows are written with 32-byte stores),
 * lse [B][H] fp32.
 * scale must be finite and > 0 (1/sqrt(d_nope + d_rope) for DeepSeek-shaped heads).
 * H must be 16, 32, 64 or 128; 1 <= B <= 4096. num_splits: the number of equal token
 * ranges each sequence is cut into (1..256), merged exactly by their log-sum-exps
 * (split-KV combine); 0 = chosen by the library: such a fixed split when it fits the
 * GPU in one pass, else a balanced schedule (the concatenated token blocks of all
 * sequences, each sequence weighted with a fixed start-up cost, cut into one equal
 * share of the weight per resident work unit; sequences cut between shares merged the
 * same way; mla_decode_schedule shows the shares).
 * Workspace: mla_decode_workspace_size(B, H, max_seqlen, num_splits) with the
 * same B, H and num_splits; max_seqlen is an upper bound of seqlens.
 */
mla_status_t mla_decode_workspace_size(int B, int H, int max_seqlen, int num_splits,
                                       size_t *bytes);
/*
 * The plan mla_decode_attention takes for these arguments (no counterpart on the pages:
 * a query of this library's launch plan). *splits = the fixed number of token ranges
 * per sequence (1 = no merge), or 0 for the balanced schedule; *launches = the kernels
 * one call launches (1, 2 with a merge, 3 with the schedule). The plan depends on the
 * device's resident-cluster count, read as mla_decode_workspace_size reads it (a default
 * when no device is visible). Either output pointer may be null.
 */
mla_status_t mla_decode_plan(int B, int H, int max_seqlen, int num_splits, int *splits,
                             int *launches);
/*
 * The balanced schedule for these sequence lengths, computed on the host with the
 * arithmetic the device uses (no counterpart on the pages; no device memory is touched).
 * seqlens [B] host int32, clamped to [0, 64 * max_blocks] (the device clamps to
 * [0, max_seqlen] of its call, which is at most that, and records an error); clusters =
 * the number of work units (the device's resident count in mla_decode_attention; any
 * value >= 1 here). A sequence with v > 0 token blocks weighs v plus a fixed start-up
 * cost; work unit c takes the weight range [c*W/P, (c+1)*W/P) of the total W
 * (P = min(clusters, W)) and the token blocks inside it. Writes the first `capacity`
 * segments as 5 int32 each: (work unit, sequence, first block, end block, part index or
 * -1 when the unit writes the sequence's output itself), in work-unit order;
 * *count = the number of segments (it may exceed capacity; nothing past capacity is
 * written); *parts (may be null) = the number of fp32 parts merged afterwards.
 * MLA_ERR_INVALID_ARG on null pointers, B outside 1..4096, max_blocks < 1, clusters < 1.
 */
mla_status_t mla_decode_schedule(const int32_t *seqlens, int B, int max_blocks, int clusters,
                                 int32_t *segs, int capacity, int *count, int *parts);
mla_status_t mla_decode_attention(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                                  const mla_bf16_t *kv_cache, int num_blocks,
                                  const int32_t *block_table, int max_blocks,
                                  const int32_t *seqlens, int B, int H, int max_seqlen,
                                  float scale, int num_splits, void *workspace,
                                  size_t ws_bytes, mla_bf16_t *out, float *lse,
                                  mla_stream_t stream);
/*
 * The balanced schedule of mla_decode_attention computed ahead of the call (no counterpart
 * on the pages: it depends only on the sequence lengths, so a decode step computes it once
 * for every layer, on the attention's stream or another one).
 * Writes the schedule into the workspace: the same workspace layout, the same arguments
 * (B, H, max_seqlen, num_splits) as the attention calls that use it; does nothing when the
 * plan for them is a fixed split. seqlens [B] device int32 as in mla_decode_attention
 * (lengths outside [0, max_seqlen] are recorded and clamped here). The workspace's first
 * 256 bytes (the error word) must be zero as for mla_decode_attention.
 * The schedule kernel reads seqlens before it waits for its predecessor in the stream (it
 * stores nothing until then), so it runs beside that kernel: seqlens must not be written by
 * a kernel that lets its successors start before it completes (programmatic dependent
 * launch); no kernel of this library writes it, and a kernel without that opt-in completes
 * before this one starts. The same holds for mla_decode_attention's own schedule launch.
 * MLA_ERR_INVALID_ARG / MLA_ERR_UNSUPPORTED / MLA_ERR_WORKSPACE as mla_decode_attention.
 */
mla_status_t mla_decode_prepare(const int32_t *seqlens, int B, int H, int max_seqlen,
                                int num_splits, void *workspace, size_t ws_bytes,
                                mla_stream_t stream);
/*
 * mla_decode_attention over a workspace that mla_decode_prepare filled for the same seqlens
 * (unchanged since), B, H, max_seqlen and num_splits: the same outputs, bit for bit, without
 * the schedule launch. The prepare call's kernel must be complete before this call's kernels
 * start (the same stream, or an event the caller waits for). A workspace not prepared for
 * these arguments gives undefined results.
 */
mla_status_t mla_decode_attention_prepared(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                                           const mla_bf16_t *kv_cache, int num_blocks,
                                           const int32_t *block_table, int max_blocks,
                                           const int32_t *seqlens, int B, int H, int max_seqlen,
                                           float scale, int num_splits, void *workspace,
                                           size_t ws_bytes, mla_bf16_t *out, float *lse,
                                           mla_stream_t stream);

/*
 * Decode attention for s_q query tokens per sequence: the draft tokens a main model
 * verifies in one pass ("When MoE meets MLA" §5.3 item 3, "DeepSeek V3 MoE inference"
 * §6). The draft tokens' own cache rows are the last s_q of the seqlens[b] rows already
 * in the cache, and draft token t (0-based) attends causally, to the rows
 * j < seqlens[b] - (s_q - 1 - t); a token that sees no row gets out = 0, lse = -inf.
 * Otherwise as mla_decode_attention, with the query rows of a sequence ordered
 * (token, head): q_lat [B][s_q][H][512], q_rope [B][s_q][H][64] bf16,
 * out [B][s_q][H][512] bf16, lse [B][s_q][H] fp32. H must be 16, 32, 64 or 128 with
 * s_q * H <= 128 (MLA_ERR_UNSUPPORTED otherwise); s_q >= 1. s_q = 1 is exactly
 * mla_decode_attention. Workspace: mla_decode_mq_workspace_size with the same B, s_q, H
 * and num_splits.
 */
mla_status_t mla_decode_mq_workspace_size(int B, int s_q, int H, int max_seqlen, int num_splits,
                                          size_t *bytes);
mla_status_t mla_decode_attention_mq(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                                     const mla_bf16_t *kv_cache, int num_blocks,
                                     const int32_t *block_table, int max_blocks,
                                     const int32_t *seqlens, int B, int s_q, int H,
                                     int max_seqlen, float scale, int num_splits, void *workspace,
                                     size_t ws_bytes, mla_bf16_t *out, float *lse,
                                     mla_stream_t stream);

/*
 * "LLM inference: from the memory wall to the compute wall" §2.2: chunked prefill of one
 * sequence in the expanded (un-absorbed) form. The chunk's tokens must already be in the
 * cache, at positions prefix .. prefix + chunk - 1 (mla_append_kv); the cached latent rows of
 * positions 0 .. prefix + chunk - 1 are projected back per head,
 *   k_nope_j = W_UK[h] c_kv_j (128),  v_j = W_UV[h] c_kv_j (128),  k_rope_j shared,
 * (kept bf16), and query i of the chunk attends causally to the positions j <= prefix + i:
 *   s_j = scale * (q_nope[i][h] . k_nope_j + q_rope[i][h] . k_rope_j),
 *   out[i][h] = sum_j softmax(s)_j v_j,  lse[i][h] = ln sum_j exp(s_j).
 * q_nope [chunk][H][128], q_rope [chunk][H][64] bf16 (rotated at their positions);
 * block_table [max_blocks] int32 of this sequence (ids checked on the device);
 * w_uk, w_uv [H][128][512] bf16; out [chunk][H][128] bf16, lse [chunk][H] fp32.
 * H must be 16, 32, 64 or 128; prefix >= 0, chunk >= 1, prefix + chunk <= 64 * max_blocks.
 * Workspace: mla_prefill_workspace_size(H, prefix, chunk) (it holds the projected K and V:
 * about 512 * H bytes per position).
 */
mla_status_t mla_prefill_workspace_size(int H, int prefix, int chunk, size_t *bytes);
mla_status_t mla_prefill_attention(const mla_bf16_t *q_nope, const mla_bf16_t *q_rope,
                                   const mla_bf16_t *kv_cache, int num_blocks,
                                   const int32_t *block_table, int max_blocks, int prefix,
                                   int chunk, int H, const mla_bf16_t *w_uk,
                                   const mla_bf16_t *w_uv, float scale, void *workspace,
                                   size_t ws_bytes, mla_bf16_t *out, float *lse,
                                   mla_stream_t stream);

/*
 * Failure-detection self-test (no counterpart on the pages: a check of this library).
 * Launches one CTA that waits, with the bounded mbarrier wait every kernel of the library
 * uses, on a barrier that nothing completes; after limit_us microseconds (1..1000000) the
 * wait gives up and MLA_ERR_TIMEOUT is recorded in the workspace error word (detail = the
 * microseconds waited), to be read with mla_check_device_status. Nothing faults and the
 * context stays usable. workspace: at least the 256-byte header, 256-byte aligned.
 */
mla_status_t mla_selftest_wait_timeout(unsigned limit_us, void *workspace, size_t ws_bytes,
                                       mla_stream_t stream);

/*
 * The split-KV merge on its own (the last step of mla_decode_attention):
 *   lse[b][h] = ln sum_s exp(lse_part[b][s][h]);
 *   out[b][h] = sum_s exp(lse_part[b][s][h] - lse[b][h]) * o_part[b][s][h]
 * Parts with lse_part = -inf weigh zero; all-empty gives out = 0, lse = -inf.
 * o_part [B][S][H][512] fp32 (each part already normalised), lse_part [B][S][H] fp32,
 * out [B][H][512] bf16, lse [B][H] fp32. Needs no workspace.
 */
mla_status_t mla_decode_combine(const float *o_part, const float *lse_part, int B, int S, int H,
                                mla_bf16_t *out, float *lse, mla_stream_t stream);

/*
 * Context-parallel decode, one rank's share ("DeepSeek V3 MoE inference" §3: decode attention
 * deployed as TP4 + SP4 + DP; "from the memory wall to the compute wall" §2.3: every head
 * reads the same compressed cache, so splitting heads does not split the bytes, splitting
 * tokens does). The cached tokens of each sequence are spread over G ranks by token range
 * (each rank holds its range's rows in its own paged cache; k_rope is stored rotated at each
 * row's absolute position, so scores do not depend on which rank holds a row). Each rank
 * calls this with its own cache, block table and seqlens (the lengths of its ranges) and
 * gets, per (b, h), the attention over its range alone, normalised, in fp32, with its
 * log-sum-exp:
 *   o_part[b][h] = sum_{j in range} softmax_range(s)_j c_kv_j,  lse_part[b][h] = ln sum exp(s_j)
 * (an empty range gives o_part = 0, lse_part = -inf). The ranks then exchange
 * (o_part, lse_part) -- an all-gather, outside this library -- and mla_decode_combine_ranks
 * merges them exactly. Arguments, checks, workspace and plans as mla_decode_attention;
 * o_part [B][H][512] fp32 (32-byte aligned), lse_part [B][H] fp32.
 */
mla_status_t mla_decode_attention_partial(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                                          const mla_bf16_t *kv_cache, int num_blocks,
                                          const int32_t *block_table, int max_blocks,
                                          const int32_t *seqlens, int B, int H, int max_seqlen,
                                          float scale, int num_splits, void *workspace,
                                          size_t ws_bytes, float *o_part, float *lse_part,
                                          mla_stream_t stream);

/*
 * The merge of G context-parallel ranks' partial results (the same exact log-sum-exp merge as
 * mla_decode_combine, with the parts laid out by rank, as an all-gather leaves them):
 *   lse[b][h] = ln sum_g exp(lse_parts[g][b][h]);
 *   out[b][h] = sum_g exp(lse_parts[g][b][h] - lse[b][h]) * o_parts[g][b][h]
 * o_parts [G][B][H][512] fp32, lse_parts [G][B][H] fp32 -> out [B][H][512] bf16,
 * lse [B][H] fp32. Ranges with lse = -inf weigh zero; all-empty gives out = 0, lse = -inf.
 * Needs no workspace. 1 <= G <= 4096, 1 <= B <= 4096.
 */
mla_status_t mla_decode_combine_ranks(const float *o_parts, const float *lse_parts, int G, int B,
                                      int H, mla_bf16_t *out, float *lse, mla_stream_t stream);

/*
 * mla_decode_attention without a workspace: the same computation and outputs, for
 * callers that cannot obtain device memory for scratch -- code running while a
 * stream is captured into a CUDA graph (an allocation there is illegal or ends the
 * capture), plugins whose host framework owns every device allocation and hands out
 * only tensor pointers, serving loops that must not call cudaMalloc/cudaFree on their
 * hot path because those calls can synchronise the device. (The pages describe no such
 * entry point; it is a property of this library.)
 *
 * The split-KV scratch (partial outputs, their log-sum-exps, the schedule's offsets and
 * the error word) lives in one array of MLA_NOALLOC_SCRATCH_BYTES (40 MiB) that is part
 * of the library image: every GPU that loads the library holds it until the process
 * exits. A request fits when the figure mla_decode_workspace_size reports for the same
 * B, H, max_seqlen and num_splits is at most that size. With num_splits = 0 every plan
 * of up to 128 query rows fits on a GPU with at most 76 resident work units (a GB300):
 * the largest is the balanced schedule's 152 partial rows of 128 heads, 38.1 MiB (for
 * instance B = 128 sequences of 8192 tokens). num_splits = 1 needs no partials and always
 * fits; explicit splits fit while B * num_splits * H * 2 KiB stays below the limit.
 * Larger requests, and every invalid argument, are rejected on the host before anything
 * is queued (MLA_ERR_WORKSPACE, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED).
 * The first call on a device looks up the array's device address (no allocation) and
 * should happen before any stream capture. All calls share the array and it keeps the
 * last call's contents (each call clears the error word it needs), so calls that overlap
 * on the GPU (other streams, other host threads) race and must be serialised by the
 * caller. Device-detected range errors skip the offending tokens as in
 * mla_decode_attention but are not reported (there is no workspace to read them from).
 * Allocates nothing.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (40u << 20)
mla_status_t mla_decode_attention_noalloc(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                                          const mla_bf16_t *kv_cache, int num_blocks,
                                          const int32_t *block_table, int max_blocks,
                                          const int32_t *seqlens, int B, int H, int max_seqlen,
                                          float scale, int num_splits, mla_bf16_t *out,
                                          float *lse, mla_stream_t stream);

/* ------------------------------------------------------ FP8 latent cache */

/*
 * FP8 (e4m3) latent cache ("LLM inference: from the memory wall to the compute wall" §5:
 * a mixed-precision FP8/FP16 KV cache; "DeepSeek V3 MLA optimisation" §3: FP8 quantisation
 * of the KV cache). The pages fix no format; this library's format:
 *   kv_codes [num_blocks][64][576] uint8: e4m3 codes (1 sign, 4 exponent bits with bias
 *     7, 3 mantissa bits; largest finite 448; no infinities) of the row divided by its
 *     scale, rounded to nearest with ties to even, saturating at 448;
 *   kv_exps [num_blocks][64] int8: per cached row (one token) the exponent e of its scale
 *     2^e, the smallest with max|x| * 2^-e <= 448 (0 for an all-zero row; at least -126).
 * A row's dequantised values are code * 2^e, which are exactly bf16 values, so attention
 * over an FP8 cache equals attention over that dequantised cache. Half the cache bytes
 * of bf16 (plus one byte per token). Both arrays: device memory, 16-byte aligned.
 */

/* rows x 576 bf16 values -> codes [rows][576] and exps [rows]. Asynchronous. */
mla_status_t mla_quantize_kv_fp8(const mla_bf16_t *rows_bf16, long rows, uint8_t *codes,
                                 int8_t *exps, mla_stream_t stream);
/* codes [rows][576] and exps [rows] -> the dequantised rows as bf16 (exact). */
mla_status_t mla_dequantize_kv_fp8(const uint8_t *codes, const int8_t *exps, long rows,
                                   mla_bf16_t *rows_bf16, mla_stream_t stream);
/* mla_append_kv into an FP8 cache: the projected, rotated row is quantised (from fp32)
 * into kv_codes / kv_exps at slot pos[b]. Same arguments and workspace as
 * mla_append_kv otherwise. */
mla_status_t mla_append_kv_fp8(const mla_bf16_t *h, int B, int d_model, const mla_bf16_t *w_dkr,
                               const int32_t *pos, const int32_t *block_table, int max_blocks,
                               uint8_t *kv_codes, int8_t *kv_exps, int num_blocks,
                               float rope_theta, void *workspace, size_t ws_bytes,
                               mla_stream_t stream);
/* mla_decode_attention over an FP8 cache (the same arguments, checks, workspace --
 * mla_decode_workspace_size -- and plans; the cache tiles are widened to bf16 on chip). */
mla_status_t mla_decode_attention_fp8(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                                      const uint8_t *kv_codes, const int8_t *kv_exps,
                                      int num_blocks, const int32_t *block_table, int max_blocks,
                                      const int32_t *seqlens, int B, int H, int max_seqlen,
                                      float scale, int num_splits, void *workspace,
                                      size_t ws_bytes, mla_bf16_t *out, float *lse,
                                      mla_stream_t stream);

/* ------------------------------------------------- absorbed projections */

/*
 * [V2] 2.1 (query compression, decoupled RoPE, W_UK absorbed into the query),
 * [MW] 2.2 and 4.2 (Q times W_DK first; fuse query generation with W_DK):
 *   c_q       = h . W_DQ^T                      (d_model -> q_lora)
 *   q_nope_i  = c_q . W_UQ_i^T                  (q_lora -> 128, head i)
 *   q_rope_i  = RoPE(c_q . W_QR_i^T, pos[b])    (q_lora -> 64, head i)
 *   q_lat_i   = q_nope_i . W_UK_i               (128 -> 512, head i)
 * Intermediates (c_q, q_nope) are kept as bf16 between the products.
 *
 * h [B][d_model]; w_dq [q_lora][d_model]; w_uq [H*128][q_lora]; w_qr [H*64][q_lora];
 * w_uk [H][128][512] (W_UK_i maps a latent to head i's key: k = W_UK_i c);
 * pos [B] int32 -> q_lat [B][H][512] bf16, q_rope [B][H][64] bf16.
 * Requires d_model and q_lora multiples of 64, H in {16, 32, 64, 128}, 1 <= B <= 4096.
 */
mla_status_t mla_absorb_q_workspace_size(int B, int d_model, int q_lora, int H, size_t *bytes);
mla_status_t mla_absorb_q(const mla_bf16_t *h, int B, int d_model, const mla_bf16_t *w_dq,
                          int q_lora, const mla_bf16_t *w_uq, const mla_bf16_t *w_qr,
                          const mla_bf16_t *w_uk, int H, const int32_t *pos, float rope_theta,
                          void *workspace, size_t ws_bytes, mla_bf16_t *q_lat,
                          mla_bf16_t *q_rope, mla_stream_t stream);

/*
 * mla_append_kv and mla_absorb_q in one call (no counterpart on the pages: both
 * down-projections of a decode step read the same hidden states h, [V2] 2.1). Results equal
 * those of the two calls (the same arithmetic, up to the order of the fp32 split sums): the
 * new latent rows written into the paged cache as mla_append_kv writes them, q_lat and q_rope
 * as mla_absorb_q returns them. h W_DQ^T and h W_DKR^T run as one GEMM launch whose k-splits
 * are reduced inside thread-block clusters; where no cluster split fits the device, the call
 * runs the two entry points one after the other. Arguments as there (the append's first,
 * then the query's; one rope_theta for both); the checks of both apply. Workspace:
 * mla_append_absorb_q_workspace_size (the larger of the two calls' workspaces).
 */
mla_status_t mla_append_absorb_q_workspace_size(int B, int d_model, int q_lora, int H,
                                                size_t *bytes);
mla_status_t mla_append_absorb_q(const mla_bf16_t *h, int B, int d_model, const mla_bf16_t *w_dkr,
                                 const int32_t *pos, const int32_t *block_table, int max_blocks,
                                 mla_bf16_t *kv_cache, int num_blocks, const mla_bf16_t *w_dq,
                                 int q_lora, const mla_bf16_t *w_uq, const mla_bf16_t *w_qr,
                                 const mla_bf16_t *w_uk, int H, float rope_theta, void *workspace,
                                 size_t ws_bytes, mla_bf16_t *q_lat, mla_bf16_t *q_rope,
                                 mla_stream_t stream);

/*
 * [V2] 2.1 (W_UV absorbed into the output projection):
 *   o_v_i = W_UV_i . o_lat_i    (512 -> 128, head i)
 *   y     = [o_v_1 | ... | o_v_H] . W_O^T        (H*128 -> d_model)
 * o_lat [B][H][512] bf16; w_uv [H][128][512]; w_o [d_model][H*128] -> y [B][d_model] bf16.
 * o_v is kept as bf16 between the products. Requires d_model a multiple of 64.
 */
mla_status_t mla_out_absorb_workspace_size(int B, int H, int d_model, size_t *bytes);
mla_status_t mla_out_absorb(const mla_bf16_t *o_lat, int B, int H, const mla_bf16_t *w_uv,
                            const mla_bf16_t *w_o, int d_model, void *workspace, size_t ws_bytes,
                            mla_bf16_t *y, mla_stream_t stream);

/*
 * The kernels one call of each projection entry point launches for these shapes on the
 * current device (no counterpart on the pages: a query of this library's launch plan).
 * A split-K product whose k-splits fit the device as thread-block clusters (every output
 * tile's cluster resident at once) reduces them inside the cluster, in one launch;
 * otherwise it writes fp32 partials and a second launch sums them. *append = 1 or 2
 * (mla_append_kv; mla_append_kv_fp8 always 2), *absorb_q = 3..6 (W_DQ 1 or 2; W_UQ, W_QR
 * and the RoPE 1 for B <= 128, else 3; W_UK 1), *out_absorb = 2 or 3 (W_UV 1; W_O 1 or
 * 2), *append_absorb_q = 3 or 5 (W_DQ with W_DKR 1, then as absorb_q) or the sum of the
 * two calls' counts. With no visible device the partial-writing plan is reported. Any output pointer may
 * be null. Same argument rules as the entry points (MLA_ERR_INVALID_ARG, or
 * MLA_ERR_UNSUPPORTED for H).
 */
mla_status_t mla_projection_launches(int B, int d_model, int q_lora, int H, int *append,
                                     int *absorb_q, int *out_absorb, int *append_absorb_q);

/* ------------------------------------------------------- device status */

/* Zero the workspace's error word (asynchronous on `stream`). */
mla_status_t mla_clear_device_status(void *workspace, mla_stream_t stream);

/*
 * Synchronise `stream`, then return the first device-detected error recorded in
 * the workspace (MLA_OK if none) and clear it. Returns MLA_ERR_CUDA if the
 * synchronisation itself fails.
 */
mla_status_t mla_check_device_status(void *workspace, mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
