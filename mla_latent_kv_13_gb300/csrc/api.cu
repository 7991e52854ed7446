// api.cu -- the C ABI of libmla (declared in include/mla.h): host-side validation,
// workspace layout, split planning and kernel launches.
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "kernels.h"

using namespace mla;

namespace {

constexpr size_t HDR = MLA_WS_HEADER_BYTES;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cudaStream_t S(mla_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

uint32_t *err_word(void *ws) { return reinterpret_cast<uint32_t *>(ws); }

mla_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

bool heads_ok(int H) { return H == 16 || H == 32 || H == 64 || H == 128; }

// K cut into ranges (multiples of 64) for the tensor-core GEMM (128 x 128 output tiles,
// one CTA per SM): minimise waves x (k-blocks per range + a fixed per-CTA cost of about
// three k-blocks for filling and draining its pipeline).
void plan_ksplit(int M, int N, int K, int batch, int &splits, int &per) {
    const int bn = gemm_block_n(M, N, K);
    const long tiles = (long)((N + bn - 1) / bn) * ((M + 127) / 128) * batch;
    const int slots = device_sm_count();
    const int kblocks = K / 64;
    int best = 1;
    long best_cost = -1;
    for (int s = 1; s <= kblocks; ++s) {
        const long waves = (tiles * s + slots - 1) / slots;
        const long cost = waves * ((kblocks + s - 1) / s + 3);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    per = ((kblocks + best - 1) / best) * 64;
    splits = (K + per - 1) / per;
}

// Token ranges per sequence. An explicit request is taken as is. Otherwise the best
// fixed split (fewest waves x tiles per range, plus the partials' traffic, assuming all
// sequences are max_seqlen long) is used when it fits in one wave of clusters; when it
// would not, 0 is returned: the balanced schedule (equal shares of the concatenated
// tiles, each sequence weighted with its start-up cost) avoids the partly empty last wave,
// at the price of restarting the pipeline at every sequence boundary inside a share.
int plan_decode_splits(int B, int H, int max_seqlen, int requested) {
    if (requested > 0) return requested;
    int T = (max_seqlen + BLOCK - 1) / BLOCK;
    if (T < 1) T = 1;
    const int slots = decode_tc_cluster_slots();
    const double part_cost = (double)H * D_C * 4 * 2 / (BLOCK * D_QK * 2);
    int best = 1;
    long best_waves = 1;
    double best_cost = -1;
    for (int s = 1; s <= 64 && s <= T; ++s) {
        const long items = (long)B * s;
        const long waves = (items + slots - 1) / slots;
        const double cost = (double)waves * ((T + s - 1) / s) +
                            (s > 1 ? (double)items * part_cost / slots : 0.0);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
            best_waves = waves;
        }
    }
    return best_waves == 1 ? best : 0;
}

// Clusters of the balanced schedule: every resident 2-CTA cluster, at most one per tile.
int sched_clusters(int B, int max_seqlen) {
    const long tiles = (long)B * ((max_seqlen + BLOCK - 1) / BLOCK);
    const int slots = decode_tc_cluster_slots();
    return (int)(tiles < 1 ? 1 : (tiles < slots ? tiles : slots));
}

struct DecodeLayout {
    size_t tile_start, wpos, part_begin, nparts, jobs, o_part, lse_part, total;
};

DecodeLayout decode_layout(int B, int H, int max_seqlen, int splits) {
    DecodeLayout L{};
    if (splits == 1) {
        L.total = HDR;
        return L;
    }
    if (splits > 1) {
        L.o_part = HDR;
        L.lse_part = L.o_part + align256((size_t)B * splits * H * D_C * sizeof(float));
        L.total = L.lse_part + align256((size_t)B * splits * H * sizeof(float));
        return L;
    }
    const int P = sched_clusters(B, max_seqlen);
    const size_t parts = 2 * (size_t)P;  // each cluster cuts at most two sequences
    L.tile_start = HDR;
    L.wpos = L.tile_start + align256((size_t)(B + 1) * 4);
    L.part_begin = L.wpos + align256((size_t)(B + 1) * 4);
    L.nparts = L.part_begin + align256((size_t)B * 4);
    L.jobs = L.nparts + align256((size_t)B * 4);
    L.o_part = L.jobs + align256((size_t)P * 16);
    L.lse_part = L.o_part + align256(parts * H * D_C * sizeof(float));
    L.total = L.lse_part + align256(parts * H * sizeof(float));
    return L;
}

}  // namespace

namespace mla {
int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}
}  // namespace mla

extern "C" {

const char *mla_status_string(mla_status_t s) {
    switch (s) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
        case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
        case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
        case MLA_ERR_OUT_OF_RANGE: return "MLA_ERR_OUT_OF_RANGE";
        case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
        case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    }
    return "MLA_ERR_UNKNOWN";
}

// ------------------------------------------------------------------ append

mla_status_t mla_append_kv_workspace_size(int B, int d_model, size_t *bytes) {
    if (!bytes || B < 1 || B > 4096 || d_model < 64 || d_model % 64) return MLA_ERR_INVALID_ARG;
    int splits, per;
    plan_ksplit(B, D_QK, d_model, 1, splits, per);
    *bytes = HDR + align256((size_t)splits * B * D_QK * sizeof(float));
    return MLA_OK;
}

mla_status_t mla_append_kv(const mla_bf16_t *h, int B, int d_model, const mla_bf16_t *w_dkr,
                           const int32_t *pos, const int32_t *block_table, int max_blocks,
                           mla_bf16_t *kv_cache, int num_blocks, float rope_theta,
                           void *workspace, size_t ws_bytes, mla_stream_t stream) {
    if (!h || !w_dkr || !pos || !block_table || !kv_cache || !workspace)
        return MLA_ERR_INVALID_ARG;
    if (B < 1 || B > 4096 || d_model < 64 || d_model % 64 || max_blocks < 1 || num_blocks < 1 ||
        !(rope_theta > 0.f) || !isfinite(rope_theta))
        return MLA_ERR_INVALID_ARG;
    if (!aligned(h, 16) || !aligned(w_dkr, 16) || !aligned(kv_cache, 16) ||
        !aligned(workspace, 256))
        return MLA_ERR_INVALID_ARG;
    size_t need;
    mla_append_kv_workspace_size(B, d_model, &need);
    if (ws_bytes < need) return MLA_ERR_WORKSPACE;

    int splits, per;
    plan_ksplit(B, D_QK, d_model, 1, splits, per);
    float *part = reinterpret_cast<float *>(static_cast<char *>(workspace) + HDR);
    GemmParams g{};
    g.A = h; g.lda = d_model; g.a_bstride = 0;
    g.B = w_dkr; g.ldb = d_model; g.b_bstride = 0;
    g.M = B; g.N = D_QK; g.K = d_model; g.batch = 1;
    // the k-splits reduced inside their cluster, whose epilogue rotates k_rope and writes
    // the rows into the cache, when the device holds every tile's cluster at once; else
    // partials and a finalize launch
    int per_c = 0, bn_c = 0;
    const int s_c = gemm_cluster_plan(B, D_QK, d_model, &per_c, &bn_c);
    if (s_c > 0) {
        g.k_splits = s_c; g.k_per_split = per_c;
        const ClusterAppend ap{pos, block_table, max_blocks, num_blocks, kv_cache, rope_theta};
        return cuda_status(launch_gemm_tc_cluster(g, bn_c, &ap, S(stream), err_word(workspace)));
    }
    g.k_splits = splits; g.k_per_split = per;
    g.c_part = part;
    cudaError_t e = launch_gemm_tc(g, false, S(stream), err_word(workspace));
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    e = launch_append_finalize(part, splits, B, pos, block_table, max_blocks, kv_cache, num_blocks,
                               rope_theta, err_word(workspace), S(stream));
    return cuda_status(e);
}

mla_status_t mla_append_kv_fp8(const mla_bf16_t *h, int B, int d_model, const mla_bf16_t *w_dkr,
                               const int32_t *pos, const int32_t *block_table, int max_blocks,
                               uint8_t *kv_codes, int8_t *kv_exps, int num_blocks,
                               float rope_theta, void *workspace, size_t ws_bytes,
                               mla_stream_t stream) {
    if (!h || !w_dkr || !pos || !block_table || !kv_codes || !kv_exps || !workspace)
        return MLA_ERR_INVALID_ARG;
    if (B < 1 || B > 4096 || d_model < 64 || d_model % 64 || max_blocks < 1 || num_blocks < 1 ||
        !(rope_theta > 0.f) || !isfinite(rope_theta))
        return MLA_ERR_INVALID_ARG;
    if (!aligned(h, 16) || !aligned(w_dkr, 16) || !aligned(kv_codes, 16) ||
        !aligned(workspace, 256))
        return MLA_ERR_INVALID_ARG;
    size_t need;
    mla_append_kv_workspace_size(B, d_model, &need);
    if (ws_bytes < need) return MLA_ERR_WORKSPACE;
    int splits, per;
    plan_ksplit(B, D_QK, d_model, 1, splits, per);
    float *part = reinterpret_cast<float *>(static_cast<char *>(workspace) + HDR);
    GemmParams g{};
    g.A = h; g.lda = d_model; g.a_bstride = 0;
    g.B = w_dkr; g.ldb = d_model; g.b_bstride = 0;
    g.M = B; g.N = D_QK; g.K = d_model; g.batch = 1;
    g.k_splits = splits; g.k_per_split = per;
    g.c_part = part;
    if (launch_gemm_tc(g, false, S(stream), err_word(workspace)) != cudaSuccess) return MLA_ERR_CUDA;
    return cuda_status(launch_append_finalize_fp8(part, splits, B, pos, block_table, max_blocks,
                                                  kv_codes, kv_exps, num_blocks, rope_theta,
                                                  err_word(workspace), S(stream)));
}

// ---------------------------------------------------------------- decode

mla_status_t mla_decode_workspace_size(int B, int H, int max_seqlen, int num_splits,
                                       size_t *bytes) {
    if (!bytes || B < 1 || B > 4096 || max_seqlen < 0 || num_splits < 0 || num_splits > 256)
        return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
    *bytes = decode_layout(B, H, max_seqlen, plan_decode_splits(B, H, max_seqlen, num_splits)).total;
    return MLA_OK;
}

mla_status_t mla_decode_plan(int B, int H, int max_seqlen, int num_splits, int *splits,
                             int *launches) {
    if (B < 1 || B > 4096 || max_seqlen < 0 || num_splits < 0 || num_splits > 256)
        return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
    const int s = plan_decode_splits(B, H, max_seqlen, num_splits);
    if (splits) *splits = s;
    if (launches) *launches = s == 0 ? 3 : (s > 1 ? 2 : 1);
    return MLA_OK;
}

mla_status_t mla_decode_schedule(const int32_t *seqlens, int B, int max_blocks, int clusters,
                                 int32_t *segs, int capacity, int *count, int *parts) {
    if (!seqlens || !count || B < 1 || B > 4096 || max_blocks < 1 || clusters < 1 ||
        capacity < 0 || (capacity > 0 && !segs))
        return MLA_ERR_INVALID_ARG;
    // the same arithmetic as the schedule kernel, on the host
    std::vector<int32_t> tile_start(B + 1), wpos(B + 1), part_begin(B), v(B);
    long T = 0, W = 0;
    for (int b = 0; b < B; ++b) {
        const int L = seqlens[b] < 0 ? 0 : std::min(seqlens[b], max_blocks * BLOCK);
        v[b] = (L + BLOCK - 1) / BLOCK;
        tile_start[b] = static_cast<int32_t>(T);
        wpos[b] = static_cast<int32_t>(W + (v[b] > 0 ? SEG_COST : 0));
        T += v[b];
        W += v[b] > 0 ? v[b] + SEG_COST : 0;
    }
    if (W > INT32_MAX) return MLA_ERR_INVALID_ARG;
    tile_start[B] = static_cast<int32_t>(T);
    wpos[B] = static_cast<int32_t>(W);
    const int P = W < clusters ? static_cast<int>(W) : clusters;
    int np_total = 0;
    for (int b = 0; b < B; ++b) {
        part_begin[b] = np_total;
        if (v[b] > 0) {
            const int c0 = cluster_of_tile(wpos[b], W, P);
            const int c1 = cluster_of_tile(wpos[b] + v[b] - 1, W, P);
            if (c1 > c0) np_total += c1 - c0 + 1;
        }
    }
    int n = 0;
    for (int cl = 0; cl < P; ++cl) {
        const long r0 = (cl * W) / P, r1 = ((cl + 1) * W) / P;
        int cursor = sched_first(wpos.data(), B, r0);
        SchedSegment sg;
        while (sched_next(tile_start.data(), wpos.data(), part_begin.data(), B, r0, r1, W, P, cl,
                          &cursor, &sg)) {
            if (n < capacity) {
                int32_t *e = segs + 5 * (size_t)n;
                e[0] = cl;
                e[1] = sg.b;
                e[2] = sg.t_begin;
                e[3] = sg.t_end;
                e[4] = sg.direct ? -1 : sg.part;
            }
            ++n;
        }
    }
    *count = n;
    if (parts) *parts = np_total;
    return MLA_OK;
}

}  // extern "C"

namespace mla {
// Host-side checks of a decode call's arguments (every one except the workspace), shared
// by every decode entry point so that a rejected call touches nothing on the device.
mla_status_t decode_validate(const void *q_lat, const void *q_rope, const void *kv_cache,
                             int num_blocks, const int32_t *block_table, int max_blocks,
                             const int32_t *seqlens, int B, int s_q, int hq, int max_seqlen,
                             float scale, int num_splits, const void *out, const float *lse) {
    if (!q_lat || !q_rope || !kv_cache || !block_table || !seqlens || !out || !lse)
        return MLA_ERR_INVALID_ARG;
    if (B < 1 || B > 4096 || num_blocks < 1 || max_blocks < 1 || max_seqlen < 0 ||
        max_seqlen > max_blocks * BLOCK || num_splits < 0 || num_splits > 256 ||
        !(scale > 0.f) || !isfinite(scale) || s_q < 1)
        return MLA_ERR_INVALID_ARG;
    if (!heads_ok(hq) || s_q * hq > 128) return MLA_ERR_UNSUPPORTED;
    if (!aligned(q_lat, 16) || !aligned(q_rope, 16) || !aligned(kv_cache, 16) ||
        !aligned(out, 32) || !aligned(lse, 4))
        return MLA_ERR_INVALID_ARG;
    return MLA_OK;
}
}  // namespace mla

namespace {
// Decode over H = s_q x hq query rows per sequence (query token t, head h at row t*hq + h);
// token t sees the rows j < seqlens[b] - (s_q - 1 - t). Plain decode: s_q = 1, hq = H.
// The output goes to `out` as bf16, or, when out_f32 is given, to out_f32 as fp32.
// The cache is bf16 rows (kv_cache), or e4m3 codes with row exponents (codes, exps).
mla_status_t decode_run(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                        const mla_bf16_t *kv_cache, int num_blocks, const int32_t *block_table,
                        int max_blocks, const int32_t *seqlens, int B, int s_q, int hq,
                        int max_seqlen, float scale, int num_splits, void *workspace,
                        size_t ws_bytes, mla_bf16_t *out, float *out_f32, float *lse,
                        mla_stream_t stream, const uint8_t *codes = nullptr,
                        const int8_t *exps = nullptr, bool prepared = false) {
    const int H = s_q * hq;
    const void *out_any = out_f32 ? static_cast<const void *>(out_f32) : out;
    const void *cache_any = codes ? static_cast<const void *>(codes) : kv_cache;
    const mla_status_t v = decode_validate(q_lat, q_rope, cache_any, num_blocks, block_table,
                                           max_blocks, seqlens, B, s_q, hq, max_seqlen, scale,
                                           num_splits, out_any, lse);
    if (v != MLA_OK) return v;
    if (codes && (!exps || !aligned(exps, 16))) return MLA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
    const int splits = plan_decode_splits(B, H, max_seqlen, num_splits);
    const DecodeLayout lay = decode_layout(B, H, max_seqlen, splits);
    if (ws_bytes < lay.total) return MLA_ERR_WORKSPACE;

    const int T = (max_seqlen + BLOCK - 1) / BLOCK;
    char *w = static_cast<char *>(workspace);
    DecodeParams p{};
    p.q_lat = q_lat; p.q_rope = q_rope; p.cache = kv_cache;
    p.codes = codes; p.exps = exps;
    p.block_table = block_table; p.seqlens = seqlens;
    p.num_blocks = num_blocks; p.max_blocks = max_blocks; p.B = B; p.H = H;
    p.max_seqlen = max_seqlen;
    p.s_q = s_q; p.hq = hq;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = out; p.out_f32 = out_f32; p.lse = lse;
    p.err = err_word(workspace);
    cudaStream_t st = S(stream);
    if (splits >= 1) {
        p.num_splits = splits;
        p.tiles_per_split = T > 0 ? (T + splits - 1) / splits : 1;
        if (splits > 1) {
            p.o_part = reinterpret_cast<float *>(w + lay.o_part);
            p.lse_part = reinterpret_cast<float *>(w + lay.lse_part);
        }
        cudaError_t e = launch_decode_tc(p, B * splits, st);
        if (e != cudaSuccess) return MLA_ERR_CUDA;
        if (splits > 1)
            e = launch_combine(p.o_part, p.lse_part, B, splits, H, (long)splits * H * D_C,
                               (long)H * D_C, (long)splits * H, H, out, out_f32, lse, st);
        return cuda_status(e);
    }
    // balanced schedule: tile offsets on the device, P persistent clusters, merge of cut sequences
    const int P = sched_clusters(B, max_seqlen);
    int32_t *tile_start = reinterpret_cast<int32_t *>(w + lay.tile_start);
    int32_t *wpos = reinterpret_cast<int32_t *>(w + lay.wpos);
    int32_t *part_begin = reinterpret_cast<int32_t *>(w + lay.part_begin);
    int32_t *nparts = reinterpret_cast<int32_t *>(w + lay.nparts);
    p.num_splits = 1;
    p.tiles_per_split = T;
    p.tile_start = tile_start;
    p.wpos = wpos;
    p.part_begin = part_begin;
    p.nparts = nparts;
    p.o_part = reinterpret_cast<float *>(w + lay.o_part);
    p.lse_part = reinterpret_cast<float *>(w + lay.lse_part);
    int4 *jobs = reinterpret_cast<int4 *>(w + lay.jobs);
    if (!prepared && launch_decode_schedule(seqlens, B, max_seqlen, P, tile_start, wpos,
                                            part_begin, nparts, jobs, p.err, st) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (launch_decode_tc(p, P, st) != cudaSuccess) return MLA_ERR_CUDA;
    return cuda_status(launch_combine_sched(p.o_part, p.lse_part, jobs, tile_start, B, P, H, out,
                                            out_f32, lse, st));
}

}  // namespace

extern "C" {

mla_status_t mla_decode_attention(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                                  const mla_bf16_t *kv_cache, int num_blocks,
                                  const int32_t *block_table, int max_blocks,
                                  const int32_t *seqlens, int B, int H, int max_seqlen,
                                  float scale, int num_splits, void *workspace,
                                  size_t ws_bytes, mla_bf16_t *out, float *lse,
                                  mla_stream_t stream) {
    return decode_run(q_lat, q_rope, kv_cache, num_blocks, block_table, max_blocks, seqlens, B,
                      1, H, max_seqlen, scale, num_splits, workspace, ws_bytes, out, nullptr, lse,
                      stream);
}

mla_status_t mla_decode_prepare(const int32_t *seqlens, int B, int H, int max_seqlen,
                                int num_splits, void *workspace, size_t ws_bytes,
                                mla_stream_t stream) {
    if (!seqlens || !workspace || B < 1 || B > 4096 || max_seqlen < 0 || num_splits < 0 ||
        num_splits > 256)
        return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
    if (!aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
    const int splits = plan_decode_splits(B, H, max_seqlen, num_splits);
    const DecodeLayout lay = decode_layout(B, H, max_seqlen, splits);
    if (ws_bytes < lay.total) return MLA_ERR_WORKSPACE;
    if (splits != 0) return MLA_OK;  // a fixed split needs no schedule
    char *w = static_cast<char *>(workspace);
    return cuda_status(launch_decode_schedule(
        seqlens, B, max_seqlen, sched_clusters(B, max_seqlen),
        reinterpret_cast<int32_t *>(w + lay.tile_start), reinterpret_cast<int32_t *>(w + lay.wpos),
        reinterpret_cast<int32_t *>(w + lay.part_begin), reinterpret_cast<int32_t *>(w + lay.nparts),
        reinterpret_cast<int4 *>(w + lay.jobs), err_word(workspace), S(stream)));
}

mla_status_t mla_decode_attention_prepared(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                                           const mla_bf16_t *kv_cache, int num_blocks,
                                           const int32_t *block_table, int max_blocks,
                                           const int32_t *seqlens, int B, int H, int max_seqlen,
                                           float scale, int num_splits, void *workspace,
                                           size_t ws_bytes, mla_bf16_t *out, float *lse,
                                           mla_stream_t stream) {
    return decode_run(q_lat, q_rope, kv_cache, num_blocks, block_table, max_blocks, seqlens, B,
                      1, H, max_seqlen, scale, num_splits, workspace, ws_bytes, out, nullptr, lse,
                      stream, nullptr, nullptr, true);
}

mla_status_t mla_decode_attention_fp8(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                                      const uint8_t *kv_codes, const int8_t *kv_exps,
                                      int num_blocks, const int32_t *block_table, int max_blocks,
                                      const int32_t *seqlens, int B, int H, int max_seqlen,
                                      float scale, int num_splits, void *workspace,
                                      size_t ws_bytes, mla_bf16_t *out, float *lse,
                                      mla_stream_t stream) {
    if (!kv_codes) return MLA_ERR_INVALID_ARG;
    return decode_run(q_lat, q_rope, nullptr, num_blocks, block_table, max_blocks, seqlens, B, 1,
                      H, max_seqlen, scale, num_splits, workspace, ws_bytes, out, nullptr, lse,
                      stream, kv_codes, kv_exps);
}

mla_status_t mla_quantize_kv_fp8(const mla_bf16_t *rows_bf16, long rows, uint8_t *codes,
                                 int8_t *exps, mla_stream_t stream) {
    if (!rows_bf16 || !codes || !exps || rows < 0 || rows > (1L << 40))
        return MLA_ERR_INVALID_ARG;
    if (!aligned(rows_bf16, 16) || !aligned(codes, 16)) return MLA_ERR_INVALID_ARG;
    return cuda_status(launch_quantize_rows(rows_bf16, rows, codes, exps, S(stream)));
}

mla_status_t mla_dequantize_kv_fp8(const uint8_t *codes, const int8_t *exps, long rows,
                                   mla_bf16_t *rows_bf16, mla_stream_t stream) {
    if (!rows_bf16 || !codes || !exps || rows < 0 || rows > (1L << 40))
        return MLA_ERR_INVALID_ARG;
    if (!aligned(rows_bf16, 16) || !aligned(codes, 16)) return MLA_ERR_INVALID_ARG;
    return cuda_status(launch_dequantize_rows(codes, exps, rows, rows_bf16, S(stream)));
}

mla_status_t mla_decode_attention_partial(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                                          const mla_bf16_t *kv_cache, int num_blocks,
                                          const int32_t *block_table, int max_blocks,
                                          const int32_t *seqlens, int B, int H, int max_seqlen,
                                          float scale, int num_splits, void *workspace,
                                          size_t ws_bytes, float *o_part, float *lse_part,
                                          mla_stream_t stream) {
    if (!o_part) return MLA_ERR_INVALID_ARG;
    return decode_run(q_lat, q_rope, kv_cache, num_blocks, block_table, max_blocks, seqlens, B,
                      1, H, max_seqlen, scale, num_splits, workspace, ws_bytes, nullptr, o_part,
                      lse_part, stream);
}

mla_status_t mla_decode_mq_workspace_size(int B, int s_q, int H, int max_seqlen, int num_splits,
                                          size_t *bytes) {
    if (s_q < 1) return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H) || s_q * H > 128) return MLA_ERR_UNSUPPORTED;
    if (!bytes || B < 1 || B > 4096 || max_seqlen < 0 || num_splits < 0 || num_splits > 256)
        return MLA_ERR_INVALID_ARG;
    const int rows = s_q * H;
    *bytes = decode_layout(B, rows, max_seqlen, plan_decode_splits(B, rows, max_seqlen, num_splits))
                 .total;
    return MLA_OK;
}

mla_status_t mla_decode_attention_mq(const mla_bf16_t *q_lat, const mla_bf16_t *q_rope,
                                     const mla_bf16_t *kv_cache, int num_blocks,
                                     const int32_t *block_table, int max_blocks,
                                     const int32_t *seqlens, int B, int s_q, int H,
                                     int max_seqlen, float scale, int num_splits, void *workspace,
                                     size_t ws_bytes, mla_bf16_t *out, float *lse,
                                     mla_stream_t stream) {
    return decode_run(q_lat, q_rope, kv_cache, num_blocks, block_table, max_blocks, seqlens, B,
                      s_q, H, max_seqlen, scale, num_splits, workspace, ws_bytes, out, nullptr, lse,
                      stream);
}

// ------------------------------------------------------------- prefill

namespace {
struct PrefillLayout {
    size_t ckv, kr, kn, v, total;
};
PrefillLayout prefill_layout(int H, int T) {
    PrefillLayout L{};
    L.ckv = HDR;
    L.kr = L.ckv + align256((size_t)T * D_C * 2);
    L.kn = L.kr + align256((size_t)T * D_ROPE * 2);
    L.v = L.kn + align256((size_t)T * H * D_NOPE * 2);
    L.total = L.v + align256((size_t)T * H * D_V * 2);
    return L;
}
}  // namespace

mla_status_t mla_prefill_workspace_size(int H, int prefix, int chunk, size_t *bytes) {
    if (!bytes || prefix < 0 || chunk < 1 || (long)prefix + chunk > (1L << 24))
        return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
    *bytes = prefill_layout(H, prefix + chunk).total;
    return MLA_OK;
}

mla_status_t mla_prefill_attention(const mla_bf16_t *q_nope, const mla_bf16_t *q_rope,
                                   const mla_bf16_t *kv_cache, int num_blocks,
                                   const int32_t *block_table, int max_blocks, int prefix,
                                   int chunk, int H, const mla_bf16_t *w_uk,
                                   const mla_bf16_t *w_uv, float scale, void *workspace,
                                   size_t ws_bytes, mla_bf16_t *out, float *lse,
                                   mla_stream_t stream) {
    if (!q_nope || !q_rope || !kv_cache || !block_table || !w_uk || !w_uv || !workspace || !out ||
        !lse)
        return MLA_ERR_INVALID_ARG;
    if (num_blocks < 1 || max_blocks < 1 || prefix < 0 || chunk < 1 ||
        (long)prefix + chunk > (long)max_blocks * BLOCK || !(scale > 0.f) || !isfinite(scale))
        return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
    if (!aligned(q_nope, 16) || !aligned(q_rope, 16) || !aligned(kv_cache, 16) ||
        !aligned(w_uk, 16) || !aligned(w_uv, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
        !aligned(workspace, 256))
        return MLA_ERR_INVALID_ARG;
    const int T = prefix + chunk;
    const PrefillLayout lay = prefill_layout(H, T);
    if (ws_bytes < lay.total) return MLA_ERR_WORKSPACE;
    char *w = static_cast<char *>(workspace);
    uint16_t *ckv = reinterpret_cast<uint16_t *>(w + lay.ckv);
    uint16_t *kr = reinterpret_cast<uint16_t *>(w + lay.kr);
    uint16_t *kn = reinterpret_cast<uint16_t *>(w + lay.kn);
    uint16_t *v = reinterpret_cast<uint16_t *>(w + lay.v);
    uint32_t *err = err_word(workspace);
    cudaStream_t st = S(stream);
    // the sequence's latent rows, then K_nope = c_kv W_UK^T and V = c_kv W_UV^T per head
    if (launch_gather_rows(kv_cache, num_blocks, block_table, max_blocks, T, ckv, kr, err, st) !=
        cudaSuccess)
        return MLA_ERR_CUDA;
    for (int k = 0; k < 2; ++k) {
        GemmParams g{};
        g.A = ckv; g.lda = D_C; g.a_bstride = 0;
        g.B = k == 0 ? w_uk : w_uv; g.ldb = D_C; g.b_bstride = 0;
        g.M = T; g.N = H * (k == 0 ? D_NOPE : D_V); g.K = D_C; g.batch = 1;
        g.k_splits = 1; g.k_per_split = D_C;
        g.c_bf16 = k == 0 ? kn : v; g.ldc = g.N; g.c_bstride = 0;
        if (launch_gemm_tc(g, false, st, err) != cudaSuccess) return MLA_ERR_CUDA;
    }
    return cuda_status(launch_prefill_tc(q_nope, q_rope, kn, kr, v, chunk, T, H, prefix, scale,
                                         out, lse, err, st));
}

mla_status_t mla_selftest_wait_timeout(unsigned limit_us, void *workspace, size_t ws_bytes,
                                       mla_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000 || !workspace || ws_bytes < MLA_WS_HEADER_BYTES ||
        !aligned(workspace, 256))
        return MLA_ERR_INVALID_ARG;
    return cuda_status(launch_bounded_wait_selftest(static_cast<uint64_t>(limit_us) * 1000u,
                                                    err_word(workspace), S(stream)));
}

mla_status_t mla_decode_combine(const float *o_part, const float *lse_part, int B, int S_, int H,
                                mla_bf16_t *out, float *lse, mla_stream_t stream) {
    if (!o_part || !lse_part || !out || !lse || B < 1 || S_ < 1 || H < 1 || H > 65535)
        return MLA_ERR_INVALID_ARG;
    if (!aligned(o_part, 16) || !aligned(out, 8) || !aligned(lse, 4)) return MLA_ERR_INVALID_ARG;
    return cuda_status(launch_combine(o_part, lse_part, B, S_, H, (long)S_ * H * D_C,
                                      (long)H * D_C, (long)S_ * H, H, out, nullptr, lse,
                                      S(stream)));
}

mla_status_t mla_decode_combine_ranks(const float *o_parts, const float *lse_parts, int G, int B,
                                      int H, mla_bf16_t *out, float *lse, mla_stream_t stream) {
    if (!o_parts || !lse_parts || !out || !lse || G < 1 || G > 4096 || B < 1 || B > 4096 ||
        H < 1 || H > 65535)
        return MLA_ERR_INVALID_ARG;
    if (!aligned(o_parts, 16) || !aligned(out, 8) || !aligned(lse, 4)) return MLA_ERR_INVALID_ARG;
    return cuda_status(launch_combine(o_parts, lse_parts, B, G, H, (long)H * D_C,
                                      (long)B * H * D_C, H, (long)B * H, out, nullptr, lse,
                                      S(stream)));
}

// ------------------------------------------------------------ absorb_q

namespace {
struct AbsorbQLayout {
    int s1, per1;     // split of c_q = h W_DQ^T
    int s2, per2;     // split of c_q W_QR^T (q_rope before rotation)
    size_t part, cq, qn, total;
};
AbsorbQLayout absorb_q_layout(int B, int d_model, int q_lora, int H) {
    AbsorbQLayout L{};
    plan_ksplit(B, q_lora, d_model, 1, L.s1, L.per1);
    plan_ksplit(B, H * D_ROPE, q_lora, 1, L.s2, L.per2);
    size_t part1 = (size_t)L.s1 * B * q_lora * sizeof(float);
    size_t part2 = (size_t)L.s2 * B * H * D_ROPE * sizeof(float);
    L.part = HDR;
    L.cq = L.part + align256(part1 > part2 ? part1 : part2);
    L.qn = L.cq + align256((size_t)B * q_lora * 2);
    L.total = L.qn + align256((size_t)B * H * D_NOPE * 2);
    return L;
}
}  // namespace

namespace {
// absorb_q after c_q: q_nope and q_rope (one launch for up to 128 sequences), then the
// per-head W_UK absorption into q_lat
mla_status_t absorb_q_from_cq(const uint16_t *cq, int B, int q_lora, const mla_bf16_t *w_uq,
                              const mla_bf16_t *w_qr, const mla_bf16_t *w_uk, int H,
                              const int32_t *pos, float rope_theta, const AbsorbQLayout &L,
                              float *part, uint16_t *qn, mla_bf16_t *q_lat, mla_bf16_t *q_rope,
                              cudaStream_t st, uint32_t *err) {
    if (B <= 128) {
        // q_nope = c_q W_UQ^T (bf16 intermediate [B][H*128]) and q_rope = RoPE(c_q W_QR^T)
        // in one launch: both read c_q, and the rotation is the second product's epilogue
        if (launch_gemm_tc_rope(cq, B, q_lora, w_uq, H * D_NOPE, qn, w_qr, H * D_ROPE, q_rope,
                                pos, rope_theta, st, err) != cudaSuccess)
            return MLA_ERR_CUDA;
    } else {
        // q_nope = c_q W_UQ^T (bf16 intermediate [B][H*128])
        GemmParams g{};
        g.A = cq; g.lda = q_lora; g.B = w_uq; g.ldb = q_lora;
        g.M = B; g.N = H * D_NOPE; g.K = q_lora; g.batch = 1;
        g.k_splits = 1; g.k_per_split = q_lora; g.c_bf16 = qn; g.ldc = H * D_NOPE;
        if (launch_gemm_tc(g, false, st, err) != cudaSuccess) return MLA_ERR_CUDA;

        // q_rope = RoPE(c_q W_QR^T)
        g = GemmParams{};
        g.A = cq; g.lda = q_lora; g.B = w_qr; g.ldb = q_lora;
        g.M = B; g.N = H * D_ROPE; g.K = q_lora; g.batch = 1;
        g.k_splits = L.s2; g.k_per_split = L.per2; g.c_part = part;
        if (launch_gemm_tc(g, false, st, err) != cudaSuccess) return MLA_ERR_CUDA;
        if (launch_qrope_finalize(part, L.s2, B, H, pos, rope_theta, q_rope, st) != cudaSuccess)
            return MLA_ERR_CUDA;
    }

    // q_lat[b, i] = q_nope[b, i] W_UK_i  (per-head product, W_UK_i stored [128][512])
    GemmParams g{};
    g.A = qn; g.lda = H * D_NOPE; g.a_bstride = D_NOPE;
    g.B = w_uk; g.ldb = D_C; g.b_bstride = (long)D_NOPE * D_C;
    g.M = B; g.N = D_C; g.K = D_NOPE; g.batch = H;
    g.k_splits = 1; g.k_per_split = D_NOPE;
    g.c_bf16 = q_lat; g.ldc = (long)H * D_C; g.c_bstride = D_C;
    return cuda_status(launch_gemm_tc(g, true, st, err));
}

}  // namespace

mla_status_t mla_absorb_q_workspace_size(int B, int d_model, int q_lora, int H, size_t *bytes) {
    if (!bytes || B < 1 || B > 4096 || d_model < 64 || d_model % 64 || q_lora < 64 ||
        q_lora % 64)
        return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
    *bytes = absorb_q_layout(B, d_model, q_lora, H).total;
    return MLA_OK;
}

mla_status_t mla_absorb_q(const mla_bf16_t *h, int B, int d_model, const mla_bf16_t *w_dq,
                          int q_lora, const mla_bf16_t *w_uq, const mla_bf16_t *w_qr,
                          const mla_bf16_t *w_uk, int H, const int32_t *pos, float rope_theta,
                          void *workspace, size_t ws_bytes, mla_bf16_t *q_lat,
                          mla_bf16_t *q_rope, mla_stream_t stream) {
    if (!h || !w_dq || !w_uq || !w_qr || !w_uk || !pos || !workspace || !q_lat || !q_rope)
        return MLA_ERR_INVALID_ARG;
    if (B < 1 || B > 4096 || d_model < 64 || d_model % 64 || q_lora < 64 || q_lora % 64 ||
        !(rope_theta > 0.f) || !isfinite(rope_theta))
        return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
    if (!aligned(h, 16) || !aligned(w_dq, 16) || !aligned(w_uq, 16) || !aligned(w_qr, 16) ||
        !aligned(w_uk, 16) || !aligned(q_lat, 16) || !aligned(q_rope, 16) ||
        !aligned(workspace, 256))
        return MLA_ERR_INVALID_ARG;
    AbsorbQLayout L = absorb_q_layout(B, d_model, q_lora, H);
    if (ws_bytes < L.total) return MLA_ERR_WORKSPACE;
    char *w = static_cast<char *>(workspace);
    float *part = reinterpret_cast<float *>(w + L.part);
    uint16_t *cq = reinterpret_cast<uint16_t *>(w + L.cq);
    uint16_t *qn = reinterpret_cast<uint16_t *>(w + L.qn);
    cudaStream_t st = S(stream);

    uint32_t *err = err_word(workspace);

    // c_q = h W_DQ^T (bf16 intermediate): k-splits reduced inside their cluster when the
    // device holds every tile's cluster at once, else partials and a finalize launch
    GemmParams g{};
    g.A = h; g.lda = d_model; g.B = w_dq; g.ldb = d_model;
    g.M = B; g.N = q_lora; g.K = d_model; g.batch = 1;
    int per_c = 0, bn_c = 0;
    const int s_c = gemm_cluster_plan(B, q_lora, d_model, &per_c, &bn_c);
    if (s_c > 0) {
        g.k_splits = s_c; g.k_per_split = per_c; g.c_bf16 = cq; g.ldc = q_lora;
        if (launch_gemm_tc_cluster(g, bn_c, nullptr, st, err) != cudaSuccess) return MLA_ERR_CUDA;
    } else {
        g.k_splits = L.s1; g.k_per_split = L.per1; g.c_part = part;
        if (launch_gemm_tc(g, false, st, err) != cudaSuccess) return MLA_ERR_CUDA;
        if (launch_reduce_bf16(part, L.s1, 1, B, q_lora, cq, q_lora, 0, st) != cudaSuccess)
            return MLA_ERR_CUDA;
    }

    return absorb_q_from_cq(cq, B, q_lora, w_uq, w_qr, w_uk, H, pos, rope_theta, L, part, qn,
                            q_lat, q_rope, st, err);
}

// ------------------------------------------------------ append + absorb_q

mla_status_t mla_append_absorb_q_workspace_size(int B, int d_model, int q_lora, int H,
                                                size_t *bytes) {
    if (!bytes) return MLA_ERR_INVALID_ARG;
    size_t a = 0, q = 0;
    mla_status_t st = mla_append_kv_workspace_size(B, d_model, &a);
    if (st != MLA_OK) return st;
    if ((st = mla_absorb_q_workspace_size(B, d_model, q_lora, H, &q)) != MLA_OK) return st;
    *bytes = a > q ? a : q;
    return MLA_OK;
}

mla_status_t mla_append_absorb_q(const mla_bf16_t *h, int B, int d_model, const mla_bf16_t *w_dkr,
                                 const int32_t *pos, const int32_t *block_table, int max_blocks,
                                 mla_bf16_t *kv_cache, int num_blocks, const mla_bf16_t *w_dq,
                                 int q_lora, const mla_bf16_t *w_uq, const mla_bf16_t *w_qr,
                                 const mla_bf16_t *w_uk, int H, float rope_theta, void *workspace,
                                 size_t ws_bytes, mla_bf16_t *q_lat, mla_bf16_t *q_rope,
                                 mla_stream_t stream) {
    if (!h || !w_dkr || !pos || !block_table || !kv_cache || !w_dq || !w_uq || !w_qr || !w_uk ||
        !workspace || !q_lat || !q_rope)
        return MLA_ERR_INVALID_ARG;
    if (B < 1 || B > 4096 || d_model < 64 || d_model % 64 || q_lora < 64 || q_lora % 64 ||
        max_blocks < 1 || num_blocks < 1 || !(rope_theta > 0.f) || !isfinite(rope_theta))
        return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
    if (!aligned(h, 16) || !aligned(w_dkr, 16) || !aligned(kv_cache, 16) || !aligned(w_dq, 16) ||
        !aligned(w_uq, 16) || !aligned(w_qr, 16) || !aligned(w_uk, 16) || !aligned(q_lat, 16) ||
        !aligned(q_rope, 16) || !aligned(workspace, 256))
        return MLA_ERR_INVALID_ARG;
    size_t need = 0;
    mla_append_absorb_q_workspace_size(B, d_model, q_lora, H, &need);
    if (ws_bytes < need) return MLA_ERR_WORKSPACE;
    AbsorbQLayout L = absorb_q_layout(B, d_model, q_lora, H);
    char *w = static_cast<char *>(workspace);
    float *part = reinterpret_cast<float *>(w + L.part);
    uint16_t *cq = reinterpret_cast<uint16_t *>(w + L.cq);
    uint16_t *qn = reinterpret_cast<uint16_t *>(w + L.qn);
    cudaStream_t st = S(stream);
    uint32_t *err = err_word(workspace);
    // c_q = h W_DQ^T and the new cache rows from h W_DKR^T in one launch, their k-splits
    // reduced inside their clusters; where no cluster split fits, the two calls one after
    // the other (same stream, same workspace)
    const ClusterAppend ap{pos, block_table, max_blocks, num_blocks, kv_cache, rope_theta};
    const cudaError_t e = launch_gemm_tc_cluster_dq_append(h, B, d_model, w_dq, q_lora, cq, w_dkr,
                                                           ap, st, err);
    if (e == cudaErrorNotSupported) {
        cudaGetLastError();
        mla_status_t r = mla_append_kv(h, B, d_model, w_dkr, pos, block_table, max_blocks,
                                       kv_cache, num_blocks, rope_theta, workspace, ws_bytes,
                                       stream);
        if (r != MLA_OK) return r;
        return mla_absorb_q(h, B, d_model, w_dq, q_lora, w_uq, w_qr, w_uk, H, pos, rope_theta,
                            workspace, ws_bytes, q_lat, q_rope, stream);
    }
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    return absorb_q_from_cq(cq, B, q_lora, w_uq, w_qr, w_uk, H, pos, rope_theta, L, part, qn,
                            q_lat, q_rope, st, err);
}

// ---------------------------------------------------------- out_absorb

namespace {
struct OutLayout {
    int s2, per2;
    size_t ov, part, total;
};
OutLayout out_layout(int B, int H, int d_model) {
    OutLayout L{};
    plan_ksplit(B, d_model, H * D_V, 1, L.s2, L.per2);
    L.ov = HDR;
    L.part = L.ov + align256((size_t)B * H * D_V * 2);
    L.total = L.part + align256((size_t)L.s2 * B * d_model * sizeof(float));
    return L;
}
}  // namespace

mla_status_t mla_out_absorb_workspace_size(int B, int H, int d_model, size_t *bytes) {
    if (!bytes || B < 1 || B > 4096 || d_model < 64 || d_model % 64) return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
    *bytes = out_layout(B, H, d_model).total;
    return MLA_OK;
}

mla_status_t mla_out_absorb(const mla_bf16_t *o_lat, int B, int H, const mla_bf16_t *w_uv,
                            const mla_bf16_t *w_o, int d_model, void *workspace, size_t ws_bytes,
                            mla_bf16_t *y, mla_stream_t stream) {
    if (!o_lat || !w_uv || !w_o || !workspace || !y) return MLA_ERR_INVALID_ARG;
    if (B < 1 || B > 4096 || d_model < 64 || d_model % 64) return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
    if (!aligned(o_lat, 16) || !aligned(w_uv, 16) || !aligned(w_o, 16) || !aligned(y, 16) ||
        !aligned(workspace, 256))
        return MLA_ERR_INVALID_ARG;
    OutLayout L = out_layout(B, H, d_model);
    if (ws_bytes < L.total) return MLA_ERR_WORKSPACE;
    char *w = static_cast<char *>(workspace);
    uint16_t *ov = reinterpret_cast<uint16_t *>(w + L.ov);
    float *part = reinterpret_cast<float *>(w + L.part);
    cudaStream_t st = S(stream);

    uint32_t *err = err_word(workspace);

    // o_v[b, i] = W_UV_i o_lat[b, i]   (per head: A = o_lat [B][512], B = W_UV_i [128][512])
    GemmParams g{};
    g.A = o_lat; g.lda = (long)H * D_C; g.a_bstride = D_C;
    g.B = w_uv; g.ldb = D_C; g.b_bstride = (long)D_V * D_C;
    g.M = B; g.N = D_V; g.K = D_C; g.batch = H;
    g.k_splits = 1; g.k_per_split = D_C;
    g.c_bf16 = ov; g.ldc = (long)H * D_V; g.c_bstride = D_V;
    if (launch_gemm_tc(g, false, st, err) != cudaSuccess) return MLA_ERR_CUDA;

    // y = o_v W_O^T (k-splits reduced inside their cluster when the device holds every
    // tile's cluster at once, else partials and a finalize launch)
    g = GemmParams{};
    g.A = ov; g.lda = (long)H * D_V; g.B = w_o; g.ldb = (long)H * D_V;
    g.M = B; g.N = d_model; g.K = H * D_V; g.batch = 1;
    int per_c = 0, bn_c = 0;
    const int s_c = gemm_cluster_plan(B, d_model, H * D_V, &per_c, &bn_c);
    if (s_c > 0) {
        g.k_splits = s_c; g.k_per_split = per_c; g.c_bf16 = y; g.ldc = d_model;
        return cuda_status(launch_gemm_tc_cluster(g, bn_c, nullptr, st, err));
    }
    g.k_splits = L.s2; g.k_per_split = L.per2; g.c_part = part;
    if (launch_gemm_tc(g, false, st, err) != cudaSuccess) return MLA_ERR_CUDA;
    return cuda_status(launch_reduce_bf16(part, L.s2, 1, B, d_model, y, d_model, 0, st));
}

mla_status_t mla_projection_launches(int B, int d_model, int q_lora, int H, int *append,
                                     int *absorb_q, int *out_absorb, int *append_absorb_q) {
    if (B < 1 || B > 4096 || d_model < 64 || d_model % 64 || q_lora < 64 || q_lora % 64)
        return MLA_ERR_INVALID_ARG;
    if (!heads_ok(H)) return MLA_ERR_UNSUPPORTED;
    int per = 0;
    if (append) *append = gemm_cluster_plan(B, D_QK, d_model, &per, nullptr) > 0 ? 1 : 2;
    if (absorb_q)
        *absorb_q = (gemm_cluster_plan(B, q_lora, d_model, &per, nullptr) > 0 ? 1 : 2) +
                    (B <= 128 ? 1 : 3) + 1;
    if (out_absorb) *out_absorb = 1 + (gemm_cluster_plan(B, d_model, H * D_V, &per, nullptr) > 0 ? 1 : 2);
    if (append_absorb_q) {
        const int rest = (B <= 128 ? 1 : 3) + 1;  // q_nope / q_rope, then W_UK
        if (gemm_cluster_fits_dq_append(B, d_model, q_lora))
            *append_absorb_q = 1 + rest;
        else
            *append_absorb_q = (gemm_cluster_plan(B, D_QK, d_model, &per, nullptr) > 0 ? 1 : 2) +
                               (gemm_cluster_plan(B, q_lora, d_model, &per, nullptr) > 0 ? 1 : 2) +
                               rest;
    }
    return MLA_OK;
}

// -------------------------------------------------------------- status

mla_status_t mla_clear_device_status(void *workspace, mla_stream_t stream) {
    if (!workspace) return MLA_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(workspace, 0, 8, S(stream)));
}

mla_status_t mla_check_device_status(void *workspace, mla_stream_t stream) {
    if (!workspace) return MLA_ERR_INVALID_ARG;
    uint32_t word[2] = {0, 0};
    if (cudaMemcpyAsync(word, workspace, sizeof word, cudaMemcpyDeviceToHost, S(stream)) !=
        cudaSuccess)
        return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return MLA_ERR_CUDA;
    if (word[0] != 0) {
        if (cudaMemsetAsync(workspace, 0, 8, S(stream)) != cudaSuccess) return MLA_ERR_CUDA;
        if (cudaStreamSynchronize(S(stream)) != cudaSuccess) return MLA_ERR_CUDA;
    }
    return static_cast<mla_status_t>(word[0]);
}

}  // extern "C"
