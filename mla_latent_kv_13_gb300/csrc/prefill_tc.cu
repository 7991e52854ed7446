// prefill_tc.cu -- causal attention of a prefill chunk in the expanded form on the
// sm_100-family tensor cores (tcgen05 + TMEM), fed by TMA.
//
// Chunked prefill is compute-bound, so the latent cache is projected back per head ("LLM
// inference: from the memory wall to the compute wall" §2.2) and ordinary multi-head
// attention runs over the prefix and the chunk: for head h and query i of the chunk
// (position prefix + i), keys j <= prefix + i,
//   s_j = scale * (q_nope . k_nope_j + q_rope . k_rope_j),  o = sum_j softmax(s)_j v_j.
// One CTA per (head, tile of 128 queries): Q [128 x 192] is staged once; K [128 keys x 192]
// and V [128 keys x 128] tiles stream through two shared-memory stages:
//   S  = Q . K^T   (M = 128 queries, N = 128 keys, K = 192; A and B from shared memory)
//   O += P . V     (M = 128, N = 128, K = 128 keys; A = P from TMEM, B = V, MN-major)
// with the online softmax (exp2 domain, lazy rescale as in decode) between them. S is
// double-buffered in TMEM, so the scores of tile t+1 are computed while the softmax works
// on tile t.
// Roles (192 threads): warp 0 TMA, warp 1 TMEM + MMA issue (converged, one elected lane
// issues through predicated instructions), warps 2-5 softmax/output (thread = query row =
// TMEM lane). Every wait is bounded (one second).
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mla {

namespace {

using namespace sm100;

constexpr int QT = 128;                      // queries per CTA
constexpr int KT = 128;                      // keys per tile
constexpr int CH = 128 * 128;                // one 64-column chunk of 128 rows (16 KB)
constexpr int Q_OFF = 0;                     // q_nope[0:64), q_nope[64:128), q_rope
constexpr int NSTG = 2;
constexpr int K_CH = 3;                      // k_nope[0:64), k_nope[64:128), k_rope
constexpr int V_CH = 2;                      // v[0:64), v[64:128)
constexpr int STG = (K_CH + V_CH) * CH;      // 80 KB
constexpr int STG_OFF = Q_OFF + 3 * CH;
constexpr int BAR_OFF = STG_OFF + NSTG * STG;
constexpr int NBAR = 16;
constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
constexpr int SMEM_TOTAL = MISC_OFF + 64 + 1024;
constexpr int NTHREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 0;                 // O: fp32 [0, 128)
constexpr uint32_t TM_S = 128;               // S: fp32 [128, 256) and [256, 384)
constexpr uint32_t TM_P = 384;               // P: bf16 pairs [384, 448)
constexpr uint64_t WAIT_NS = 1000000000ull;
constexpr float TAU = 8.0f;

constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 128, false, true);

static_assert(SMEM_TOTAL <= 232448, "shared memory budget");
static_assert(STG_OFF % 1024 == 0 && STG % 1024 == 0, "swizzle atoms");

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
    uint64_t t0 = globaltimer_ns();
    while (!mbar_test(bar, parity))
        if (globaltimer_ns() - t0 > 200000000ull) return;
}

struct PrefillArgs {
    int C, T, H, prefix;
    float scale_log2;
    uint16_t *out;  // [C][H][128]
    float *lse;     // [C][H]
    uint32_t *err;
};

__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap m_qn, const __grid_constant__ CUtensorMap m_qr,
                      const __grid_constant__ CUtensorMap m_kn, const __grid_constant__ CUtensorMap m_kr,
                      const __grid_constant__ CUtensorMap m_v, PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sb - raw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y;
    const int i0 = blockIdx.x * QT;
    // keys the tile's last query sees: [0, prefix + min(i0 + 127, C - 1)]
    const int last_key = a.prefix + min(i0 + QT - 1, a.C - 1);
    const int nkt = last_key / KT + 1;

    const uint32_t bar = sb + BAR_OFF;
    auto kv_full = [&](int s) { return bar + 8u * s; };
    auto kv_empty = [&](int s) { return bar + 8u * (NSTG + s); };
    const uint32_t q_full = bar + 8u * (2 * NSTG);
    const uint32_t p_full = q_full + 8, pv_done = q_full + 16, mma_drain = q_full + 24;
    // S buffer x (tiles t with t % 2 == x): computed / read out by the softmax
    auto s_full = [&](int x) { return q_full + 32 + 8u * x; };
    auto s_free = [&](int x) { return q_full + 48 + 8u * x; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + MISC_OFF + 4);

    if (tid == 0) {
        for (int s = 0; s < NSTG; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        mbar_init(q_full, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(s_free(x), 4);
        }
        mbar_init(p_full, 4);
        mbar_init(pv_done, 1);
        mbar_init(mma_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&m_qn);
        tma_prefetch_map(&m_kn);
        tma_prefetch_map(&m_v);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_launch_dependents();
    grid_dependency_wait();  // q, k, v and the gathered rows come from predecessor kernels

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, 3 * CH);
            tma_load_3d(sb + Q_OFF, &m_qn, q_full, 0, h, i0);
            tma_load_3d(sb + Q_OFF + CH, &m_qn, q_full, 64, h, i0);
            tma_load_3d(sb + Q_OFF + 2 * CH, &m_qr, q_full, 0, h, i0);
            int issued = 0;
            for (int t = 0; t < nkt; ++t) {
                const int s = t % NSTG;
                if (!mbar_wait(kv_empty(s), ((t / NSTG) & 1) ^ 1, abort_flag, WAIT_NS)) break;
                const uint32_t st = sb + STG_OFF + s * STG;
                const int j0 = t * KT;
                mbar_arrive_expect_tx(kv_full(s), STG);
                tma_load_3d(st, &m_kn, kv_full(s), 0, h, j0);
                tma_load_3d(st + CH, &m_kn, kv_full(s), 64, h, j0);
                tma_load_2d(st + 2 * CH, &m_kr, kv_full(s), 0, j0);
                tma_load_3d(st + 3 * CH, &m_v, kv_full(s), 0, h, j0);
                tma_load_3d(st + 4 * CH, &m_v, kv_full(s), 64, h, j0);
                issued = t + 1;
            }
            drain(q_full, 0);
            for (int t = max(0, issued - NSTG); t < issued; ++t) drain(kv_full(t % NSTG), (t / NSTG) & 1);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA
        // The whole warp runs the issue loop (decisions from lane 0's view of the barriers,
        // non-suspending polls) and one elected lane issues through predicated
        // instructions: a tcgen05.mma issued by a lone lane of a diverged warp costs that
        // thread more than the tensor pipe's own time per instruction.
        {
            const bool leader = elect_one();
            auto lane0 = [&](bool v) { return __shfl_sync(0xffffffffu, v, 0); };
            bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag, WAIT_NS));
            if (ok) tc_fence_after();
            int s_next = 0, pv_next = 0;
            uint64_t t_idle = 0;  // start of the current idle stretch (0: progress since)
            uint32_t spins = 0;
            while (ok && pv_next < nkt) {
                // S(t) into buffer t % 2 once the softmax has read tile t-2 out of it
                if (lane0(s_next < nkt && mbar_poll(kv_full(s_next % NSTG), (s_next / NSTG) & 1) &&
                          (s_next < 2 || mbar_poll(s_free(s_next & 1), ((s_next >> 1) - 1) & 1)))) {
                    tc_fence_after();
                    const uint32_t st = sb + STG_OFF + (s_next % NSTG) * STG;
                    const uint32_t ts = tmem + TM_S + 128 * (s_next & 1);
#pragma unroll
                    for (int c = 0; c < K_CH; ++c)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma_if(leader, ts, sdesc_sw128(sb + Q_OFF + c * CH + kk * 32, 16, 1024),
                                      sdesc_sw128(st + c * CH + kk * 32, 16, 1024), IDESC_S,
                                      (c | kk) != 0);
                    tc_commit_if(leader, s_full(s_next & 1));
                    __syncwarp();
                    ++s_next;
                    t_idle = 0;
                    continue;
                }
                if (lane0(pv_next < s_next && mbar_poll(p_full, pv_next & 1))) {
                    tc_fence_after();
                    const uint32_t vt = sb + STG_OFF + (pv_next % NSTG) * STG + 3 * CH;
#pragma unroll
                    for (int kk = 0; kk < KT / 16; ++kk)
                        tc_mma_ts_if(leader, tmem + TM_O, tmem + TM_P + 8 * kk,
                                     sdesc_sw128(vt + kk * 2048, CH, 1024), IDESC_PV,
                                     (pv_next > 0 || kk > 0));
                    tc_commit_if(leader, kv_empty(pv_next % NSTG));
                    tc_commit_if(leader, pv_done);
                    __syncwarp();
                    ++pv_next;
                    t_idle = 0;
                    continue;
                }
                if ((++spins & 63) == 0) {
                    const uint64_t now = globaltimer_ns();
                    if (t_idle == 0) t_idle = now;
                    bool stop = *abort_flag != 0;
                    if (!stop && now - t_idle > WAIT_NS) {
                        if (lane == 0) *abort_flag = 1;
                        stop = true;
                    }
                    ok = !lane0(stop);
                }
            }
            if (leader) {
                tc_commit(mma_drain);
                drain(mma_drain, 0);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- softmax / output
        const int wq = warp & 3;
        const int row = wq * 32 + lane;  // query row == TMEM lane
        const int i = i0 + row;          // query index in the chunk
        const bool live = i < a.C;
        const int limit = live ? a.prefix + i : -1;  // last key this query sees
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        auto wait_w = [&](uint32_t bar_, uint32_t par) {
            return __all_sync(0xffffffffu, mbar_wait(bar_, par, abort_flag, WAIT_NS));
        };
        for (int t = 0; ok && t < nkt; ++t) {
            if (!(ok = wait_w(s_full(t & 1), (t >> 1) & 1))) break;
            tc_fence_after();
            uint32_t raw_s[128];
            const uint32_t ts = tl + TM_S + 128 * (t & 1);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld32(ts + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&raw_s[32 * c]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free(t & 1));
            const int vis = min(KT, max(0, limit - t * KT + 1));  // visible keys of the tile
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < KT; ++c)
                if (c < vis) mx = fmaxf(mx, __uint_as_float(raw_s[c]));
            mx *= a.scale_log2;
            const bool raise = mx > m + TAU;
            if (__any_sync(0xffffffffu, raise)) {
                const float m_new = raise ? mx : m;
                const float alpha = raise ? fast_exp2(m - m_new) : 1.f;
                if (t > 0) {
                    if (!(ok = wait_w(pv_done, (t - 1) & 1))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tl + TM_O + 32 * c, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
                        tmem_st32(tl + TM_O + 32 * c, r);
                    }
                    tmem_st_wait();
                }
                l *= alpha;
                m = m_new;
            }
            // P = exp2(scale * s - m) as bf16 pairs, 0 past the visible keys
            const float nm = m != -INFINITY ? -m : 0.f;
            uint32_t pk[64];
            float es = 0.f;
#pragma unroll
            for (int k = 0; k < 64; ++k) {
                const float p0 = 2 * k < vis
                                     ? fast_exp2(fmaf(__uint_as_float(raw_s[2 * k]), a.scale_log2, nm))
                                     : 0.f;
                const float p1 = 2 * k + 1 < vis
                                     ? fast_exp2(fmaf(__uint_as_float(raw_s[2 * k + 1]), a.scale_log2, nm))
                                     : 0.f;
                pk[k] = pack_bf16x2(p0, p1);
                es += p0 + p1;
            }
            l += es;
            if (t > 0 && !(ok = wait_w(pv_done, (t - 1) & 1))) break;  // P columns free
            tmem_st32(tl + TM_P, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            tmem_st32(tl + TM_P + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        // ------------------------------------------------------------- output
        if (ok && wait_w(pv_done, (nkt - 1) & 1)) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(tl + TM_O + 32 * c, r);
                tmem_ld_wait();
                if (live) {
                    uint4 *dst = reinterpret_cast<uint4 *>(
                        a.out + ((size_t)i * a.H + h) * D_NOPE + 32 * c);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_uint4(
                            pack_bf16x2(__uint_as_float(r[8 * k + 0]) * inv,
                                        __uint_as_float(r[8 * k + 1]) * inv),
                            pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv,
                                        __uint_as_float(r[8 * k + 3]) * inv),
                            pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv,
                                        __uint_as_float(r[8 * k + 5]) * inv),
                            pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv,
                                        __uint_as_float(r[8 * k + 7]) * inv));
                }
            }
            if (live)
                a.lse[(size_t)i * a.H + h] =
                    l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    }
    if (tid == 0 && *abort_flag) flag_error(a.err, MLA_ERR_TIMEOUT, blockIdx.x);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Cache rows of one sequence's first T positions, gathered contiguous: c_kv [T][512] and
// k_rope [T][64]. Out-of-range block ids are reported and their rows written as zeros.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t *cache, int num_blocks,
                                                          const int32_t *block_table,
                                                          int max_blocks, int T, uint16_t *ckv,
                                                          uint16_t *kr, uint32_t *err) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int j = blockIdx.x;  // position
    const int blk = j / BLOCK < max_blocks ? block_table[j / BLOCK] : -1;
    const bool ok = blk >= 0 && blk < num_blocks;
    if (!ok && threadIdx.x == 0) flag_error(err, MLA_ERR_OUT_OF_RANGE, j);
    // 576 bf16 = 72 chunks of 16 bytes: 64 for c_kv, 8 for k_rope
    for (int c = threadIdx.x; c < 72; c += blockDim.x) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (ok) v = reinterpret_cast<const uint4 *>(cache + ((size_t)blk * BLOCK + j % BLOCK) * D_QK)[c];
        if (c < 64) reinterpret_cast<uint4 *>(ckv + (size_t)j * D_C)[c] = v;
        else reinterpret_cast<uint4 *>(kr + (size_t)j * D_ROPE)[c - 64] = v;
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// bf16 tensor [rows][heads][d] (d innermost) as a 3-D map; boxes of 64 x 1 x 128 rows with
// 128-byte swizzle (one head's 128 rows of 64 elements: the layout of a 2-D 64 x 128 box).
bool map_3d(CUtensorMap *m, const void *base, uint64_t d, uint64_t heads, uint64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {d, heads, rows};
    cuuint64_t strides[2] = {d * 2, d * heads * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map_2d_rows(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gather_rows(const uint16_t *cache, int num_blocks, const int32_t *block_table,
                               int max_blocks, int T, uint16_t *ckv, uint16_t *kr, uint32_t *err,
                               cudaStream_t stream) {
    return launch_pdl(gather_rows_kernel, dim3(T), dim3(96), 0, stream, cache, num_blocks,
                      block_table, max_blocks, T, ckv, kr, err);
}

cudaError_t launch_prefill_tc(const uint16_t *q_nope, const uint16_t *q_rope,
                              const uint16_t *k_nope, const uint16_t *k_rope, const uint16_t *v,
                              int C, int T, int H, int prefix, float scale, uint16_t *out,
                              float *lse, uint32_t *err, cudaStream_t stream) {
    CUtensorMap mqn, mqr, mkn, mkr, mv;
    if (!map_3d(&mqn, q_nope, D_NOPE, H, C) || !map_3d(&mqr, q_rope, D_ROPE, H, C) ||
        !map_3d(&mkn, k_nope, D_NOPE, H, T) || !map_2d_rows(&mkr, k_rope, D_ROPE, T) ||
        !map_3d(&mv, v, D_V, H, T))
        return cudaErrorInvalidValue;
    PrefillArgs a{};
    a.C = C; a.T = T; a.H = H; a.prefix = prefix;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.out = out; a.lse = lse; a.err = err;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    dim3 grid((C + QT - 1) / QT, H);
    return launch_pdl(prefill_tc_kernel, grid, dim3(NTHREADS), SMEM_TOTAL, stream, mqn, mqr, mkn, mkr,
                      mv, a);
}

}  // namespace mla
