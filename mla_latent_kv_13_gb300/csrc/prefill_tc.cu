// prefill_tc.cu -- causal attention of a prefill chunk in the expanded form on the
// sm_100-family tensor cores (tcgen05 + TMEM), fed by TMA.
//
// Chunked prefill is compute-bound, so the latent cache is projected back per head ("LLM
// inference: from the memory wall to the compute wall" §2.2) and ordinary multi-head
// attention runs over the prefix and the chunk: for head h and query i of the chunk
// (position prefix + i), keys j <= prefix + i,
//   s_j = scale * (q_nope . k_nope_j + q_rope . k_rope_j),  o = sum_j softmax(s)_j v_j.
// One CTA per (head, 256 queries), as two tiles of 128 queries (A and B) that share the
// key/value tiles: Q [2 x 128 x 192] is staged once; K [128 keys x 192] tiles stream through
// two shared-memory stages and V [128 keys x 128] through one:
//   S_g  = Q_g . K^T   (M = 128 queries, N = 128 keys, K = 192; A and B from shared memory)
//   O_g += P_g . V     (M = 128, N = 128, K = 128 keys; A = P from TMEM, B = V, MN-major)
// with the online softmax (exp2 domain, lazy rescale as in decode) between them. Each tile
// has its own softmax warpgroup, O and S in TMEM, and P is written over the S columns it came
// from. The two tiles' products and softmaxes interleave ("ping-pong"): while one group
// turns its scores into P, the tensor pipe runs the other group's P.V and next scores, so
// neither the softmax (128 exponentials per row and tile, one warp per SMSP and group) nor
// the products wait for each other as a single tile does.
// Roles (320 threads): warp 0 TMA, warp 1 TMEM + MMA issue (converged, one elected lane
// issues through predicated instructions, whichever product is ready first), warps 2-5
// softmax/output of tile A and warps 6-9 of tile B (thread = query row = TMEM lane). Every
// wait is bounded (one second).
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mla {

namespace {

using namespace sm100;

constexpr int QT = 128;                      // queries per tile; a CTA holds tiles A and B
constexpr int KT = 128;                      // keys per tile
constexpr int CH = 128 * 128;                // one 64-column chunk of 128 rows (16 KB)
constexpr int QCH = 3;                       // q_nope[0:64), q_nope[64:128), q_rope
constexpr int K_CH = 3;                      // k_nope[0:64), k_nope[64:128), k_rope
constexpr int V_CH = 2;                      // v[0:64), v[64:128)
constexpr int NK = 2;                        // K stages (V has one)
constexpr int Q_OFF = 0;                     // Q of tile A, then of tile B
constexpr int K_OFF = Q_OFF + 2 * QCH * CH;
constexpr int V_OFF = K_OFF + NK * K_CH * CH;
constexpr int BAR_OFF = V_OFF + V_CH * CH;
constexpr int NBAR = 16;
constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
constexpr int SMEM_TOTAL = MISC_OFF + 64 + 1024;
constexpr int NTHREADS = 320;
constexpr uint32_t TMEM_COLS = 512;
// O of tile g: fp32 [128 g, 128 g + 128); S of tile g: fp32 [256 + 128 g, +128), its P
// (bf16 pairs) over the first 64 of those columns
constexpr uint32_t TM_O = 0, TM_S = 256;
constexpr uint64_t WAIT_NS = 1000000000ull;
constexpr float TAU = 8.0f;

constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 128, false, true);

static_assert(SMEM_TOTAL <= 232448, "shared memory budget");
static_assert(K_OFF % 1024 == 0 && V_OFF % 1024 == 0 && CH % 1024 == 0, "swizzle atoms");

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
    uint64_t t0 = globaltimer_ns();
    while (!mbar_test(bar, parity))
        if (globaltimer_ns() - t0 > 200000000ull) return;
}
// 16 consecutive 32-bit columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
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
    const int i0 = blockIdx.x * (2 * QT);
    // key tiles seen by query tile g: through the key of its last live query (none when
    // the tile holds no live query)
    auto tiles_of = [&](int g) {
        const int first = i0 + g * QT;
        return first >= a.C ? 0 : (a.prefix + min(first + QT - 1, a.C - 1)) / KT + 1;
    };
    const int ntile[2] = {tiles_of(0), tiles_of(1)};
    const int nk = max(ntile[0], ntile[1]);

    const uint32_t bar = sb + BAR_OFF;
    auto k_full = [&](int s) { return bar + 8u * s; };
    auto k_empty = [&](int s) { return bar + 8u * (NK + s); };
    const uint32_t v_full = bar + 8u * (2 * NK), v_empty = v_full + 8;
    const uint32_t q_full = v_full + 16, mma_drain = v_full + 24;
    auto s_full = [&](int g) { return v_full + 32 + 8u * g; };   // S_g(t) computed
    auto p_full = [&](int g) { return v_full + 48 + 8u * g; };   // P_g(t) in TMEM (4 warps)
    auto pv_done = [&](int g) { return v_full + 64 + 8u * g; };  // O_g += P_g(t) V(t) done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + MISC_OFF + 4);

    if (tid == 0) {
        for (int s = 0; s < NK; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
        }
        mbar_init(v_full, 1);
        mbar_init(v_empty, 1);
        mbar_init(q_full, 1);
        mbar_init(mma_drain, 1);
        for (int g = 0; g < 2; ++g) {
            mbar_init(s_full(g), 1);
            mbar_init(p_full(g), 4);
            mbar_init(pv_done(g), 1);
        }
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
        // K(0), K(1), V(0), then K(t + 1) before V(t): K(t + 1) frees with the scores of
        // tile t - 1, V(t) only with the products P.V of tile t - 1, which come later
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, 2 * QCH * CH);
            for (int g = 0; g < 2; ++g) {
                const uint32_t q = sb + Q_OFF + g * QCH * CH;
                tma_load_3d(q, &m_qn, q_full, 0, h, i0 + g * QT);
                tma_load_3d(q + CH, &m_qn, q_full, 64, h, i0 + g * QT);
                tma_load_3d(q + 2 * CH, &m_qr, q_full, 0, h, i0 + g * QT);
            }
            auto load_k = [&](int t) {
                const int s = t % NK;
                if (!mbar_wait(k_empty(s), ((t / NK) & 1) ^ 1, abort_flag, WAIT_NS)) return false;
                const uint32_t st = sb + K_OFF + s * K_CH * CH;
                const int j0 = t * KT;
                mbar_arrive_expect_tx(k_full(s), K_CH * CH);
                tma_load_3d(st, &m_kn, k_full(s), 0, h, j0);
                tma_load_3d(st + CH, &m_kn, k_full(s), 64, h, j0);
                tma_load_2d(st + 2 * CH, &m_kr, k_full(s), 0, j0);
                return true;
            };
            auto load_v = [&](int t) {
                if (!mbar_wait(v_empty, (t & 1) ^ 1, abort_flag, WAIT_NS)) return false;
                const int j0 = t * KT;
                mbar_arrive_expect_tx(v_full, V_CH * CH);
                tma_load_3d(sb + V_OFF, &m_v, v_full, 0, h, j0);
                tma_load_3d(sb + V_OFF + CH, &m_v, v_full, 64, h, j0);
                return true;
            };
            int ik = 0, iv = 0;  // tiles whose K / V loads were issued
            bool ok = true;
            for (int t = 0; ok && t < min(nk, NK); ++t)
                if ((ok = load_k(t))) ik = t + 1;
            if (ok && nk > 0 && (ok = load_v(0))) iv = 1;
            for (int t = 1; ok && t < nk; ++t) {
                if (t + 1 < nk) {
                    if (!(ok = load_k(t + 1))) break;
                    ik = t + 2;
                }
                if ((ok = load_v(t))) iv = t + 1;
            }
            drain(q_full, 0);
            for (int t = max(0, ik - NK); t < ik; ++t) drain(k_full(t % NK), (t / NK) & 1);
            if (iv > 0) drain(v_full, (iv - 1) & 1);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA
        // Per tile g, in order: S_g(0), P_g(0).V(0), S_g(1), ...; S_g(t + 1) overwrites the
        // columns P_g(t) sits in, so it waits for P_g(t).V(t). The two tiles' streams are
        // issued in whatever order their inputs become ready. A key or value tile is
        // released by the commit after the last product that reads it (the second tile to
        // use it, or the only one).
        const bool leader = elect_one();
        auto lane0 = [&](bool v) { return __shfl_sync(0xffffffffu, v, 0); };
        bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag, WAIT_NS));
        if (ok) tc_fence_after();
        int ns[2] = {0, 0}, np[2] = {0, 0};  // next S tile, next P.V tile, per query tile
        uint64_t t_idle = 0;
        uint32_t spins = 0;
        while (ok && (np[0] < ntile[0] || np[1] < ntile[1])) {
            bool progress = false;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const int o = g ^ 1;
                // P_g(t) . V(t)
                const int tp = np[g];
                if (tp < ns[g] &&
                    lane0(mbar_poll(p_full(g), tp & 1) && mbar_poll(v_full, tp & 1))) {
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < KT / 16; ++kk)
                        tc_mma_ts_if(leader, tmem + TM_O + 128 * g, tmem + TM_S + 128 * g + 8 * kk,
                                     sdesc_sw128(sb + V_OFF + kk * 2048, CH, 1024), IDESC_PV,
                                     (tp > 0 || kk > 0));
                    tc_commit_if(leader, pv_done(g));
                    if (np[o] > tp || tp >= ntile[o]) tc_commit_if(leader, v_empty);
                    __syncwarp();
                    ++np[g];
                    progress = true;
                }
                // S_g(t): its key tile loaded, its columns free (P_g(t - 1) . V(t - 1) done)
                const int ts = ns[g];
                if (ts < ntile[g] && ts == np[g] &&
                    lane0(mbar_poll(k_full(ts % NK), (ts / NK) & 1) &&
                          (ts == 0 || mbar_poll(pv_done(g), (ts - 1) & 1)))) {
                    tc_fence_after();
                    const uint32_t q = sb + Q_OFF + g * QCH * CH;
                    const uint32_t st = sb + K_OFF + (ts % NK) * K_CH * CH;
#pragma unroll
                    for (int c = 0; c < K_CH; ++c)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma_if(leader, tmem + TM_S + 128 * g,
                                      sdesc_sw128(q + c * CH + kk * 32, 16, 1024),
                                      sdesc_sw128(st + c * CH + kk * 32, 16, 1024), IDESC_S,
                                      (c | kk) != 0);
                    tc_commit_if(leader, s_full(g));
                    if (ns[o] > ts || ts >= ntile[o]) tc_commit_if(leader, k_empty(ts % NK));
                    __syncwarp();
                    ++ns[g];
                    progress = true;
                }
            }
            if (progress) {
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
        __syncwarp();
    } else {
        // ---------------------------------------------------- softmax / output
        const int g = (warp - 2) >> 2;   // warps 2-5: tile A, 6-9: tile B
        const int wq = warp & 3;         // TMEM lane quadrant of this warp
        const int row = wq * 32 + lane;  // query row == TMEM lane
        const int i = i0 + g * QT + row;  // query index in the chunk
        const bool live = i < a.C;
        const int limit = live ? a.prefix + i : -1;  // last key this query sees
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const uint32_t tO = tl + TM_O + 128 * g, tS = tl + TM_S + 128 * g;
        const int nt = ntile[g];
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        auto wait_w = [&](uint32_t bar_, uint32_t par) {
            return __all_sync(0xffffffffu, mbar_wait(bar_, par, abort_flag, WAIT_NS));
        };
        for (int t = 0; ok && t < nt; ++t) {
            if (!(ok = wait_w(s_full(g), t & 1))) break;
            tc_fence_after();
            const int vis = min(KT, max(0, limit - t * KT + 1));  // visible keys of the tile
            // pass 1: the row maximum over the visible keys (all four loads in flight)
            float mx = -INFINITY;
            {
                uint32_t r[128];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
                tmem_ld_wait();
                if (vis == KT) {  // every key visible (all but the diagonal tiles)
#pragma unroll
                    for (int k = 0; k < KT; ++k) mx = fmaxf(mx, __uint_as_float(r[k]));
                } else {
#pragma unroll
                    for (int k = 0; k < KT; ++k)
                        if (k < vis) mx = fmaxf(mx, __uint_as_float(r[k]));
                }
            }
            mx *= a.scale_log2;
            const bool raise = mx > m + TAU;
            if (__any_sync(0xffffffffu, raise)) {
                const float m_new = raise ? mx : m;
                const float alpha = raise ? fast_exp2(m - m_new) : 1.f;
                if (t > 0) {
                    if (!(ok = wait_w(pv_done(g), (t - 1) & 1))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tO + 32 * c, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
                        tmem_st32(tO + 32 * c, r);
                    }
                    tmem_st_wait();
                }
                l *= alpha;
                m = m_new;
            }
            // pass 2: P = exp2(scale * s - m) as bf16 pairs, 0 past the visible keys, over
            // the S columns already read (keys 32c.. become columns 16c.., behind the reads)
            const float nm = m != -INFINITY ? -m : 0.f;
            float es = 0.f;
#pragma unroll 1
            for (int c2 = 0; c2 < 2; ++c2) {  // 64 keys per load round
                uint32_t r[64];
                tmem_ld32(tS + 64 * c2, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                tmem_ld32(tS + 64 * c2 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                tmem_ld_wait();
                const bool full = vis >= 64 * c2 + 64;  // every key of this round visible
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int c = 2 * c2 + h2;
                    uint32_t pk[16];
                    if (full) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const float p0 = fast_exp2(fmaf(__uint_as_float(r[32 * h2 + 2 * k]), a.scale_log2, nm));
                            const float p1 =
                                fast_exp2(fmaf(__uint_as_float(r[32 * h2 + 2 * k + 1]), a.scale_log2, nm));
                            pk[k] = pack_bf16x2(p0, p1);
                            es += p0 + p1;
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const int j = 32 * c + 2 * k;
                            const float p0 = j < vis ? fast_exp2(fmaf(__uint_as_float(r[32 * h2 + 2 * k]),
                                                                      a.scale_log2, nm))
                                                     : 0.f;
                            const float p1 = j + 1 < vis ? fast_exp2(fmaf(__uint_as_float(r[32 * h2 + 2 * k + 1]),
                                                                          a.scale_log2, nm))
                                                         : 0.f;
                            pk[k] = pack_bf16x2(p0, p1);
                            es += p0 + p1;
                        }
                    }
                    tmem_st16(tS + 16 * c, pk);
                }
            }
            l += es;
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(g));
        }
        // ------------------------------------------------------------- output
        if (ok && nt > 0 && wait_w(pv_done(g), (nt - 1) & 1)) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                tmem_ld32(tO + 32 * c, r);
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
    dim3 grid((C + 2 * QT - 1) / (2 * QT), H);
    return launch_pdl(prefill_tc_kernel, grid, dim3(NTHREADS), SMEM_TOTAL, stream, mqn, mqr, mkn, mkr,
                      mv, a);
}

}  // namespace mla
