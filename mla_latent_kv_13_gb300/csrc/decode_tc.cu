// decode_tc.cu -- absorbed MLA decode attention on the sm_100-family tensor cores
// (tcgen05 + TMEM), fed by TMA, one 2-CTA thread-block cluster per work item.
//
// Work item = (sequence b, token range s); with the balanced schedule a cluster runs the
// segments of one equal share of all sequences' tiles in turn. All heads of a sequence score the same
// latent cache rows [c_kv (512) | k_rope (64)], so the 128 head rows form the M=128
// side of both products and a 64-token cache tile the N (scores) or K (output) side:
//   S   = Q [128 x 576] . K^T [576 x 64]      (scores)
//   O  += P [128 x 64]  . V   [64 x 512]      (latent output, V = c_kv part)
// The fp32 accumulator O [128 x 512] alone fills a whole SM's tensor memory, so the
// two CTAs of a cluster split the latent columns: CTA r stages only its columns of
// each tile -- r = 0: c_kv[0:256); r = 1: c_kv[256:512) and k_rope -- computes the
// partial scores over them, swaps the 128 x 64 fp32 partial with its peer through
// distributed shared memory (bulk copies), and both CTAs then run the same softmax on
// the same full scores (bit-identical, since fp32 addition commutes) and accumulate
// their own 256 output columns. No cache byte is read twice and no product is
// computed twice; the only duplicated work is the (cheap) softmax.
//
// Roles per CTA (192 threads): warp 0 issues TMA loads (one elected lane); warp 1
// allocates TMEM and issues tcgen05.mma / tcgen05.commit (one elected lane); warps
// 2-5 (thread = head row = TMEM lane) load Q into TMEM, combine the two partial
// scores, run the online softmax in the exp2 domain, write P (bf16) into TMEM and
// finish the output. The exchange is a ping-pong over two 32 KB buffers per CTA: the
// peer's partial of tile k lands in buffer (k+1) % 2; once a warp has read its 32 rows
// of it, it overwrites them with its own partial of tile k+1 and bulk-copies them into
// the peer's buffer k % 2 -- which the peer emptied before it sent tile k. Arrival of
// data is the only signal: a buffer is always free by the time a copy targets it. The
// exchange (64 fp32 per head row per tile, ~20 B/clk of distributed shared memory per
// SM) thus runs one tile ahead on the copy engine, overlapping the softmax of the
// current tile, and each warp ships its own rows without waiting for the others.
// Both products read their A operand (Q, P) from TMEM and their B operand (the
// cache tile, 128-byte swizzled as TMA wrote it) from shared memory. The running maximum
// is only raised (and O rescaled in TMEM) when a score exceeds it by more than 2^8,
// so after the first tile of a sequence O is almost never touched between MMAs.
// Every mbarrier wait is bounded (about one second); a wait that gives up records
// MLA_ERR_TIMEOUT in the error word and the CTA drains and exits.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mla {

namespace {

using namespace sm100;

#ifndef MLA_DECODE_STAGES
#define MLA_DECODE_STAGES 4
#endif

constexpr int TOK = 64;
constexpr int NS = MLA_DECODE_STAGES;        // cache-tile stages
constexpr int KVCH = 64 * 128;               // one tile chunk: 64 tokens x 64 bf16 (8 KB)
constexpr int MAXCH = 5;                     // rank 1 stages 5 chunks (4 latent + rope)
constexpr int KV_OFF = 0;
constexpr int KV_STAGE = MAXCH * KVCH;       // 40960
constexpr int XROW = 256;                    // exchange row: 64 fp32, 16-byte chunks XOR-swizzled
constexpr int XQ = 32 * XROW;                // the 32 rows of one warp (8 KB)
constexpr int XBUF = 4 * XQ;                 // 32768
constexpr int X_OFF = KV_OFF + NS * KV_STAGE;  // two exchange buffers (ping-pong)
constexpr int BAR_OFF = X_OFF + 2 * XBUF;
constexpr int NBAR = 24;
constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
constexpr int SMEM_USED = MISC_OFF + 64;
constexpr int SMEM_TOTAL = SMEM_USED + 1024;  // slack to align the base to 1024 B

constexpr int NTHREADS = 192;                // 6 warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 0;                 // O: fp32 columns [0, 256)
constexpr uint32_t TM_S = 256;               // S: fp32 columns [256, 320)
constexpr uint32_t TM_Q = 320;               // Q: bf16 pairs, columns [320, 480)
constexpr uint32_t TM_P = 480;               // P: bf16 pairs, columns [480, 512)
constexpr uint64_t WAIT_NS = 1000000000ull;  // bounded waits: 1 s
constexpr uint64_t DRAIN_NS = 200000000ull;
constexpr float TAU = 8.0f;                  // lazy-rescale threshold (log2 units)
constexpr int PF_DIST = 4;                   // tiles prefetched into L2 beyond the stage ring

constexpr uint32_t IDESC_S = idesc_bf16(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, false, true);

static_assert(SMEM_TOTAL <= 232448, "shared memory budget");
static_assert(X_OFF >= KV_OFF + NS * KV_STAGE && BAR_OFF >= X_OFF + 2 * XBUF &&
                  MISC_OFF >= BAR_OFF + NBAR * 8,
              "shared-memory regions must not overlap");
static_assert(X_OFF % 16 == 0 && XQ % 16 == 0, "bulk-copy alignment");
static_assert((BAR_OFF % 8) == 0, "mbarrier alignment");

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
__device__ __forceinline__ float4 ld_shared_v4f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Wait that ignores the abort flag: used only to drain copies before exit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return;
    uint64_t t0 = globaltimer_ns();
    while (!mbar_test(bar, parity))
        if (globaltimer_ns() - t0 > DRAIN_NS) return;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap map_kv, DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sb - raw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int H = p.H;
    const int nch = rank == 0 ? 4 : 5;  // 64-column chunks of Q and of each tile owned here

    const uint32_t bar = sb + BAR_OFF;
    auto kv_full = [&](int s) { return bar + 8u * s; };
    auto kv_empty = [&](int s) { return bar + 8u * (NS + s); };
    const uint32_t q_ready = bar + 8u * (2 * NS);
    const uint32_t s_full = q_ready + 8;
    const uint32_t s_free = q_ready + 16;
    const uint32_t p_full = q_ready + 24;
    const uint32_t pv_done = q_ready + 32;
    const uint32_t mma_drain = q_ready + 40;
    // the peer's partial scores of the rows of warp quadrant q have landed in buffer x
    auto recv_full = [&](int q, int x) { return q_ready + 48 + 8u * (2 * q + x); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + MISC_OFF + 4);

    auto init_barriers = [&]() {
        for (int s = 0; s < NS; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        mbar_init(q_ready, 4);
        mbar_init(s_full, 1);
        mbar_init(s_free, 4);
        mbar_init(p_full, 4);
        mbar_init(pv_done, 1);
        mbar_init(mma_drain, 1);
        for (int k = 0; k < 8; ++k) mbar_init(recv_full(k >> 1, k & 1), 1);
        fence_mbar_init();
    };
    if (tid == 0) {
        init_barriers();
        *abort_flag = 0;
    }
    if (warp == 0 && lane == 0) tma_prefetch_map(&map_kv);
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers exist before any remote operation
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_launch_dependents();
    grid_dependency_wait();  // q, the cache rows and the schedule come from predecessor kernels

    // ---- work: one (sequence, token range) per cluster, or, with the balanced
    // schedule, the segments of this cluster's equal share of the concatenated tiles
    const bool sched = p.tile_start != nullptr;
    const int cl = blockIdx.x >> 1;
    int P = gridDim.x >> 1;
    long T = 0, r0 = 0, r1 = 0;
    int seg_b = 0;
    if (sched) {
        T = p.tile_start[p.B];
        if (T < P) P = static_cast<int>(T);  // as in the schedule: no empty ranges
        if (cl < P) {
            r0 = (cl * T) / P;
            r1 = ((cl + 1) * T) / P;
        }
        int lo = 0, hi = p.B - 1;  // largest b with tile_start[b] <= r0
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.tile_start[mid] <= r0) lo = mid;
            else hi = mid - 1;
        }
        seg_b = lo;
    }

    for (int seg = 0;; ++seg) {
    // -------- this segment: sequence b, tiles [t_begin, t_end), output slot
    int b, t_begin, t_end, part;
    bool direct;
    if (!sched) {
        if (seg > 0) break;
        const int item = blockIdx.x >> 1;
        b = item / p.num_splits;
        const int split = item % p.num_splits;
        t_begin = split * p.tiles_per_split;
        t_end = t_begin + p.tiles_per_split;  // clipped to the sequence below
        direct = p.num_splits == 1;
        part = b * p.num_splits + split;
    } else {
        while (seg_b < p.B && p.tile_start[seg_b + 1] == p.tile_start[seg_b]) ++seg_b;
        if (seg_b >= p.B || p.tile_start[seg_b] >= r1 || r0 >= r1) break;
        b = seg_b++;
        const long ts = p.tile_start[b], te = p.tile_start[b + 1];
        t_begin = static_cast<int>((r0 > ts ? r0 : ts) - ts);
        t_end = static_cast<int>((r1 < te ? r1 : te) - ts);
        direct = ts >= r0 && te <= r1;
        part = direct ? 0 : p.part_begin[b] + (cl - cluster_of_tile(ts, T, P));
    }
    int L = p.seqlens[b];
    if (L < 0 || L > p.max_blocks * TOK) {
        if (!sched && tid == 0 && rank == 0 && t_begin == 0)
            flag_error(p.err, MLA_ERR_OUT_OF_RANGE, b);
        L = L < 0 ? 0 : p.max_blocks * TOK;
    }
    const int ntiles = (L + TOK - 1) / TOK;
    t_end = min(ntiles, t_end);
    const int n = max(0, t_end - t_begin);
    const int32_t *btab = p.block_table + (size_t)b * p.max_blocks;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n > 0) {
            // Tiles beyond the shared-memory ring are prefetched into L2, so that a load
            // issued when a stage frees up is served from L2 rather than from HBM.
            auto prefetch = [&](int t) {
                if (t >= n) return;
                const int blk = btab[t_begin + t];
                if (blk < 0 || blk >= p.num_blocks) return;
                for (int c = 0; c < nch; ++c)
                    tma_prefetch_l2_2d(&map_kv, 64 * (4 * rank + c), blk * TOK);
            };
            for (int t = NS; t < NS + PF_DIST; ++t) prefetch(t);
            int issued = 0;
            for (int i = 0; i < n; ++i) {
                const int s = i % NS;
                if (!mbar_wait(kv_empty(s), ((i / NS) & 1) ^ 1, abort_flag, WAIT_NS)) break;
                const int blk = btab[t_begin + i];
                if (blk >= 0 && blk < p.num_blocks) {
                    mbar_arrive_expect_tx(kv_full(s), nch * KVCH);
                    for (int c = 0; c < nch; ++c)
                        tma_load_2d(sb + KV_OFF + s * KV_STAGE + c * KVCH, &map_kv, kv_full(s),
                                    64 * (4 * rank + c), blk * TOK);
                } else {
                    if (rank == 0) flag_error(p.err, MLA_ERR_OUT_OF_RANGE, b);
                    mbar_arrive(kv_full(s));  // no data: the consumers mask the tile
                }
                issued = i + 1;
                if (i >= NS) prefetch(i + PF_DIST);
            }
            // copies still in flight must land before this CTA may exit
            for (int i = max(0, issued - NS); i < issued; ++i)
                drain_wait(kv_full(i % NS), (i / NS) & 1);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA
        if (lane == 0 && n > 0) {
            auto issue_s = [&](int i) {
                const uint32_t kv = sb + KV_OFF + (i % NS) * KV_STAGE;
                for (int c = 0; c < nch; ++c)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_ts(tmem + TM_S, tmem + TM_Q + 32 * c + 8 * kk,
                                  sdesc_sw128(kv + c * KVCH + kk * 32, 16, 1024), IDESC_S,
                                  (c | kk) != 0);
                tc_commit(s_full);
            };
            // Scores of tile k need its cache tile (kv_full) and the S columns back from
            // the softmax (s_free of tile k-1); the output product of tile i needs P(i)
            // (p_full). Issue whichever is ready first, so that a tile still in flight
            // from HBM never holds up the output product of an earlier tile.
            bool ok = mbar_wait(q_ready, 0, abort_flag, WAIT_NS);
            if (ok) tc_fence_after();
            int s_next = 0, pv_next = 0;
            uint64_t t_last = globaltimer_ns();
            uint32_t spins = 0;
            while (ok && pv_next < n) {
                if (s_next < n && mbar_test(kv_full(s_next % NS), (s_next / NS) & 1) &&
                    (s_next == 0 || mbar_test(s_free, (s_next - 1) & 1))) {
                    tc_fence_after();
                    issue_s(s_next);
                    ++s_next;
                    t_last = globaltimer_ns();
                    continue;
                }
                if (pv_next < s_next && mbar_test(p_full, pv_next & 1)) {
                    tc_fence_after();
                    const int i = pv_next;
                    const uint32_t kv = sb + KV_OFF + (i % NS) * KV_STAGE;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_ts(tmem + TM_O, tmem + TM_P + 8 * kk,
                                  sdesc_sw128(kv + kk * 2048, KVCH, 1024), IDESC_PV,
                                  (i > 0 || kk > 0));
                    tc_commit(kv_empty(i % NS));
                    tc_commit(pv_done);
                    ++pv_next;
                    t_last = globaltimer_ns();
                    continue;
                }
                if ((++spins & 63) == 0) {
                    if (*abort_flag) ok = false;
                    else if (globaltimer_ns() - t_last > WAIT_NS) {
                        *abort_flag = 1;
                        ok = false;
                    }
                }
            }
            // every MMA this thread issued has finished before TMEM is released
            tc_commit(mma_drain);
            drain_wait(mma_drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- softmax / output
        const int wq = warp & 3;
        const int row = wq * 32 + lane;  // head row == TMEM lane
        const bool live_row = row < H;
        // row = (query token t, head): token t of s_q sees the rows j < L - (s_q - 1 - t)
        const int back = live_row ? p.s_q - 1 - row / p.hq : 0;
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const uint32_t xrow = row * XROW;
        // rows of this warp that hold a head: only those are exchanged (both CTAs agree)
        const int nlive = min(32, max(0, H - wq * 32));
        const uint32_t xbytes = static_cast<uint32_t>(nlive) * XROW;
        const uint32_t xq = sb + X_OFF + wq * XQ;            // + XBUF for buffer 1
        const uint32_t xq_peer = mapa(xq, peer);
        const uint32_t recv_peer = mapa(recv_full(wq, 0), peer);  // + 8 for buffer 1
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        // waits are warp-uniform: a lane that gives up takes its whole warp with it
        auto wait_w = [&](uint32_t bar_, uint32_t par) {
            return __all_sync(0xffffffffu, mbar_wait(bar_, par, abort_flag, WAIT_NS));
        };
        auto wait_wc = [&](uint32_t bar_, uint32_t par) {
            return __all_sync(0xffffffffu, mbar_wait<true>(bar_, par, abort_flag, WAIT_NS));
        };

        if (n > 0) {
            // Q rows of this CTA's columns into TMEM (A operand of the score product):
            // rank 0: q_lat[0:256); rank 1: q_lat[256:512) and q_rope. Rows >= H are 0.
            const uint4 *qsrc =
                reinterpret_cast<const uint4 *>(p.q_lat + ((size_t)b * H + row) * D_C + 256 * rank);
            const uint4 *rsrc =
                reinterpret_cast<const uint4 *>(p.q_rope + ((size_t)b * H + row) * D_ROPE);
            for (int c = 0; c < nch; ++c) {
                uint32_t r[32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (live_row) v = c < 4 ? qsrc[8 * c + k] : rsrc[k];
                    r[4 * k] = v.x;
                    r[4 * k + 1] = v.y;
                    r[4 * k + 2] = v.z;
                    r[4 * k + 3] = v.w;
                }
                tmem_st32(tl + TM_Q + 32 * c, r);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        }

        // Read this CTA's partial scores of tile k out of TMEM (releasing the S buffer),
        // stage this warp's rows of them in buffer k % 2 (the peer's tile k-1 there has
        // been read) and copy them into the peer's buffer (k+1) % 2.
        uint32_t own[64];
        auto stage_partial = [&](int k) -> bool {
            if (!wait_w(s_full, k & 1)) return false;
            tc_fence_after();
            tmem_ld32(tl + TM_S, *reinterpret_cast<uint32_t(*)[32]>(&own[0]));
            tmem_ld32(tl + TM_S + 32, *reinterpret_cast<uint32_t(*)[32]>(&own[32]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
            if (nlive > 0) {
                const uint32_t buf = (k & 1) * XBUF;
                const uint32_t dst = sb + X_OFF + buf + xrow;
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    st_shared_v4(dst + ((c ^ (row & 7)) << 4), own[4 * c], own[4 * c + 1],
                                 own[4 * c + 2], own[4 * c + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const uint32_t nb = XBUF - buf;  // the peer's buffer (k+1) % 2
                    bulk_copy_to_peer(xq_peer + nb, xq + buf, xbytes,
                                      recv_peer + 8u * ((k + 1) & 1));
                    bulk_commit();
                }
            }
            return true;
        };

        if (n > 0) ok = stage_partial(0);
        int blk_next = n > 0 ? btab[t_begin] : 0;  // block ids are fetched one tile ahead
        for (int i = 0; ok && i < n; ++i) {
            const int tile = t_begin + i;
            const int blk = blk_next;
            if (i + 1 < n) blk_next = btab[tile + 1];
            float s[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) s[j] = __uint_as_float(own[j]);
            // the peer's partial of tile i (buffer (i+1) % 2) -> full scores
            if (nlive > 0) {
                const int x = (i + 1) & 1;
                if (lane == 0) mbar_arrive_expect_tx(recv_full(wq, x), xbytes);
                if (!(ok = wait_wc(recv_full(wq, x), (i >> 1) & 1))) break;
                const uint32_t src = sb + X_OFF + x * XBUF + xrow;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float4 v = ld_shared_v4f(src + ((k ^ (row & 7)) << 4));
                    s[4 * k + 0] += v.x;
                    s[4 * k + 1] += v.y;
                    s[4 * k + 2] += v.z;
                    s[4 * k + 3] += v.w;
                }
                __syncwarp();
            }
            // then the next tile's partial into the rows just read, so its transfer
            // overlaps this softmax
            if (i + 1 < n && !(ok = stage_partial(i + 1))) break;

            // online softmax of tile i on this head row
            const bool blk_ok = blk >= 0 && blk < p.num_blocks;
            const int tvalid = blk_ok ? min(TOK, L - tile * TOK) : 0;  // valid tokens of the tile
            // columns this row keeps
            const int valid = live_row ? min(tvalid, max(0, L - back - tile * TOK)) : 0;
            if (valid < TOK) {
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    if (j >= valid) s[j] = -INFINITY;
            }
            float mx = s[0];
#pragma unroll
            for (int j = 1; j < 64; ++j) mx = fmaxf(mx, s[j]);
            mx *= p.scale_log2;  // scale > 0: the max of the scaled scores
            const bool raise = mx > m + TAU;
            if (__any_sync(0xffffffffu, raise)) {
                const float m_new = raise ? mx : m;
                const float alpha = raise ? fast_exp2(m - m_new) : 1.f;
                if (i > 0) {
                    // O holds tiles < i: wait until P.V of tile i-1 has landed, then rescale
                    if (!(ok = wait_w(pv_done, (i - 1) & 1))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tl + TM_O + 32 * c, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
                        tmem_st32(tl + TM_O + 32 * c, r);
                    }
                    tmem_st_wait();
                }
                l *= alpha;
                m = m_new;
            }
            // P = exp2(scale * s - m) as bf16 pairs for the P.V product
            uint32_t pk[32];
            const bool live = m != -INFINITY;
            const float nm = live ? -m : 0.f;
            float es = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float p0 = fast_exp2(fmaf(s[2 * j], p.scale_log2, nm));
                const float p1 = fast_exp2(fmaf(s[2 * j + 1], p.scale_log2, nm));
                pk[j] = pack_bf16x2(p0, p1);
                es += p0 + p1;
            }
            l += live ? es : 0.f;
            if (i > 0 && !(ok = wait_w(pv_done, (i - 1) & 1))) break;  // P columns free
            tmem_st32(tl + TM_P, pk);
            // rows past the valid tokens (the whole tile if its block is bad) may hold
            // stale or poisoned data: zero them in the four chunks P.V reads, since
            // 0 * NaN would still poison the product
            if (tvalid < TOK) {
                const uint32_t st = sb + KV_OFF + (i % NS) * KV_STAGE;
                const int nchunks = (TOK - tvalid) * 32;  // 16-byte chunks: rows x 4 x 8
                for (int e = row; e < nchunks; e += 128) {
                    const int r = tvalid + (e >> 5), c = (e >> 3) & 3, k = e & 7;
                    st_shared_v4(st + c * KVCH + r * 128 + k * 16, 0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }

        // ------------------------------------------------------------- output
        const int col0 = 256 * rank;
        if (n > 0 && ok && wait_w(pv_done, (n - 1) & 1)) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t r[32];
                tmem_ld32(tl + TM_O + 32 * c, r);
                tmem_ld_wait();
                if (row < H) {
                    if (direct) {
                        uint4 *dst = reinterpret_cast<uint4 *>(
                            p.out + ((size_t)b * H + row) * D_C + col0 + 32 * c);
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
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(
                            p.o_part + ((size_t)part * H + row) * D_C + col0 + 32 * c);
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            dst[k] = make_float4(__uint_as_float(r[4 * k]) * inv,
                                                 __uint_as_float(r[4 * k + 1]) * inv,
                                                 __uint_as_float(r[4 * k + 2]) * inv,
                                                 __uint_as_float(r[4 * k + 3]) * inv);
                    }
                }
            }
        } else if (row < H) {
            // empty range (or aborted): zero output, lse = -inf
            if (direct) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((size_t)b * H + row) * D_C + col0);
                for (int k = 0; k < 32; ++k) dst[k] = make_uint4(0u, 0u, 0u, 0u);
            } else {
                float4 *dst = reinterpret_cast<float4 *>(
                    p.o_part + ((size_t)part * H + row) * D_C + col0);
                for (int k = 0; k < 64; ++k) dst[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            l = 0.f;
        }
        if (rank == 0 && row < H) {
            const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
            if (direct)
                p.lse[(size_t)b * H + row] = lse;
            else
                p.lse_part[(size_t)part * H + row] = lse;
        }
    }

    // -------- end of segment: every copy into this CTA has landed (each was waited for),
    // our own copies have read their rows, every role is idle; then barriers restart
    if (warp >= 2 && lane == 0) bulk_wait_read_all();
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (!sched || *abort_flag) break;
    if (tid == 0) init_barriers();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    }  // segments

    if (tid == 0 && *abort_flag) flag_error(p.err, MLA_ERR_TIMEOUT, blockIdx.x);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no remote access into this CTA after this point
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

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

// Row-major bf16 matrix [rows][cols] (row pitch = cols) as a 2-D tensor map with
// 128-byte swizzled boxes of box_rows x 64 columns.
bool encode_bf16_2d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                    uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int decode_tc_cluster_slots() {
    static int slots = 0;
    if (slots > 0) return slots;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * 1024, 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_TOTAL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_TOTAL) == cudaSuccess &&
        cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel, &cfg) == cudaSuccess && n > 0)
        slots = n;
    else
        slots = device_sm_count() / 2;
    return slots;
}

cudaError_t launch_decode_tc(const DecodeParams &p, int clusters, cudaStream_t stream) {
    CUtensorMap mkv;
    if (!encode_bf16_2d(&mkv, p.cache, D_QK, (uint64_t)p.num_blocks * TOK, TOK))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    dim3 grid(2 * clusters);
    return launch_pdl(decode_tc_kernel, grid, dim3(NTHREADS), SMEM_TOTAL, stream, mkv, p);
}

}  // namespace mla
