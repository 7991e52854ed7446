// decode_tc.cu -- absorbed MLA decode attention on the sm_100-family tensor cores
// (tcgen05 + TMEM), fed by TMA, one 2-CTA thread-block cluster per work item.
//
// Work item = (sequence b, token range s); with the balanced schedule a cluster runs the
// segments of its share of all sequences' tiles in turn (shares equal in tiles plus a fixed
// start-up cost per sequence). All heads of a sequence
// score the same latent cache rows [c_kv (512) | k_rope (64)], so the 128 head rows form
// the M = 128 side of both products:
//   S   = Q [128 x 576] . K^T [576 x tokens]   (scores)
//   O  += P [128 x tokens] . V [tokens x 512]  (latent output, V = c_kv part)
// The fp32 accumulator O [128 x 512] alone would fill a whole SM's tensor memory, so the
// two CTAs of a cluster split the output columns (CTA r keeps O[:, 256r : 256r+256]) and
// split each 64-token cache tile by tokens for the scores: CTA r scores tokens
// [32r, 32r+32) over all 576 columns. Each CTA therefore stages, per tile, its own 32
// tokens in full (9 chunks of 64 columns) and the peer's 32 tokens in its own 256 output
// columns (4 chunks); no partial score crosses the cluster. What does cross is the
// probability half: each CTA turns its 128 x 32 scores into P (bf16) against a running
// per-row reference and stores P with (reference, row sum) straight from registers into
// the peer's shared memory (st.async, completing bytes on the peer's mbarrier: 9 KB per
// tile each way); both CTAs then agree on the larger reference (rescaling whichever half
// was computed against the smaller one -- rare after the first tile, since the
// reference is only raised when a score exceeds it by more than 2^8) and run P . V over
// all 64 tokens for their own columns.
//
// Tensor memory (512 columns): O fp32 [0, 256), then S fp32 (one 32-column buffer, or two
// for at most 64 query rows, so that the scores of the next tile are computed while the
// softmax still works on this one), then Q as bf16 pairs of as many column chunks as fit
// (7 or 6); the remaining Q chunks (k_rope last) are read from shared memory. The chunks
// of a tile sit in three rings sized by how long they are held: the own tokens' own
// output columns (both products, 4 slots), the own tokens' other columns and k_rope
// (scores only, 2 slots) and the peer tokens' own output columns (P . V only, loaded late,
// 3 or 2 slots). P halves are double-buffered: the local half is the A operand of P . V
// for the own tokens, the received half for the peer's.
//
// Roles per CTA (224 threads): warp 0 loads the own tokens' chunks (TMA, one lane);
// warp 1 allocates TMEM and issues the score MMAs; warp 6 issues P . V and loads the
// peer tokens' chunks; warps 2-5 (thread = head row = TMEM lane) load Q, run the online
// softmax in the exp2 domain, exchange P and finish the output. Each MMA warp runs its
// loop converged and issues from one elected lane with a predicated instruction: a
// tcgen05.mma issued by a lone lane of a diverged warp costs that thread several times
// the tensor pipe's own time per instruction at these small N. P . V has its own warp
// because a warp issuing the 36 small score MMAs of a tile stays busy for about their
// execution time.
// Every mbarrier wait is bounded (about one second); a wait that gives up records
// MLA_ERR_TIMEOUT in the error word and the CTA drains and exits.
#include "common.cuh"
#include "fp8.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mla {

namespace {

using namespace sm100;

constexpr int TOK = 64;                       // tokens per cache tile (one page)
constexpr int HALF = 32;                      // tokens of a tile scored by each CTA
constexpr int CH = HALF * 128;                // one chunk: 32 tokens x 64 bf16 (4 KB)
constexpr int NOWN = 9;                       // own tokens: 8 c_kv chunks + k_rope
// The chunks of a tile live in three rings, by how long they are needed:
//   KV: own tokens x own output columns (4 chunks) -- both products, until P.V
//   K : own tokens x the other 4 c_kv chunks and k_rope (5 chunks) -- scores only
//   V : peer tokens x own output columns (4 chunks) -- P.V only, loaded later
constexpr int KV_SLOT = 4 * CH, K_SLOT = 5 * CH, V_SLOT = 4 * CH;
constexpr int QCH = 128 * 128;                // one Q chunk in smem: 128 rows x 128 B
constexpr int PGRP = 8 * 64 + 8 * 8;          // 8 rows: their 32 bf16 of P, then (reference, sum)
constexpr int PBUF = 16 * PGRP;               // P half of 128 rows with its row data (9 KB)
constexpr int PWARP = 4 * PGRP;               // the 32 rows of one warp (contiguous)
constexpr int NBAR = 56;
// MISC: TMEM address, abort flags, and the counts of remote operations exchanged when a
// pair stops early (byte offsets below)
constexpr int MISC_BYTES = 128;
constexpr int M_TMEM = 0, M_ABORT = 4, M_PEER_ABORT = 8, M_PEER_PV = 12, M_PEER_SENT = 16,
              M_SENT = 32, M_RECV = 48, M_PV = 64;
constexpr int EXP_SLOT = 64;                  // FP8: one slot's 64 row exponents (int8 each)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 0;                  // O: fp32 columns [0, 256)
// Q rows staged between segments in the idle rings and local P buffers (from KV_OFF up to
// the peer's P buffers, which stay untouched): one row (q_lat then q_rope) per 1168
// bytes, so that the 8 lanes of a 16-byte shared-memory access hit 8 bank groups
constexpr int QSTG = 2 * (D_C + D_ROPE) + 16;

// Two layouts of shared and tensor memory. TMEM holds O (256 columns), the scores S (32
// columns per buffer) and as many Q chunks as fit (32 columns each, bf16 pairs); the other
// Q chunks are A operands in shared memory, which cost the tensor pipe more per score MMA.
//   DS = true : two S buffers, so the next tile's scores are computed while the softmax
//               still reads this one; Q chunks 0..5 in TMEM, 6..8 in smem; V ring 2 slots.
//   DS = false: one S buffer; Q chunks 0..6 in TMEM, 7..8 in smem; V ring 3 slots.
// Measured (B = 128 x 8192 tokens at 128 heads; 32 x 32768 at 64): the double buffer
// takes the 64-row case from 271 to 257 us, but the 128-row case from 292 to 305 us, where
// the tensor pipe's time per tile (the extra shared-memory operand) sets the period. The
// host takes DS for at most 64 query rows.
template <bool DS> struct Layout {
    static constexpr int NSB = DS ? 2 : 1;    // S buffers
    static constexpr int NKV = 4, NK = 2;     // slots of the KV and K rings
    static constexpr int NV = DS ? 2 : 3;     // slots of the V ring
    static constexpr int NQT = DS ? 6 : 7;    // Q chunks held in TMEM (the rest in smem)
    static constexpr int NQS = NOWN - NQT;    // Q chunks in smem (the last ones, k_rope last)
    static constexpr int QS_OFF = 0;
    static constexpr int KV_OFF = QS_OFF + NQS * QCH;
    static constexpr int K_OFF = KV_OFF + NKV * KV_SLOT;
    static constexpr int V_OFF = K_OFF + NK * K_SLOT;
    static constexpr int SEND_OFF = V_OFF + NV * V_SLOT;  // local P half, x2
    static constexpr int RECV_OFF = SEND_OFF + 2 * PBUF;  // peer's P half, x2
    static constexpr int BAR_OFF = RECV_OFF + 2 * PBUF;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
    static constexpr int EXP_OFF = MISC_OFF + MISC_BYTES;  // FP8: exponents of every slot
    static constexpr int SMEM_USED = EXP_OFF + (NKV + NK + NV) * EXP_SLOT;
    static constexpr int SMEM_TOTAL = SMEM_USED + 1024;  // slack to align the base to 1024 B
    static constexpr uint32_t TM_S = 256;                // S buffers: fp32 columns
    static constexpr uint32_t TM_Q = TM_S + 32 * NSB;    // Q chunks 0..NQT-1: bf16 pairs

    static_assert(SMEM_TOTAL <= 232448, "shared memory budget");
    static_assert(QS_OFF % 1024 == 0 && KV_OFF % 1024 == 0 && K_OFF % 1024 == 0 &&
                      V_OFF % 1024 == 0 && CH % 1024 == 0,
                  "128-byte-swizzled operands need 1024-byte-aligned atoms");
    static_assert(SEND_OFF % 16 == 0 && RECV_OFF % 16 == 0 && PGRP % 16 == 0, "16-byte stores");
    static_assert(BAR_OFF % 8 == 0, "mbarrier alignment");
    static_assert(3 * (NKV + NK + NV) + 23 <= NBAR, "mbarrier count");
    static_assert(EXP_OFF % 16 == 0, "bulk copies of the row exponents");
    static_assert(KV_OFF + 128 * QSTG <= RECV_OFF && QSTG % 16 == 0, "Q staging area");
    static_assert(QS_OFF + NQS * QCH <= KV_OFF, "staged Q rows never overlap the Q chunks in smem");
    static_assert(TM_Q + 32 * NQT == TMEM_COLS, "tensor-memory budget");
};
constexpr int SMEM_TOTAL = Layout<false>::SMEM_TOTAL > Layout<true>::SMEM_TOTAL
                               ? Layout<false>::SMEM_TOTAL
                               : Layout<true>::SMEM_TOTAL;  // the larger, for occupancy

constexpr int NTHREADS = 224;                 // 7 warps
constexpr int NTHREADS_FP8 = 320;             // + 3 warps widening the FP8 tiles
constexpr uint64_t WAIT_NS = 1000000000ull;   // bounded waits: 1 s
constexpr uint64_t DRAIN_NS = 200000000ull;
constexpr float TAU = 8.0f;                   // lazy-rescale threshold (log2 units)
constexpr uint32_t XBYTES = PWARP;            // one warp's message: P rows + (reference, sum)

constexpr uint32_t IDESC_S = idesc_bf16(128, HALF, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, false, true);


__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ float2 ld_shared_v2f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}
// bf16 pair (lo, hi) scaled by f, rounded back to bf16 (round to nearest even)
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, float f) {
    return pack_bf16x2(__uint_as_float(v << 16) * f, __uint_as_float(v & 0xFFFF0000u) * f);
}

// Wait that ignores the abort flag: used only to drain copies and signals before exit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return;
    uint64_t t0 = globaltimer_ns();
    while (!mbar_test(bar, parity))
        if (globaltimer_ns() - t0 > DRAIN_NS) return;
}

// FP8 = true: the cache is e4m3 codes with one power-of-two scale per token (row
// exponents in p.exps). TMA brings each 32-token x 64-column chunk of codes (2 KB) into
// the upper half of its bf16 slot, with the block's 64 exponents beside the slot; three
// more warps (one per ring) widen the chunks in place to bf16 code * 2^e -- exact, since
// such a value has at most four significant bits -- and release the slot to the products
// on a second barrier. Everything downstream is the bf16 path, unchanged.
template <bool FP8, bool DS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FP8 ? NTHREADS_FP8 : NTHREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap map_kv, DecodeParams p) {
    using LY = Layout<DS>;
    constexpr int NSB = LY::NSB, NKV = LY::NKV, NK = LY::NK, NV = LY::NV, NQT = LY::NQT;
    constexpr int QS_OFF = LY::QS_OFF, KV_OFF = LY::KV_OFF, K_OFF = LY::K_OFF,
                  V_OFF = LY::V_OFF, SEND_OFF = LY::SEND_OFF, RECV_OFF = LY::RECV_OFF,
                  BAR_OFF = LY::BAR_OFF, MISC_OFF = LY::MISC_OFF, EXP_OFF = LY::EXP_OFF;
    constexpr uint32_t TM_S = LY::TM_S, TM_Q = LY::TM_Q;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sb - raw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int H = p.H;

    const uint32_t bar = sb + BAR_OFF;
    auto kv_full = [&](int s) { return bar + 8u * s; };
    auto kv_empty = [&](int s) { return bar + 8u * (NKV + s); };
    auto k_full = [&](int s) { return bar + 8u * (2 * NKV + s); };
    auto k_empty = [&](int s) { return bar + 8u * (2 * NKV + NK + s); };
    auto v_full = [&](int s) { return bar + 8u * (2 * NKV + 2 * NK + s); };
    auto v_empty = [&](int s) { return bar + 8u * (2 * NKV + 2 * NK + NV + s); };
    const uint32_t q_ready = bar + 8u * (2 * NKV + 2 * NK + 2 * NV);
    // scores of tile parity x in their TMEM buffer / read out by the softmax warps
    auto s_full = [&](int x) { return q_ready + 8 + 8u * x; };
    auto s_free = [&](int x) { return q_ready + 24 + 8u * x; };
    auto p_ready = [&](int x) { return q_ready + 40 + 8u * x; };  // both P halves of tile parity x
    auto pv_done = [&](int x) { return q_ready + 56 + 8u * x; };  // P.V of tile parity x finished
    // the peer's P.V of tile parity x finished (our P half in its buffer x may be
    // overwritten); arrived on by the peer's tcgen05.commit
    auto rfree = [&](int x) { return q_ready + 72 + 8u * x; };
    const uint32_t mma_drain = q_ready + 88;
    const uint32_t pv_drain = q_ready + 96;
    const uint32_t qs_full = q_ready + 104;  // the next segment's Q rows staged
    // the peer's P half of the rows of warp quadrant q has landed in buffer x
    auto recv_full = [&](int q, int x) { return q_ready + 112 + 8u * (2 * q + x); };
    // FP8: the slot's codes have been widened to bf16 (the bf16 kernel uses the full
    // barriers directly)
    auto kv_ready = [&](int s) { return FP8 ? q_ready + 176 + 8u * s : kv_full(s); };
    auto k_ready = [&](int s) { return FP8 ? q_ready + 176 + 8u * (NKV + s) : k_full(s); };
    auto v_ready = [&](int s) { return FP8 ? q_ready + 176 + 8u * (NKV + NK + s) : v_full(s); };
    auto exp_kv = [&](int s) { return sb + EXP_OFF + EXP_SLOT * s; };
    auto exp_k = [&](int s) { return sb + EXP_OFF + EXP_SLOT * (NKV + s); };
    auto exp_v = [&](int s) { return sb + EXP_OFF + EXP_SLOT * (NKV + NK + s); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + MISC_OFF + M_TMEM);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + MISC_OFF + M_ABORT);
    volatile int *misc = reinterpret_cast<volatile int *>(smem + MISC_OFF);
    const uint32_t misc_peer = mapa(sb + MISC_OFF, peer);  // the peer's MISC area

    auto init_barriers = [&]() {
        for (int s = 0; s < NKV; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        for (int s = 0; s < NK; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        mbar_init(q_ready, 4);
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x), 1);
            mbar_init(s_free(x), 4);
            mbar_init(p_ready(x), 4);
            mbar_init(pv_done(x), 1);
            mbar_init(rfree(x), 1);
        }
        mbar_init(mma_drain, 1);
        mbar_init(pv_drain, 1);
        mbar_init(qs_full, 4);
        for (int k = 0; k < 8; ++k) mbar_init(recv_full(k >> 1, k & 1), 1);
        if (FP8) {
            for (int s = 0; s < NKV; ++s) mbar_init(kv_ready(s), 1);
            for (int s = 0; s < NK; ++s) mbar_init(k_ready(s), 1);
            for (int s = 0; s < NV; ++s) mbar_init(v_ready(s), 1);
        }
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
    grid_dependency_wait();  // q, the cache rows and the schedule come from predecessor kernels
    // only now: the merge kernel that follows reads the schedule's job list before its own
    // dependency wait
    grid_launch_dependents();

    // ---- work: one (sequence, token range) per cluster, or, with the balanced
    // schedule, the segments of this cluster's equal share of the weighted tile list
    const bool sched = p.tile_start != nullptr;
    const int cl = blockIdx.x >> 1;
    int P = gridDim.x >> 1;
    long W = 0, r0 = 0, r1 = 0;
    int seg_b = 0;
    if (sched) {
        W = p.wpos[p.B];
        if (W < P) P = static_cast<int>(W);  // as in the schedule: no empty ranges
        if (cl < P) {
            r0 = (cl * W) / P;
            r1 = ((cl + 1) * W) / P;
        }
        seg_b = sched_first(p.wpos, p.B, r0);
    }

    int q_for = -1;  // softmax warps: the sequence whose Q rows are in TMEM / shared memory
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
        SchedSegment sg;
        if (!sched_next(p.tile_start, p.wpos, p.part_begin, p.B, r0, r1, W, P, cl, &seg_b, &sg))
            break;
        b = sg.b;
        t_begin = sg.t_begin;
        t_end = sg.t_end;
        direct = sg.direct;
        part = sg.part;
    }
    int L = p.seqlens[b];
    // a length outside [0, max_seqlen] is an error, recorded once per sequence (by the
    // work item holding its first tile) and clamped exactly as the schedule clamps it, so
    // both work distributions give the same result
    if (L < 0 || L > p.max_seqlen) {
        if (tid == 0 && rank == 0 && t_begin == 0) flag_error(p.err, MLA_ERR_OUT_OF_RANGE, b);
        L = L < 0 ? 0 : p.max_seqlen;
    }
    const int ntiles = (L + TOK - 1) / TOK;
    t_end = min(ntiles, t_end);
    const int n = max(0, t_end - t_begin);
    const int32_t *btab = p.block_table + (size_t)b * p.max_blocks;
    // remote operations of this segment, counted for an early stop of the pair:
    // P halves sent to the peer (st.async; the receive barrier of each is armed right
    // after), peer halves received, P.V commits multicast to the peer's rfree barriers
    int n_sent = 0, n_recv = 0, n_pv = 0;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n > 0) {
            // The rings are the only lookahead for the cache tiles: prefetching tiles beyond
            // them into L2 (2, 4 or 6 tiles ahead, or the next segment's first tiles) made
            // every workload slower, and the longer distances raised the DRAM reads (the
            // prefetched lines left L2 before their loads came). Near the end of a scheduled
            // segment only the next segment's Q rows are sent to L2.
            auto prefetch_next = [&]() {
                const int nb = sched_peek(p.tile_start, p.wpos, p.B, r1, seg_b);
                if (nb < 0) return;  // no further sequence in this cluster's share
                bulk_prefetch_l2(p.q_lat + (size_t)nb * H * D_C, static_cast<uint32_t>(H * D_C * 2));
                bulk_prefetch_l2(p.q_rope + (size_t)nb * H * D_ROPE,
                                 static_cast<uint32_t>(H * D_ROPE * 2));
            };
            const int next_at = sched ? max(0, n - (NKV + 8)) : -1;
            // L2 priorities: the own tokens' chunks in the peer's output columns are read
            // again by the peer (its V ring) and keep the normal priority; every other
            // chunk is read once and is marked to leave L2 first, so that the chunks still
            // awaiting their second read are not the ones evicted
            const uint64_t pol_once = l2_policy_evict_first();
            const uint64_t pol_twice = l2_policy_evict_normal();
            int issued_kv = 0, issued_k = 0;
            for (int i = 0; i < n; ++i) {
                const int skv = i % NKV, sk = i % NK;
                const int blk = btab[t_begin + i];
                const bool blk_ok = blk >= 0 && blk < p.num_blocks;
                if (!blk_ok && rank == 0) flag_error(p.err, MLA_ERR_OUT_OF_RANGE, b);
                const int y_own = blk * TOK + HALF * rank;
                // own tokens x own output columns
                if (!mbar_wait(kv_empty(skv), ((i / NKV) & 1) ^ 1, abort_flag, WAIT_NS)) break;
                if (blk_ok) {
                    // FP8: codes into the upper half of each chunk, exponents beside the slot
                    const uint32_t dst = sb + KV_OFF + skv * KV_SLOT + (FP8 ? CH / 2 : 0);
                    mbar_arrive_expect_tx(kv_full(skv), FP8 ? KV_SLOT / 2 + EXP_SLOT : KV_SLOT);
                    if (FP8) bulk_load(exp_kv(skv), p.exps + (size_t)blk * TOK, EXP_SLOT, kv_full(skv));
                    for (int k = 0; k < 4; ++k)
                        tma_load_2d_hint(dst + k * CH, &map_kv, kv_full(skv), 64 * (4 * rank + k),
                                         y_own, pol_once);
                } else {
                    mbar_arrive(kv_full(skv));  // no data: the consumers mask the tile
                }
                issued_kv = i + 1;
                // own tokens x the other c_kv columns and k_rope
                if (!mbar_wait(k_empty(sk), ((i / NK) & 1) ^ 1, abort_flag, WAIT_NS)) break;
                if (blk_ok) {
                    const uint32_t dst = sb + K_OFF + sk * K_SLOT + (FP8 ? CH / 2 : 0);
                    mbar_arrive_expect_tx(k_full(sk), FP8 ? K_SLOT / 2 + EXP_SLOT : K_SLOT);
                    if (FP8) bulk_load(exp_k(sk), p.exps + (size_t)blk * TOK, EXP_SLOT, k_full(sk));
                    for (int k = 0; k < 4; ++k)
                        tma_load_2d_hint(dst + k * CH, &map_kv, k_full(sk), 64 * (4 * peer + k),
                                         y_own, pol_twice);
                    tma_load_2d_hint(dst + 4 * CH, &map_kv, k_full(sk), D_C, y_own, pol_once);
                } else {
                    mbar_arrive(k_full(sk));
                }
                issued_k = i + 1;
                if (i == next_at) prefetch_next();
            }
            // copies still in flight must land before this CTA may exit
            for (int i = max(0, issued_kv - NKV); i < issued_kv; ++i)
                drain_wait(kv_full(i % NKV), (i / NKV) & 1);
            for (int i = max(0, issued_k - NK); i < issued_k; ++i)
                drain_wait(k_full(i % NK), (i / NK) & 1);
        }
    } else if (warp == 6) {
        // ------------------------------------ output product and its value chunks
        // P . V is issued by its own warp: a warp issuing the 36 small score MMAs of a
        // tile stays busy for about their execution time, and P . V must not queue
        // behind that. The peer's tokens of a tile in this CTA's output columns are needed
        // only here, so this warp also loads them, into a short ring whose slot frees when
        // the P . V that read it is done.
        if (n > 0) {
            const bool leader = elect_one();
            auto wait_all = [&](uint32_t bar_, uint32_t par) {
                return __all_sync(0xffffffffu, mbar_wait(bar_, par, abort_flag, WAIT_NS));
            };
            const uint64_t pol_once = l2_policy_evict_first();  // the second and last read
            auto load_v = [&](int j) {
                const int sv = j % NV;
                const int blk = btab[t_begin + j];
                if (blk >= 0 && blk < p.num_blocks) {
                    const uint32_t dst = sb + V_OFF + sv * V_SLOT + (FP8 ? CH / 2 : 0);
                    mbar_arrive_expect_tx(v_full(sv), FP8 ? V_SLOT / 2 + EXP_SLOT : V_SLOT);
                    if (FP8) bulk_load(exp_v(sv), p.exps + (size_t)blk * TOK, EXP_SLOT, v_full(sv));
                    for (int k = 0; k < 4; ++k)
                        tma_load_2d_hint(dst + k * CH, &map_kv, v_full(sv), 64 * (4 * rank + k),
                                         blk * TOK + HALF * peer, pol_once);
                } else {
                    mbar_arrive(v_full(sv));  // no data: the softmax zeroes the slot
                }
            };
            // O[:, own columns] += P [128 x 64] . V [64 x 256]: tokens [32h, 32h+32) come from
            // the local P half and the own-token chunks when h is this CTA's half, else from
            // the received half and the peer-token chunks
            auto issue_pv = [&](int i) {
                const uint32_t kv = sb + KV_OFF + (i % NKV) * KV_SLOT;
                const uint32_t vv = sb + V_OFF + (i % NV) * V_SLOT;
                const int x = i & 1;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const bool mine = h == static_cast<int>(rank);
                    const uint32_t a = sb + (mine ? SEND_OFF : RECV_OFF) + x * PBUF;
                    const uint32_t v = mine ? kv : vv;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        tc_mma_if(leader, tmem + TM_O, sdesc_kmajor_plain(a + kk * 256, 128, PGRP),
                                  sdesc_sw128(v + kk * 2048, CH, 1024), IDESC_PV,
                                  (i > 0 || h > 0 || kk > 0));
                }
                tc_commit_if(leader, kv_empty(i % NKV));
                tc_commit_if(leader, v_empty(i % NV));
                tc_commit_if(leader, pv_done(x));
                tc_commit_multicast_if(leader, rfree(x), static_cast<uint16_t>(1u << peer));
            };
            int loaded = min(n, NV);
            if (lane == 0)
                for (int j = 0; j < loaded; ++j) load_v(j);
            bool ok = true;
            for (int i = 0; ok && i < n; ++i) {
                // refill the slot of tile i-1 once its P . V is done
                if (i >= 1 && loaded < n) {
                    if (!(ok = wait_all(v_empty((i - 1) % NV), ((i - 1) / NV) & 1))) break;
                    if (lane == 0) load_v(loaded);
                    ++loaded;
                }
                if (!(ok = wait_all(p_ready(i & 1), (i >> 1) & 1))) break;
                if (!(ok = wait_all(v_ready(i % NV), (i / NV) & 1))) break;
                tc_fence_after();
                issue_pv(i);
                ++n_pv;
                __syncwarp();
            }
            // every MMA this warp issued has finished, every copy it started has landed
            if (leader) {
                tc_commit(pv_drain);
                drain_wait(pv_drain, 0);
            }
            if (lane == 0)
                for (int j = max(0, loaded - NV); j < loaded; ++j)
                    drain_wait(v_full(j % NV), (j / NV) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA
        // The whole warp runs the issue loop and one elected lane issues (the instruction
        // is predicated, not branched to): a tcgen05.mma issued by a lone lane of a
        // diverged warp costs that thread several times the tensor pipe's own time per
        // instruction at these small N.
        if (n > 0) {
            const bool leader = elect_one();
            auto wait_all = [&](uint32_t bar_, uint32_t par) {
                return __all_sync(0xffffffffu, mbar_wait(bar_, par, abort_flag, WAIT_NS));
            };
            const uint32_t qs = sb + QS_OFF;
            // scores of this CTA's 32 tokens of tile i over all 576 columns, into the S
            // buffer of the tile's parity
            auto issue_s = [&](int i) {
                const uint32_t kv = sb + KV_OFF + (i % NKV) * KV_SLOT;
                const uint32_t ko = sb + K_OFF + (i % NK) * K_SLOT;
                const uint32_t sd = tmem + TM_S + 32u * (i % NSB);
#pragma unroll
                for (int d = 0; d < NOWN; ++d)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // column chunk d of the own tokens: in the KV ring if it is one of
                        // this CTA's output chunks, else in the K ring (k_rope last)
                        const int o = d - 4 * static_cast<int>(rank);
                        const uint32_t src =
                            (o >= 0 && o < 4) ? kv + o * CH
                                              : ko + (d < 8 ? d - 4 * static_cast<int>(peer) : 4) * CH;
                        const uint64_t bdesc = sdesc_sw128(src + kk * 32, 16, 1024);
                        if (d < NQT)
                            tc_mma_ts_if(leader, sd, tmem + TM_Q + 32 * d + 8 * kk, bdesc, IDESC_S,
                                         (d | kk) != 0);
                        else
                            tc_mma_if(leader, sd,
                                      sdesc_sw128(qs + (d - NQT) * QCH + kk * 32, 16, 1024), bdesc,
                                      IDESC_S, 1);
                    }
                tc_commit_if(leader, s_full(i % NSB));
                tc_commit_if(leader, k_empty(i % NK));
            };
            // scores of tile k need its cache chunks and their S buffer back from the
            // softmax (s_free of tile k - NSB): with two buffers the scores of the next
            // tile are computed while the softmax still works on this one
            bool ok = wait_all(q_ready, 0);
            for (int k = 0; ok && k < n; ++k) {
                if (!(ok = wait_all(kv_ready(k % NKV), (k / NKV) & 1))) break;
                if (!(ok = wait_all(k_ready(k % NK), (k / NK) & 1))) break;
                if (k >= NSB && !(ok = wait_all(s_free(k % NSB), (k / NSB - 1) & 1))) break;
                tc_fence_after();
                issue_s(k);
                __syncwarp();
            }
            // every MMA this warp issued has finished before TMEM is released
            if (leader) {
                tc_commit(mma_drain);
                drain_wait(mma_drain, 0);
            }
        }
        __syncwarp();
    } else if (FP8 && warp >= 7) {
        // --------------------------------------------- FP8: widen the tiles to bf16
        // Warp 7 widens the K ring (the score products wait for it first), 8 the KV ring,
        // 9 the V ring, tile by tile as the codes land, chunk by chunk: the warp reads all
        // of a chunk's codes from its upper half into registers, syncs, then writes the
        // 64 bf16 values of each row as one 128-byte-swizzled row over the whole chunk
        // (the layout the bf16 TMA writes).
        if (n > 0) {
            const int ring = warp == 7 ? 1 : (warp == 8 ? 0 : 2);  // 0 KV, 1 K, 2 V
            const int c0 = 0, cstep = 1;
            const int nslot = ring == 0 ? NKV : (ring == 1 ? NK : NV);
            const int nch = ring == 1 ? 5 : 4;
            // the chunks' tokens: this CTA's own 32 for KV and K, the peer's for V
            const int tok0 = HALF * static_cast<int>(ring == 2 ? peer : rank);
            for (int i = 0; i < n; ++i) {
                const int sl = i % nslot;
                const uint32_t full = ring == 0 ? kv_full(sl) : (ring == 1 ? k_full(sl) : v_full(sl));
                if (!__all_sync(0xffffffffu,
                                mbar_wait(full, (i / nslot) & 1, abort_flag, WAIT_NS)))
                    break;
                const uint32_t base =
                    sb + (ring == 0 ? KV_OFF + sl * KV_SLOT
                                    : (ring == 1 ? K_OFF + sl * K_SLOT : V_OFF + sl * V_SLOT));
                const uint32_t ex =
                    ring == 0 ? exp_kv(sl) : (ring == 1 ? exp_k(sl) : exp_v(sl));
                // Load k (of 4) reads 512 contiguous bytes of the staged codes -- rows
                // 8k .. 8k+7, 64 bytes each -- so lane L holds row r_k = 8k + L/4, columns
                // 16(L%4) .. 16(L%4)+15: free of bank conflicts. Each row's scale exponent
                // is the same for every chunk of the tile.
                uint32_t s2a[4], s2b[4];
                bool two_steps = false;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = 8 * k + (lane >> 2);
                    const int e = static_cast<int8_t>(
                        *reinterpret_cast<const volatile uint8_t *>(smem + (ex - sb) + tok0 + r));
                    const int ee = e < -126 ? -126 : (e > 127 ? 127 : e);
                    // code * 2^e = (the shifted f16 pattern, value * 2^-112) * 2^(112 + e), in
                    // two exact steps when 112 + e > 127
                    s2a[k] = bf16x2_pow2(112 + ee > 127 ? 127 : 112 + ee);
                    s2b[k] = bf16x2_pow2(112 + ee > 127 ? 112 + ee - 127 : 0);
                    two_steps |= 112 + ee > 127;
                }
                two_steps = __any_sync(0xffffffffu, two_steps);
#pragma unroll 1
                for (int c = c0; c < nch; c += cstep) {
                    const uint32_t ch = base + c * CH;
                    uint4 raw[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) raw[k] = ld_shared_v4(ch + CH / 2 + k * 512 + lane * 16);
                    __syncwarp();  // every code is in registers before the chunk is overwritten
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int r = 8 * k + (lane >> 2);
                        const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
                        uint32_t o[8];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            o[2 * q] = e4m3x2_to_bf16x2_mul(static_cast<uint16_t>(w[q] & 0xFFFFu), s2a[k]);
                            o[2 * q + 1] = e4m3x2_to_bf16x2_mul(static_cast<uint16_t>(w[q] >> 16), s2a[k]);
                        }
                        if (two_steps) {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(o[q]) : "r"(s2b[k]));
                        }
                        // columns 16(L%4) .. +15 are the 16-byte pieces 2(L%4), 2(L%4)+1
                        const int pc = 2 * (lane & 3);
                        st_shared_v4(ch + r * 128 + ((pc ^ (r & 7)) << 4), o[0], o[1], o[2], o[3]);
                        st_shared_v4(ch + r * 128 + (((pc + 1) ^ (r & 7)) << 4), o[4], o[5], o[6],
                                     o[7]);
                    }
                    __syncwarp();
                }
                fence_proxy_async_smem();  // the tensor core reads what these stores wrote
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(ring == 0 ? kv_ready(sl) : (ring == 1 ? k_ready(sl) : v_ready(sl)));
            }
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
        // warps with at least one head row exchange their P rows (both CTAs agree)
        const bool wlive = wq * 32 < H;
        // this row in a P half: K-major 8 x 16-byte core matrices, no swizzle (next 8 K
        // elements +128 B, next 8 rows +PGRP B); each 8-row group ends with the rows'
        // (reference, row sum)
        const uint32_t prow = (row >> 3) * PGRP + (row & 7) * 16;
        const uint32_t mrow = (row >> 3) * PGRP + 512 + (row & 7) * 8;
        const uint32_t send = sb + SEND_OFF, recv = sb + RECV_OFF;
        const uint32_t recv_peer = mapa(recv, peer);
        const uint32_t rbar_peer = mapa(recv_full(wq, 0), peer);  // + 8 for buffer 1
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        // waits are warp-uniform: a lane that gives up takes its whole warp with it
        auto wait_w = [&](uint32_t bar_, uint32_t par) {
            return __all_sync(0xffffffffu, mbar_wait(bar_, par, abort_flag, WAIT_NS));
        };
        auto wait_wc = [&](uint32_t bar_, uint32_t par) {
            return __all_sync(0xffffffffu, mbar_wait<true>(bar_, par, abort_flag, WAIT_NS));
        };
        // Q rows of sequence bq: chunks 0..6 into TMEM (A operand of the score product),
        // chunks 7..8 (c_kv columns 448..511 and k_rope) into shared memory, 128-byte
        // swizzled as the cache tiles are. Rows >= H are 0. Three chunks per memory round
        // trip (more in flight at once costs the main loop registers).
        auto load_q = [&](int bq) {
            const uint4 *qsrc =
                reinterpret_cast<const uint4 *>(p.q_lat + ((size_t)bq * H + row) * D_C);
            const uint4 *rsrc =
                reinterpret_cast<const uint4 *>(p.q_rope + ((size_t)bq * H + row) * D_ROPE);
            const uint32_t qrow = sb + QS_OFF + (row >> 3) * 1024 + (row & 7) * 128;
            for (int c0 = 0; c0 < NOWN; c0 += 3) {
                uint4 v[3][8];
#pragma unroll
                for (int u = 0; u < 3; ++u)
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int c = c0 + u;
                        v[u][k] = make_uint4(0u, 0u, 0u, 0u);
                        if (live_row && c < NOWN) v[u][k] = c < 8 ? qsrc[8 * c + k] : rsrc[k];
                    }
#pragma unroll
                for (int u = 0; u < 3; ++u) {
                    const int c = c0 + u;
                    if (c >= NOWN) break;
                    if (c < NQT) {
                        uint32_t r[32];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            r[4 * k] = v[u][k].x;
                            r[4 * k + 1] = v[u][k].y;
                            r[4 * k + 2] = v[u][k].z;
                            r[4 * k + 3] = v[u][k].w;
                        }
                        tmem_st32(tl + TM_Q + 32 * c, r);
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            st_shared_v4(qrow + (c - NQT) * QCH + ((k ^ (row & 7)) << 4), v[u][k].x,
                                         v[u][k].y, v[u][k].z, v[u][k].w);
                    }
                }
            }
        };

        if (n > 0) {
            if (q_for != b) load_q(b);
            q_for = b;
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        }

        int blk_next = n > 0 ? btab[t_begin] : 0;  // block ids are fetched one tile ahead
        for (int i = 0; ok && i < n; ++i) {
            const int tile = t_begin + i;
            const int blk = blk_next;
            if (i + 1 < n) blk_next = btab[tile + 1];
            const int x = i & 1;
            const uint32_t kvs = sb + KV_OFF + (i % NKV) * KV_SLOT;
            const uint32_t vs = sb + V_OFF + (i % NV) * V_SLOT;

            // ---- scores of this CTA's 32 tokens, out of TMEM (releasing S)
            if (!(ok = wait_w(s_full(i % NSB), (i / NSB) & 1))) break;
            tc_fence_after();
            uint32_t sr[32];
            tmem_ld32(tl + TM_S + 32u * (i % NSB), sr);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free(i % NSB));

            const bool blk_ok = blk >= 0 && blk < p.num_blocks;
            const int tvalid = blk_ok ? min(TOK, L - tile * TOK) : 0;  // valid tokens of the tile
            // tokens of the tile this row keeps, and how many of them are this CTA's
            const int valid = live_row ? min(tvalid, max(0, L - back - tile * TOK)) : 0;
            const int ov = min(HALF, max(0, valid - HALF * static_cast<int>(rank)));
            float s[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) s[j] = j < ov ? __uint_as_float(sr[j]) : -INFINITY;
            float mx;
            {
                float t[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) t[j] = fmaxf(s[j], s[j + 16]);
#pragma unroll
                for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                    for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
                mx = t[0] * p.scale_log2;  // scale > 0: the max of the scaled scores
            }
            // local reference: raised only when a score exceeds it by more than TAU
            const float m_new = mx > m + TAU ? mx : m;

            // P (local half) = exp2(scale * s - reference), bf16 pairs
            auto make_p = [&](float ref, uint32_t (&pk)[16]) {
                const float nm = ref != -INFINITY ? -ref : 0.f;
                float es = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float p0 = fast_exp2(fmaf(s[2 * j], p.scale_log2, nm));
                    const float p1 = fast_exp2(fmaf(s[2 * j + 1], p.scale_log2, nm));
                    pk[j] = pack_bf16x2(p0, p1);
                    es += p0 + p1;
                }
                return ref != -INFINITY ? es : 0.f;
            };
            auto put_p = [&](const uint32_t (&pk)[16]) {
                const uint32_t dst = send + x * PBUF + prow;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    st_shared_v4(dst + k * 128, pk[4 * k], pk[4 * k + 1], pk[4 * k + 2],
                                 pk[4 * k + 3]);
            };
            uint32_t pk[16];
            float e_own = make_p(m_new, pk);

            // buffer x (local half) is free once P.V of tile i-2 has read it
            if (i >= 2 && !(ok = wait_w(pv_done(x), ((i >> 1) - 1) & 1))) break;
            float m_peer = -INFINITY, e_peer = 0.f;
            if (wlive) {
                put_p(pk);
                // the peer's buffer x is free once its P.V of tile i-2 is done; the P row
                // and its (reference, sum) go straight from registers into it
                if (i >= 2 && !(ok = wait_wc(rfree(x), ((i >> 1) - 1) & 1))) break;
                {
                    const uint32_t dst = recv_peer + x * PBUF + prow, rb = rbar_peer + 8u * x;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        st_async_v4(dst + k * 128, pk[4 * k], pk[4 * k + 1], pk[4 * k + 2],
                                    pk[4 * k + 3], rb);
                    st_async_v2(recv_peer + x * PBUF + mrow, __float_as_uint(m_new),
                                __float_as_uint(e_own), rb);
                }
                if (lane == 0) mbar_arrive_expect_tx(recv_full(wq, x), XBYTES);
                ++n_sent;
                // ---- the peer's half of tile i
                if (!(ok = wait_wc(recv_full(wq, x), (i >> 1) & 1))) break;
                ++n_recv;
                const float2 pm = ld_shared_v2f(recv + x * PBUF + mrow);
                m_peer = pm.x;
                e_peer = pm.y;
            }

            // ---- common reference: the larger of the two; the half computed against the
            // smaller one is brought to it (the local half recomputed from the scores, the
            // received half rescaled)
            const float m_fin = fmaxf(m_new, m_peer);
            const bool fix_own = m_new != m_fin, fix_peer = m_peer != m_fin;
            if (fix_own) {
                e_own = make_p(m_fin, pk);
                put_p(pk);
            }
            if (fix_peer) {
                const float f = fast_exp2(m_peer - m_fin);
                const uint32_t src = recv + x * PBUF + prow;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint4 v = ld_shared_v4(src + k * 128);
                    st_shared_v4(src + k * 128, scale_bf16x2(v.x, f), scale_bf16x2(v.y, f),
                                 scale_bf16x2(v.z, f), scale_bf16x2(v.w, f));
                }
                e_peer *= f;
            }

            // ---- O and l follow the reference
            const bool raise = m_fin != m;
            if (__any_sync(0xffffffffu, raise)) {
                const float alpha = raise ? fast_exp2(m - m_fin) : 1.f;
                if (i > 0) {
                    // O holds tiles < i: wait until P.V of tile i-1 has landed, then rescale
                    if (!(ok = wait_w(pv_done(x ^ 1), ((i - 1) >> 1) & 1))) break;
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
                m = m_fin;
            }
            // tokens in order (low half first) in both CTAs: the same l bit for bit
            l += rank == 0 ? e_own + e_peer : e_peer + e_own;

            // rows past the valid tokens (the whole tile if its block is bad) may hold stale
            // or poisoned data: zero them in the chunks P.V reads, since 0 * NaN would
            // still poison the product
            if (tvalid < TOK) {
                // the value chunks of the peer's tokens may still be in flight
                if (!(ok = wait_w(v_ready(i % NV), (i / NV) & 1))) break;
                const int own_from = min(HALF, max(0, tvalid - HALF * static_cast<int>(rank)));
                const int peer_from = min(HALF, max(0, tvalid - HALF * static_cast<int>(peer)));
                const int n_own = (HALF - own_from) * 32;  // 16-byte pieces: rows x 4 x 8
                const int n_all = n_own + (HALF - peer_from) * 32;
                for (int e = row; e < n_all; e += 128) {
                    const bool o = e < n_own;
                    const int ee = o ? e : e - n_own;
                    const int r = (o ? own_from : peer_from) + (ee >> 5), c = (ee >> 3) & 3,
                              k = ee & 7;
                    const uint32_t base = (o ? kvs : vs) + c * CH;
                    st_shared_v4(base + r * 128 + k * 16, 0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_ready(x));
        }
        // ------------------------------------------------------------- output
        const int nb = sched && ok && n > 0 ? sched_peek(p.tile_start, p.wpos, p.B, r1, seg_b)
                                            : -1;
        const int col0 = 256 * rank;
        // fp32 rows: a part of a cut sequence, or the whole output when the caller asked
        // for fp32 (partial attention over one rank's token range)
        const bool out32 = !direct || p.out_f32 != nullptr;
        float *const orow32 =
            !out32 ? nullptr
                   : (direct ? p.out_f32 + ((size_t)b * H + row) * D_C
                             : p.o_part + ((size_t)part * H + row) * D_C) + col0;
        if (n > 0 && ok && wait_w(pv_done((n - 1) & 1), ((n - 1) >> 1) & 1)) {
            tc_fence_after();
            // Every product of this segment is done, so the rings are idle: the next
            // scheduled segment's Q rows are copied into them (one bulk copy per row and
            // array) while the output rows are written, then moved to their places.
            if (nb >= 0) {
                const int live = min(max(H - 32 * wq, 0), 32);
                if (lane == 0) mbar_arrive_expect_tx(qs_full, live * 2 * (D_C + D_ROPE));
                __syncwarp();
                if (live_row) {
                    const uint32_t dst = sb + KV_OFF + row * QSTG;
                    bulk_load(dst, p.q_lat + ((size_t)nb * H + row) * D_C, 2 * D_C, qs_full);
                    bulk_load(dst + 2 * D_C, p.q_rope + ((size_t)nb * H + row) * D_ROPE,
                              2 * D_ROPE, qs_full);
                }
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t r[32];
                tmem_ld32(tl + TM_O + 32 * c, r);
                tmem_ld_wait();
                if (row < H) {
                    // each thread writes its row: 32-byte stores, so that every request
                    // carries a whole sector (16-byte ones over 32 rows per warp instruction
                    // made the L1-to-L2 requests, not the bytes, the limit)
                    if (!out32) {
                        uint16_t *dst = p.out + ((size_t)b * H + row) * D_C + col0 + 32 * c;
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            uint32_t w[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                w[j] = pack_bf16x2(__uint_as_float(r[16 * k + 2 * j]) * inv,
                                                   __uint_as_float(r[16 * k + 2 * j + 1]) * inv);
                            st_global_v8(dst + 16 * k, w[0], w[1], w[2], w[3], w[4], w[5], w[6],
                                         w[7]);
                        }
                    } else {
                        // parts are kept in L2 (evict-last) until the merge that follows reads
                        // them: the tail part of a cut sequence is written early in the launch
                        const uint64_t pol = direct ? l2_policy_evict_normal() : l2_policy_evict_last();
                        float *dst = orow32 + 32 * c;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            st_global_v8_hint(
                                dst + 8 * k, __float_as_uint(__uint_as_float(r[8 * k]) * inv),
                                __float_as_uint(__uint_as_float(r[8 * k + 1]) * inv),
                                __float_as_uint(__uint_as_float(r[8 * k + 2]) * inv),
                                __float_as_uint(__uint_as_float(r[8 * k + 3]) * inv),
                                __float_as_uint(__uint_as_float(r[8 * k + 4]) * inv),
                                __float_as_uint(__uint_as_float(r[8 * k + 5]) * inv),
                                __float_as_uint(__uint_as_float(r[8 * k + 6]) * inv),
                                __float_as_uint(__uint_as_float(r[8 * k + 7]) * inv), pol);
                    }
                }
            }
            if (nb >= 0) {
                if ((ok = wait_w(qs_full, 0))) {
                    const uint32_t src = sb + KV_OFF + row * QSTG;
                    const uint32_t qrow = sb + QS_OFF + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll 1
                    for (int c = 0; c < NOWN; ++c) {
                        uint4 v[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            v[k] = live_row ? ld_shared_v4(src + 128 * c + 16 * k)
                                            : make_uint4(0u, 0u, 0u, 0u);
                        if (c < NQT) {
                            uint32_t r[32];
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                r[4 * k] = v[k].x;
                                r[4 * k + 1] = v[k].y;
                                r[4 * k + 2] = v[k].z;
                                r[4 * k + 3] = v[k].w;
                            }
                            tmem_st32(tl + TM_Q + 32 * c, r);
                        } else {
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                st_shared_v4(qrow + (c - NQT) * QCH + ((k ^ (row & 7)) << 4),
                                             v[k].x, v[k].y, v[k].z, v[k].w);
                        }
                    }
                    q_for = nb;
                } else if (lane == 0) {
                    drain_wait(qs_full, 0);  // copies still in flight land before exit
                }
            }
        } else if (row < H) {
            // empty range (or aborted): zero output, lse = -inf
            if (!out32) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((size_t)b * H + row) * D_C + col0);
                for (int k = 0; k < 32; ++k) dst[k] = make_uint4(0u, 0u, 0u, 0u);
            } else {
                float4 *dst = reinterpret_cast<float4 *>(orow32);
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
    // our own copies have read their rows, the peer's signals that its P.V has read our
    // halves have all arrived, every role is idle; then barriers restart
    if (warp >= 2 && lane == 0) bulk_wait_read_all();
    if (tid == 64 && n > 0 && !*abort_flag) {
        for (int x = 0; x < 2; ++x) {
            const int cnt = (n + 1 - x) / 2;  // tiles of parity x
            if (cnt > 0) drain_wait(rfree(x), (cnt - 1) & 1);
        }
    }
    if (warp >= 2 && warp < 6 && lane == 0) {
        misc[(M_SENT >> 2) + (warp - 2)] = n_sent;  // = receive barriers armed
        misc[(M_RECV >> 2) + (warp - 2)] = n_recv;
    }
    if (warp == 6 && lane == 0) misc[M_PV >> 2] = n_pv;
    if (tid == 0) st_cluster_u32(misc_peer + M_PEER_ABORT, *abort_flag ? 1u : 0u);
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    // Both CTAs now see both abort flags and take the same branch.
    if (*abort_flag || misc[M_PEER_ABORT >> 2]) {
        // The pair stops early. Before either CTA may exit, every remote operation the
        // peer issued into this CTA must have landed: its P halves (st.async, completing
        // on recv_full) and its P.V commits (multicast arrivals on rfree). Each CTA tells
        // the peer how many of each it issued, then waits (bounded) for the peer's.
        // Neither CTA issues anything remote after the barrier above, and the peer can
        // be at most two P halves ahead of what this CTA received (it sends tile t + 2
        // only after this CTA's P.V of tile t released its buffer), so each barrier has
        // at most one phase outstanding and the parity waits below are unambiguous.
        if (tid == 0) {
            st_cluster_u32(misc_peer + M_PEER_PV, static_cast<uint32_t>(misc[M_PV >> 2]));
            for (int q = 0; q < 4; ++q)
                st_cluster_u32(misc_peer + M_PEER_SENT + 4 * q,
                               static_cast<uint32_t>(misc[(M_SENT >> 2) + q]));
        }
        __syncthreads();
        cluster_sync();
        if (warp >= 2 && warp < 6 && lane == 0) {
            const int q = warp - 2;
            const int sent = misc[(M_PEER_SENT >> 2) + q], armed = misc[(M_SENT >> 2) + q];
            for (int t = misc[(M_RECV >> 2) + q]; t < sent; ++t) {
                if (t >= armed) mbar_arrive_expect_tx(recv_full(q, t & 1), XBYTES);
                drain_wait(recv_full(q, t & 1), (t >> 1) & 1);
            }
        }
        if (tid == 64) {
            const int pv = misc[M_PEER_PV >> 2];
            for (int x = 0; x < 2; ++x) {
                const int cnt = (pv + 1 - x) / 2;  // the peer's P.V commits of parity x
                if (cnt > 0) drain_wait(rfree(x), (cnt - 1) & 1);
            }
        }
        if (tid == 0) *abort_flag = 1;
        break;  // the final cluster barrier follows
    }
    if (!sched) break;
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

namespace {
// Two S buffers for at most 64 query rows, one above (the layouts' comment gives why).
template <bool FP8, bool DS>
cudaError_t launch_variant(const CUtensorMap &mkv, const DecodeParams &p, dim3 grid,
                           cudaStream_t stream) {
    constexpr int smem = Layout<DS>::SMEM_TOTAL;
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<FP8, DS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_tc_kernel<FP8, DS>, grid, dim3(FP8 ? NTHREADS_FP8 : NTHREADS), smem,
                      stream, mkv, p);
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
    if (cudaFuncSetAttribute(decode_tc_kernel<false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL) == cudaSuccess &&
        cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<false, false>, &cfg) == cudaSuccess &&
        n > 0)
        slots = n;
    else
        slots = device_sm_count() / 2;
    return slots;
}

cudaError_t launch_decode_tc(const DecodeParams &p, int clusters, cudaStream_t stream) {
    CUtensorMap mkv;
    dim3 grid(2 * clusters);
    if (p.codes) {
        // e4m3 codes [num_blocks * 64 rows][576 bytes], 32-row x 64-byte boxes, no swizzle
        EncodeTiledFn fn = encode_fn();
        if (!fn) return cudaErrorInvalidValue;
        cuuint64_t dims[2] = {D_QK, (cuuint64_t)p.num_blocks * TOK};
        cuuint64_t strides[1] = {D_QK};
        cuuint32_t box[2] = {64, HALF};
        cuuint32_t estr[2] = {1, 1};
        if (fn(&mkv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(p.codes), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        return p.H <= 64 ? launch_variant<true, true>(mkv, p, grid, stream)
                         : launch_variant<true, false>(mkv, p, grid, stream);
    }
    if (!encode_bf16_2d(&mkv, p.cache, D_QK, (uint64_t)p.num_blocks * TOK, HALF))
        return cudaErrorInvalidValue;
    return p.H <= 64 ? launch_variant<false, true>(mkv, p, grid, stream)
                     : launch_variant<false, false>(mkv, p, grid, stream);
}

}  // namespace mla
