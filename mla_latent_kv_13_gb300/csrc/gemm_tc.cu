// gemm_tc.cu -- bf16 GEMM for the absorbed projections on the sm_100-family tensor
// cores: TMA-fed, tcgen05.mma into TMEM, one 128 x BN output tile per CTA (BN = 256 for
// long, wide products: the activation tile, re-read once per output tile, then costs
// half as much traffic per weight byte).
//
// C[m][n] = sum_k A[m][k] * B(k, n), fp32 accumulation, where the batch rows (the
// decode batch, M <= 128 per tile) are A and the weights are B:
//   "TN": B stored [N][K] (row n is output feature n: the [out, in] layout), or
//   "NN": B stored [K][N] (W_UK, whose rows are per-head key dims).
// Operands are addressed through 2-D tensor maps; a batch index (one per head for the
// per-head products) shifts the A columns and the B rows by fixed amounts, so one map
// serves every head. K is cut into k_splits ranges: these products are weight-bandwidth
// bound (M = batch is small), and the split keeps every SM streaming weights even when
// there are few output tiles. The ranges' fp32 partials are either written out for a
// finalize kernel, or (CRED kernels) reduced inside the thread-block cluster that holds
// all the k-splits of one output tile: each CTA stages its partial in its idle stage ring,
// then sums a share of the tile's rows over every CTA's shared memory, in split order, and
// writes them as bf16 -- no partials in global memory and no second launch.
//
// Roles (192 threads): warp 0 issues TMA (one lane), warp 1 owns TMEM and issues the
// MMAs (the whole warp waits, one elected lane issues through predicated instructions),
// warps 2-5 read the accumulator out of TMEM and write it: into the stage ring, idle once
// the products are done, as 128-byte-swizzled boxes that one thread stores with TMA (whole
// lines instead of one row per thread), or directly where the output layout does not fit
// one tensor map. Waits are bounded (one second); a wait that gives up records
// MLA_ERR_TIMEOUT.
// The stage ring holds min(6, k-blocks of a CTA) stages (4 at width 256) and shared
// memory is sized to it, so products with little K per tile (the per-head absorptions)
// run several CTAs per SM instead of one; products with many 256-wide tiles and short K
// take two stages for the same reason.
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mla {

namespace {

using namespace sm100;

constexpr int BM = 128, BK = 64;
constexpr int TILE_A = BM * BK * 2;         // 16 KB
constexpr int NN_GROUP = BK * 64 * 2;       // NN B tile: one 64-column group of BK rows (8 KB)
constexpr int SMEM_EXTRA = 256 + 1024;      // barriers + slack to align the base
constexpr int NTHREADS = 192;
constexpr uint64_t WAIT_NS = 1000000000ull;

template <int BN> struct Tile {
    static constexpr int TILE_B = BN * BK * 2;           // 16 to 32 KB
    static constexpr int STAGE = TILE_A + TILE_B;
    static constexpr int NS = BN == 128 ? 6 : (BN == 256 ? 4 : 5);  // stages at most
    static constexpr int SMEM_TOTAL = NS * STAGE + SMEM_EXTRA;
    static_assert(SMEM_TOTAL <= 232448, "shared memory budget");
};

struct TcGemmArgs {
    int M, N, K, batch, k_splits, k_per_split;
    int ns;     // stages in the ring (1..NS)
    int tma_c;  // output written from shared memory by TMA stores (map_c): 1 = bf16 C,
                //   2 = fp32 split-K partials (3-D map: columns, rows, split x batch)
    int a_bx;   // A column offset per batch
    int b_bx;   // B (TN) column offset per batch
    int b_by;   // B row offset per batch (TN: rows of N; NN: rows of K)
    float *c_part;
    uint16_t *c_bf16;
    long ldc, c_bstride;
    uint32_t *err;
    // ROPE kernels: column tiles t1 and up are a second product, with the weights of map_b2
    // and the output map_c2, and each pair of columns (2i, 2i+1) of a 64-column head rotated
    // by the angle rope_pos[row] * rope.f[i] (decoupled RoPE); n1, n2 = the products' widths
    int t1, n1, n2;
    const int32_t *rope_pos;
    RopeFreqs rope;  // also the k_rope rotation of CRED = 2 kernels
    // CRED = 2: positions, block table [M][ap_max_blocks] and the paged cache
    // [ap_num_blocks * BLOCK][D_QK] the new rows go to
    const int32_t *ap_pos, *ap_bt;
    int ap_max_blocks, ap_num_blocks;
    uint16_t *ap_cache;
};

// Store the box at (x, y) of a tensor map from this CTA's shared memory (bulk async-group;
// x * element size a multiple of 16 bytes, x and y not negative).
__device__ __forceinline__ void tma_store_2d(const void *map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_store_3d(const void *map, uint32_t src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// 16 bytes of fp32 from a shared::cluster address (this CTA's or a peer's shared memory)
__device__ __forceinline__ float4 ld_cluster_v4f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
    uint64_t t0 = globaltimer_ns();
    while (!mbar_test(bar, parity))
        if (globaltimer_ns() - t0 > 200000000ull) return;
}

// CRED: 0 = no cluster reduction; 1 = reduced into bf16 C; 2 = reduced into the new latent
// cache rows of append (row b of the product is sequence b's token at pos[b]: the k_rope
// pairs rotated by that position, the row written into its block of the paged cache);
// 3 = two products of one activation, column tiles t1 and up the second (weights map_b2):
// the first reduced into bf16 C, the second into append's cache rows
template <bool NN, int BN, bool ROPE, int CRED>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_c,
                   const __grid_constant__ CUtensorMap map_b2,
                   const __grid_constant__ CUtensorMap map_c2, TcGemmArgs g) {
    constexpr int STAGE = Tile<BN>::STAGE;
    constexpr uint32_t TMEM_COLS = BN <= 128 ? 128 : 256;  // a power of two
    constexpr uint32_t IDESC = idesc_bf16(BM, BN, false, NN);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sb - raw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
    // ROPE and CRED = 3 kernels: a tile of the second product reads map_b2 (ROPE: and writes
    // map_c2) from its own column nb0 (each product's last tile may be ragged)
    constexpr bool TWO = ROPE || CRED == 3;
    const bool second = TWO && static_cast<int>(blockIdx.x) >= g.t1;
    const int nb0 = second ? (static_cast<int>(blockIdx.x) - g.t1) * BN : n0;
    const CUtensorMap *const mbp = second ? &map_b2 : &map_b;
    const int batch = blockIdx.z / g.k_splits, split = blockIdx.z % g.k_splits;
    const int k_begin = split * g.k_per_split;
    const int k_end = min(g.K, k_begin + g.k_per_split);
    const int nkb = (k_end - k_begin + BK - 1) / BK;

    const int ns = g.ns;
    // CRED: the ring also holds the staged fp32 partial tile (BM x BN) once the products are done
    const int bar_off = CRED != 0 ? max(ns * STAGE, BM * BN * 4) : ns * STAGE;
    const uint32_t bar = sb + bar_off;
    auto full = [&](int s) { return bar + 8u * s; };
    auto empty = [&](int s) { return bar + 8u * (ns + s); };
    const uint32_t done = bar + 8u * (2 * ns);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + bar_off + 8 * (2 * ns + 1));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + bar_off + 8 * (2 * ns + 2));

    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(mbp);
        if (g.tma_c) tma_prefetch_map(second ? &map_c2 : &map_c);
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

    if (warp == 0) {
        if (lane == 0) {
            // the weights (B) never come from a predecessor kernel: their first tiles head for
            // L2 while the predecessor finishes; the activations (A) only after it has
            for (int kb = 0; kb < min(nkb, ns); ++kb) {
                const int k = k_begin + kb * BK;
                if (!NN) {
                    tma_prefetch_l2_2d(mbp, batch * g.b_bx + k, batch * g.b_by + nb0);
                } else {
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_prefetch_l2_2d(&map_b, n0 + 64 * j, batch * g.b_by + k);
                }
            }
            grid_dependency_wait();
            int issued = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % ns;
                if (!mbar_wait(empty(s), ((kb / ns) & 1) ^ 1, abort_flag, WAIT_NS)) break;
                const int k = k_begin + kb * BK;
                const uint32_t sa = sb + s * STAGE, sbb = sa + TILE_A;
                mbar_arrive_expect_tx(full(s), STAGE);
                tma_load_2d(sa, &map_a, full(s), batch * g.a_bx + k, m0);
                if (!NN) {
                    tma_load_2d(sbb, mbp, full(s), batch * g.b_bx + k, batch * g.b_by + nb0);
                } else {
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(sbb + j * NN_GROUP, &map_b, full(s), n0 + 64 * j,
                                    batch * g.b_by + k);
                }
                issued = kb + 1;
            }
            for (int kb = max(0, issued - ns); kb < issued; ++kb) drain(full(kb % ns), (kb / ns) & 1);
        }
    } else if (warp == 1) {
        // The whole warp waits and one elected lane issues through predicated instructions:
        // a tcgen05.mma issued by a lone lane of a diverged warp costs that thread more than
        // the tensor pipe's own time per instruction.
        const bool leader = elect_one();
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % ns;
            if (!__all_sync(0xffffffffu, mbar_wait(full(s), (kb / ns) & 1, abort_flag, WAIT_NS)))
                break;
            tc_fence_after();
            const uint32_t sa = sb + s * STAGE, sbb = sa + TILE_A;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t ad = sdesc_sw128(sa + kk * 32, 16, 1024);
                const uint64_t bd = NN ? sdesc_sw128(sbb + kk * 2048, NN_GROUP, 1024)
                                       : sdesc_sw128(sbb + kk * 32, 16, 1024);
                tc_mma_if(leader, tmem, ad, bd, IDESC, (kb | kk) != 0);
            }
            tc_commit_if(leader, empty(s));
            __syncwarp();
        }
        if (leader) {
            tc_commit(done);  // arrives once every MMA above has finished
            drain(done, 0);
        }
        __syncwarp();
    } else {
        // epilogue: thread = output row m0 + (warp % 4) * 32 + lane
        const int wq = warp & 3;
        const int m = m0 + wq * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        // ROPE: the row's 32 rotations, formed while the products run (positions come from
        // the caller, so only after the dependency wait)
        float rc[ROPE ? 32 : 1], rs[ROPE ? 32 : 1];
        if constexpr (ROPE) {
            if (second) {
                grid_dependency_wait();
                const int pm = m < g.M ? g.rope_pos[m] : 0;
#pragma unroll
                for (int i = 0; i < 32; ++i) rope_cos_sin(pm, g.rope.f[i], rc[i], rs[i]);
            }
        }
        const bool ok =
            __all_sync(0xffffffffu, nkb > 0 && mbar_wait(done, 0, abort_flag, WAIT_NS));
        if constexpr (CRED != 0) {
            // this k-range's fp32 partial into the idle ring: row r at r * BN * 4 bytes, its
            // 16-byte pieces permuted by r % 8 (8 consecutive rows, or 8 consecutive pieces of
            // one row, then fall in distinct bank groups)
            if (ok) {
                tc_fence_after();
                const int r = wq * 32 + lane;
                const uint32_t rowp = sb + r * (BN * 4);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tl + 32 * c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        st_shared_v4(rowp + (((8 * c + k) ^ (r & 7)) << 4), v[4 * k], v[4 * k + 1],
                                     v[4 * k + 2], v[4 * k + 3]);
                }
            }
        } else if (ok && g.tma_c == 2) {
            // fp32 partials the same way: each 32-column chunk is one 128-byte-swizzled
            // 128 x 32 box of the [split x batch][M][N] partial array
            tc_fence_after();
            const int r = wq * 32 + lane;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tl + 32 * c, v);
                tmem_ld_wait();
                const uint32_t rowp = sb + c * (BM * 128) + r * 128;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    st_shared_v4(rowp + ((k ^ (r & 7)) << 4), v[4 * k], v[4 * k + 1], v[4 * k + 2],
                                 v[4 * k + 3]);
            }
            fence_proxy_async_smem();
            asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
            if (warp == 2 && lane == 0) {
                for (int c = 0; c < BN / 32 && n0 + 32 * c < g.N; ++c)
                    tma_store_3d(&map_c, sb + c * (BM * 128), n0 + 32 * c, m0,
                                 split * g.batch + batch);
                bulk_commit();
                bulk_wait_read_all();  // the boxes have left shared memory before exit
            }
        } else if (ok && g.tma_c) {
            // bf16 tile through shared memory: every product is done, so the stage ring is
            // idle; each 64-column group becomes one 128-byte-swizzled 128 x 64 box (row r at
            // r * 128 bytes, its 16-byte chunks permuted by r % 8), written by one TMA store
            tc_fence_after();
            const int r = wq * 32 + lane;
            if (second) {
                if constexpr (ROPE) {
                    // 64-column heads: chunk c holds the pairs 16 (c % 2) .. 16 (c % 2) + 15
#pragma unroll 1
                    for (int c2 = 0; c2 < BN / 64; ++c2) {
                        const uint32_t rowp = sb + c2 * (BM * 128) + r * 128;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            uint32_t v[32];
                            tmem_ld32(tl + 32 * (2 * c2 + hh), v);
                            tmem_ld_wait();
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                uint32_t w[4];
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const int j = 4 * k + q;  // the pair's index in the chunk
                                    const float x0 = __uint_as_float(v[2 * j]);
                                    const float x1 = __uint_as_float(v[2 * j + 1]);
                                    const float c_ = rc[16 * hh + j], s_ = rs[16 * hh + j];
                                    w[q] = pack_bf16x2(x0 * c_ - x1 * s_, x0 * s_ + x1 * c_);
                                }
                                const int ch = hh * 4 + k;
                                st_shared_v4(rowp + ((ch ^ (r & 7)) << 4), w[0], w[1], w[2], w[3]);
                            }
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tl + 32 * c, v);
                    tmem_ld_wait();
                    const uint32_t rowp = sb + (c >> 1) * (BM * 128) + r * 128;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int ch = (c & 1) * 4 + k;
                        st_shared_v4(rowp + ((ch ^ (r & 7)) << 4),
                                     pack_bf16x2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
                                     pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                                     pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                                     pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
                    }
                }
            }
            fence_proxy_async_smem();
            asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
            if (warp == 2 && lane == 0) {
                const int nlim = ROPE ? (second ? g.n2 : g.n1) : g.N;
                for (int j = 0; j < BN / 64 && nb0 + 64 * j < nlim; ++j) {
                    if (second)
                        tma_store_2d(&map_c2, sb + j * (BM * 128), nb0 + 64 * j, m0);
                    else
                        tma_store_2d(&map_c, sb + j * (BM * 128),
                                     static_cast<int>(batch * g.c_bstride) + n0 + 64 * j, m0);
                }
                bulk_commit();
                bulk_wait_read_all();  // the boxes have left shared memory before exit
            }
        } else if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tl + 32 * c, r);
                tmem_ld_wait();
                const int nb = n0 + 32 * c;
                if (m < g.M && nb < g.N) {
                    if (g.c_part) {
                        float *dst = g.c_part + (((size_t)split * g.batch + batch) * g.M + m) *
                                                    (size_t)g.N + nb;
                        if (nb + 32 <= g.N) {
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                reinterpret_cast<float4 *>(dst)[k] =
                                    make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                                __uint_as_float(r[4 * k + 2]),
                                                __uint_as_float(r[4 * k + 3]));
                        } else {
                            for (int j = 0; j < g.N - nb; ++j) dst[j] = __uint_as_float(r[j]);
                        }
                    } else {
                        uint16_t *dst = g.c_bf16 + batch * g.c_bstride + (size_t)m * g.ldc + nb;
                        if (nb + 32 <= g.N) {
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                reinterpret_cast<uint4 *>(dst)[k] = make_uint4(
                                    pack_bf16x2(__uint_as_float(r[8 * k]), __uint_as_float(r[8 * k + 1])),
                                    pack_bf16x2(__uint_as_float(r[8 * k + 2]), __uint_as_float(r[8 * k + 3])),
                                    pack_bf16x2(__uint_as_float(r[8 * k + 4]), __uint_as_float(r[8 * k + 5])),
                                    pack_bf16x2(__uint_as_float(r[8 * k + 6]), __uint_as_float(r[8 * k + 7])));
                        } else {
                            for (int j = 0; j < g.N - nb; ++j) dst[j] = f32_to_bf16(__uint_as_float(r[j]));
                        }
                    }
                }
            }
        }
    }
    if constexpr (CRED != 0) {
        // The cluster is the k-splits of this output tile (cluster rank = split). Once every
        // CTA has staged its partial, CTA r sums rows [r rp, r rp + rp) of the tile over the
        // splits in order (the finalize kernel's order, so both paths give the same bits) and
        // writes them bf16; the second barrier keeps every CTA's shared memory alive until
        // the others have read it. Every thread reaches both barriers, whatever its waits gave.
        __syncwarp();
        cluster_sync();
        const int S = g.k_splits;
        const int mrows = min(BM, g.M - m0);
        const int rp = (mrows + S - 1) / S;
        const int r_begin = static_cast<int>(cluster_ctarank()) * rp;
        const int r_end = min(mrows, r_begin + rp);
        constexpr int U = BN / 4;  // 16-byte pieces of a staged row
        uint32_t src[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) src[q] = q < S ? mapa(sb, static_cast<uint32_t>(q)) : 0u;
        const int nlim = CRED == 3 ? (second ? g.n2 : g.n1) : g.N;
        for (int e = tid; e < (r_end - r_begin) * U; e += NTHREADS) {
            const int r = r_begin + e / U, j = e % U;
            const int n = nb0 + 4 * j;
            if (n >= nlim) continue;
            const uint32_t off = static_cast<uint32_t>(r * (BN * 4) + ((j ^ (r & 7)) << 4));
            float4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < S) v[q] = ld_cluster_v4f(src[q] + off);
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q < S) {
                    a0 += v[q].x;
                    a1 += v[q].y;
                    a2 += v[q].z;
                    a3 += v[q].w;
                }
            uint16_t *dst;
            if (CRED == 1 || (CRED == 3 && !second)) {
                dst = g.c_bf16 + (size_t)(m0 + r) * g.ldc + n;
            } else {
                // a position or block outside the cache is an error: flagged once per row
                // (first column piece of the first column tile) and the row dropped
                const int b = m0 + r;
                const int pp = g.ap_pos[b];
                const int blk = pp >= 0 && pp < g.ap_max_blocks * BLOCK
                                    ? g.ap_bt[(size_t)b * g.ap_max_blocks + pp / BLOCK]
                                    : -1;
                if (blk < 0 || blk >= g.ap_num_blocks) {
                    if (j == 0 && nb0 == 0) flag_error(g.err, MLA_ERR_OUT_OF_RANGE, b);
                    continue;
                }
                if (n >= D_C) {
                    rope_pair(a0, a1, pp, g.rope.f[(n - D_C) / 2]);
                    rope_pair(a2, a3, pp, g.rope.f[(n - D_C) / 2 + 1]);
                }
                dst = g.ap_cache + ((size_t)blk * BLOCK + pp % BLOCK) * D_QK + n;
            }
            *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(a0, a1), pack_bf16x2(a2, a3));
        }
        cluster_sync();
    }
    if (tid == 0 && *abort_flag) flag_error(g.err, MLA_ERR_TIMEOUT, blockIdx.x);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
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

// bf16 matrix with `rows` rows of `cols` elements, row pitch `ld` elements, as a 2-D map
// with 128-byte swizzled boxes of box_rows x 64 columns.
bool map_2d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t ld,
            uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 array [slices][rows][cols] (contiguous) as a 3-D map with 128-byte-swizzled boxes of
// 32 columns x 128 rows x 1 slice.
bool map_3d_f32(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t slices) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cols, rows, slices};
    cuuint64_t strides[2] = {cols * 4, cols * rows * 4};
    cuuint32_t box[3] = {32, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// shared memory of a CTA of gemm_tc_kernel<.., BN, .., CRED> with ns ring stages
template <int BN, int CRED> int tile_smem(int ns) {
    const int ring = ns * Tile<BN>::STAGE;
    return (CRED != 0 && ring < BM * BN * 4 ? BM * BN * 4 : ring) + SMEM_EXTRA;
}

template <bool NN, int BN, bool ROPE = false, int CRED = 0>
cudaError_t launch_tile(const CUtensorMap &ma, const CUtensorMap &mb, TcGemmArgs g,
                        const GemmParams &p, cudaStream_t stream,
                        const CUtensorMap *mb2 = nullptr, const CUtensorMap *mc1 = nullptr,
                        const CUtensorMap *mc2 = nullptr) {
    using T = Tile<BN>;
    dim3 grid((p.N + BN - 1) / BN, (p.M + BM - 1) / BM, p.batch * p.k_splits);
    const int kblocks = (p.k_per_split + BK - 1) / BK;
    g.ns = kblocks < 1 ? 1 : (kblocks < T::NS ? kblocks : T::NS);
    // Many output tiles of a short product (the prefill up-projections: K = 512, thousands
    // of 128 x 256 tiles): two stages, so that two CTAs share an SM and one's epilogue
    // overlaps the other's loads and MMAs.
    if (CRED == 0 && BN == 256 && (long)grid.x * grid.y * grid.z >= 4L * device_sm_count() &&
        kblocks <= 16)
        g.ns = g.ns < 2 ? g.ns : 2;
    const int smem = tile_smem<BN, CRED>(g.ns);
    // bf16 output through TMA stores when every batch's slice is a column range of one
    // [M][ldc] matrix (x offsets multiples of 64 elements) and the ring holds the tile
    CUtensorMap mc = ma;
    g.tma_c = 0;
    if (CRED != 0) {  // the cluster's reduction writes the output itself
    } else if (ROPE) {  // both outputs through the maps the caller made
        mc = *mc1;
        g.tma_c = 1;
    } else if (p.c_bf16 && !p.c_part && p.N % 64 == 0 && p.c_bstride % 64 == 0 && p.ldc % 8 == 0 &&
        (reinterpret_cast<uintptr_t>(p.c_bf16) & 15) == 0 &&
        (long)(p.batch - 1) * p.c_bstride + p.N <= p.ldc && g.ns * T::STAGE >= BM * BN * 2 &&
        map_2d(&mc, p.c_bf16, (uint64_t)p.ldc, (uint64_t)p.M, (uint64_t)p.ldc, BM))
        g.tma_c = 1;
    else if (p.c_part && p.N % 32 == 0 && (reinterpret_cast<uintptr_t>(p.c_part) & 15) == 0 &&
             g.ns * T::STAGE >= BM * BN * 4 &&
             map_3d_f32(&mc, p.c_part, (uint64_t)p.N, (uint64_t)p.M,
                        (uint64_t)p.k_splits * p.batch))
        g.tma_c = 2;
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<NN, BN, ROPE, CRED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    if (CRED == 0)
        return launch_pdl(gemm_tc_kernel<NN, BN, ROPE, CRED>, grid, dim3(NTHREADS), smem, stream,
                          ma, mb, mc, mb2 ? *mb2 : mb, mc2 ? *mc2 : mc, g);
    // one cluster per output tile: its k-splits along z
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = static_cast<unsigned>(p.k_splits);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<NN, BN, ROPE, CRED>, ma, mb, mc,
                              mb2 ? *mb2 : mb, mc2 ? *mc2 : mc, g);
}

// Clusters of `s` CTAs of a cluster-reduced gemm_tc_kernel at width BN with `ns` ring stages
// that the device holds at once (cudaOccupancyMaxActiveClusters); cached per (BN, s) for the
// last ring asked about.
template <int BN> int cluster_capacity(int s, int ns) {
    static int cap[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
    static int cap_ns[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
    if (s < 2 || s > 8) return 0;
    if (cap[s] > 0 && cap_ns[s] == ns) return cap[s];
    auto kern = gemm_tc_kernel<false, BN, false, 1>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Tile<BN>::SMEM_TOTAL) != cudaSuccess) {
        cudaGetLastError();  // no device: nothing left behind for the next error check
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, s);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = tile_smem<BN, 1>(ns);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = static_cast<unsigned>(s);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 0) {
        cudaGetLastError();  // a refused query leaves no sticky error behind
        return 0;
    }
    cap[s] = n;
    cap_ns[s] = ns;
    return n;
}

RopeFreqs rope_freqs(float theta) {
    RopeFreqs r;
    for (int i = 0; i < D_ROPE / 2; ++i)
        r.f[i] = std::pow(static_cast<double>(theta), -2.0 * i / static_cast<double>(D_ROPE));
    return r;
}

}  // namespace

// 256-wide tiles halve the activation re-reads per weight byte, which pays on long,
// wide products (the output projection); shorter ones do better with a deeper ring and
// fewer k-splits at width 128 (measured).
int gemm_block_n(int N, int K) { return (N >= 4096 && K >= 4096 && N % 256 == 0) ? 256 : 128; }
int gemm_block_n(int M, int N, int K) {
    // many row tiles (prefill up-projections): fewer, longer-lived CTAs at width 256
    if (M >= 1024 && N >= 4096 && N % 256 == 0) return 256;
    // short products (per-head W_UK, K = 128): half as many CTAs, A read half as often
    if (K <= 256 && N >= 512 && N % 256 == 0) return 256;
    return gemm_block_n(N, K);
}

namespace {
// The most k-splits (2..8, at least two k-blocks each, every split non-empty) whose clusters
// of `tiles` output tiles of width bn the device holds at once with room to spare; 0 if none.
int cluster_splits(long tiles, int bn, int kblocks, int *per_out) {
    for (int s = 8; s >= 2; --s) {
        const int per = (kblocks + s - 1) / s;  // k-blocks per split
        const int splits = (kblocks + per - 1) / per;
        if (per < 2 || splits != s) continue;
        const int nsmax = bn == 128 ? Tile<128>::NS : (bn == 224 ? Tile<224>::NS : Tile<256>::NS);
        const int ns = per < nsmax ? per : nsmax;  // the ring launch_tile gives it
        const int cap = bn == 128   ? cluster_capacity<128>(s, ns)
                        : bn == 224 ? cluster_capacity<224>(s, ns)
                                    : cluster_capacity<256>(s, ns);
        // a tenth of the clusters' room left free: clusters are placed only where a whole
        // group of SMs is idle, and with every slot needed one SM still busy with the
        // previous kernel sends a cluster into a second wave (5 splits of the 7168 x 16384
        // output product, 28 clusters where the device holds 28, took 68 us; 4 splits 53)
        if (tiles * 10 <= (long)cap * 9) {
            *per_out = per;
            return s;
        }
    }
    return 0;
}
}  // namespace

// Cluster-reduced split-K for a TN product of one batch with bf16 output: the tile width and
// the most k-splits (2..8, at least two k-blocks each) whose clusters the device holds for
// every output tile at once, with room to spare, taking the width that runs the most CTAs;
// 0 if no such split exists (the caller then writes partials for a finalize kernel).
int gemm_cluster_plan(int M, int N, int K, int *k_per_split, int *block_n) {
    if (M < 1 || N < 4 || N % 4 || K < 2 * BK || K % BK) return 0;
    const int kblocks = K / BK;
    // tile widths: the product's own, and 224 in place of 256 when it divides N (more tiles
    // for the same clusters: the 7168-wide output projection as 32 tiles instead of 28)
    int widths[2] = {gemm_block_n(M, N, K), 0};
    if (widths[0] == 256 && N % 224 == 0) widths[1] = 224;
    int best_s = 0, best_per = 0, best_bn = 0;
    long best_ctas = 0;
    for (int w = 0; w < 2 && widths[w]; ++w) {
        const int bn = widths[w];
        const long tiles = (long)((N + bn - 1) / bn) * ((M + BM - 1) / BM);
        int per = 0;
        const int s = cluster_splits(tiles, bn, kblocks, &per);
        if (s > 0 && tiles * s > best_ctas) {  // the width that runs the most CTAs
            best_ctas = tiles * s;
            best_s = s;
            best_per = per;
            best_bn = bn;
        }
    }
    if (best_s == 0) return 0;
    *k_per_split = best_per * BK;
    if (block_n) *block_n = best_bn;
    return best_s;
}

cudaError_t launch_gemm_tc_cluster(const GemmParams &p, int bn, const ClusterAppend *ap,
                                   cudaStream_t stream, uint32_t *err) {
    if (p.batch != 1 || p.c_part || p.k_splits < 2 || p.k_splits > 8 || p.N % 4)
        return cudaErrorInvalidValue;
    if (!ap && (!p.c_bf16 || p.ldc % 4 || (reinterpret_cast<uintptr_t>(p.c_bf16) & 7)))
        return cudaErrorInvalidValue;
    if (ap && (p.N != D_QK || !ap->pos || !ap->block_table || !ap->cache ||
               (reinterpret_cast<uintptr_t>(ap->cache) & 7)))
        return cudaErrorInvalidValue;
    TcGemmArgs g{};
    g.M = p.M; g.N = p.N; g.K = p.K; g.batch = 1;
    g.k_splits = p.k_splits; g.k_per_split = p.k_per_split;
    g.c_bf16 = p.c_bf16; g.ldc = p.ldc;
    g.err = err;
    if (bn != 128 && bn != 224 && bn != 256) return cudaErrorInvalidValue;
    CUtensorMap ma, mb;
    if (!map_2d(&ma, p.A, (uint64_t)p.lda, (uint64_t)p.M, (uint64_t)p.lda, BM) ||
        !map_2d(&mb, p.B, (uint64_t)p.ldb, (uint64_t)p.N, (uint64_t)p.ldb, bn))
        return cudaErrorInvalidValue;
    if (ap) {
        if (bn != 128) return cudaErrorInvalidValue;
        g.ap_pos = ap->pos; g.ap_bt = ap->block_table; g.ap_max_blocks = ap->max_blocks;
        g.ap_num_blocks = ap->num_blocks; g.ap_cache = ap->cache;
        g.rope = rope_freqs(ap->theta);
        return launch_tile<false, 128, false, 2>(ma, mb, g, p, stream);
    }
    return bn == 256   ? launch_tile<false, 256, false, 1>(ma, mb, g, p, stream)
           : bn == 224 ? launch_tile<false, 224, false, 1>(ma, mb, g, p, stream)
                       : launch_tile<false, 128, false, 1>(ma, mb, g, p, stream);
}

bool gemm_cluster_fits_dq_append(int M, int N1, int K) {
    if (M < 1 || N1 < 4 || N1 % 4 || K < 2 * BK || K % BK) return false;
    const long tiles = (long)((N1 + 127) / 128 + (D_QK + 127) / 128) * ((M + BM - 1) / BM);
    int per = 0;
    return cluster_splits(tiles, 128, K / BK, &per) > 0;
}

// C1 = A B1^T (bf16, row pitch N1) and append's cache rows from A B2^T (N2 = 576), with both
// products' k-splits reduced inside their clusters, in one launch (128-column tiles, each
// product with its own tile range): the two down-projections of a decode step read the same
// hidden states. Returns cudaErrorNotSupported when no cluster split fits the device (the
// caller then runs the products separately).
cudaError_t launch_gemm_tc_cluster_dq_append(const uint16_t *A, int M, int K, const uint16_t *B1,
                                            int N1, uint16_t *C1, const uint16_t *B2,
                                            const ClusterAppend &ap, cudaStream_t stream,
                                            uint32_t *err) {
    constexpr int bn = 128;
    const int N2 = D_QK;
    if (M < 1 || N1 < 4 || N1 % 4 || K < 2 * BK || K % BK || !ap.pos || !ap.block_table ||
        !ap.cache || (reinterpret_cast<uintptr_t>(ap.cache) & 7) ||
        (reinterpret_cast<uintptr_t>(C1) & 7))
        return cudaErrorInvalidValue;
    const int t1 = (N1 + bn - 1) / bn, t2 = (N2 + bn - 1) / bn;
    const long tiles = (long)(t1 + t2) * ((M + BM - 1) / BM);
    int per = 0;
    const int s = cluster_splits(tiles, bn, K / BK, &per);
    if (s == 0) return cudaErrorNotSupported;
    GemmParams p{};
    p.A = A; p.lda = K; p.B = B1; p.ldb = K;
    p.M = M; p.N = (t1 + t2) * bn; p.K = K; p.batch = 1;  // N: the grid's column tiles
    p.k_splits = s; p.k_per_split = per * BK; p.c_bf16 = C1; p.ldc = N1;
    TcGemmArgs g{};
    g.M = M; g.N = N1 + N2; g.K = K; g.batch = 1;
    g.k_splits = s; g.k_per_split = per * BK;
    g.c_bf16 = C1; g.ldc = N1;
    g.err = err;
    g.t1 = t1; g.n1 = N1; g.n2 = N2;
    g.ap_pos = ap.pos; g.ap_bt = ap.block_table; g.ap_max_blocks = ap.max_blocks;
    g.ap_num_blocks = ap.num_blocks; g.ap_cache = ap.cache;
    g.rope = rope_freqs(ap.theta);
    CUtensorMap ma, mb1, mb2;
    if (!map_2d(&ma, A, (uint64_t)K, (uint64_t)M, (uint64_t)K, BM) ||
        !map_2d(&mb1, B1, (uint64_t)K, (uint64_t)N1, (uint64_t)K, bn) ||
        !map_2d(&mb2, B2, (uint64_t)K, (uint64_t)N2, (uint64_t)K, bn))
        return cudaErrorInvalidValue;
    return launch_tile<false, bn, false, 3>(ma, mb1, g, p, stream, &mb2);
}

// Shapes: A is the [rows_a][lda] matrix holding every batch's [M][K] slice at column
// offset batch * a_bx; B is [rows_b][ldb] with every batch's slice at row offset
// batch * b_by (TN: [N][K] slice; NN: [K][N] slice).
cudaError_t launch_gemm_tc(const GemmParams &p, bool nn, cudaStream_t stream, uint32_t *err) {
    TcGemmArgs g{};
    g.M = p.M; g.N = p.N; g.K = p.K; g.batch = p.batch;
    g.k_splits = p.k_splits; g.k_per_split = p.k_per_split;
    g.c_part = p.c_part; g.c_bf16 = p.c_bf16; g.ldc = p.ldc; g.c_bstride = p.c_bstride;
    g.err = err;
    // A: rows = M, columns = lda (the batch slices side by side)
    g.a_bx = static_cast<int>(p.a_bstride);
    CUtensorMap ma, mb;
    if (!map_2d(&ma, p.A, (uint64_t)p.lda, (uint64_t)p.M, (uint64_t)p.lda, BM))
        return cudaErrorInvalidValue;
    const int bn = gemm_block_n(p.M, p.N, p.K);
    g.b_bx = 0;
    g.b_by = static_cast<int>(p.b_bstride / p.ldb);
    if (!nn) {
        // B slices are [N][K] blocks stacked by rows (b_bstride = rows * ldb elements)
        const uint64_t rows = (uint64_t)p.N + (uint64_t)g.b_by * (p.batch - 1);
        if (!map_2d(&mb, p.B, (uint64_t)p.ldb, rows, (uint64_t)p.ldb, bn))
            return cudaErrorInvalidValue;
    } else {
        // B slices are [K][N] blocks stacked by rows, loaded as 64-column groups of BK rows
        const uint64_t rows = (uint64_t)p.K + (uint64_t)g.b_by * (p.batch - 1);
        if (!map_2d(&mb, p.B, (uint64_t)p.ldb, rows, (uint64_t)p.ldb, BK))
            return cudaErrorInvalidValue;
    }
    if (nn) return bn == 256 ? launch_tile<true, 256>(ma, mb, g, p, stream)
                             : launch_tile<true, 128>(ma, mb, g, p, stream);
    return bn == 256 ? launch_tile<false, 256>(ma, mb, g, p, stream)
                     : launch_tile<false, 128>(ma, mb, g, p, stream);
}

// C1 = A B1^T and C2 = RoPE(A B2^T) in one launch: the output tiles of both products side by
// side (TN, no k-split), each 64-column head of C2 rotated pairwise by pos[row] *
// theta^(-2i/64) in the epilogue. The tile width is the narrowest of 128, 192 and 256 whose
// tiles fill at most one wave (at 128 heads: 192 columns, 86 + 43 = 129 CTAs, where 256 gave
// 96), so that as many SMs as possible stream the weights. A [M][K], B1 [N1][K], B2 [N2][K],
// C1 [M][N1], C2 [M][N2], all bf16; N1 and N2 multiples of 64, K of 64, M <= 128.
cudaError_t launch_gemm_tc_rope(const uint16_t *A, int M, int K, const uint16_t *B1, int N1,
                                uint16_t *C1, const uint16_t *B2, int N2, uint16_t *C2,
                                const int32_t *pos, float theta, cudaStream_t stream,
                                uint32_t *err) {
    if (N1 % 64 || N2 % 64 || N1 < 64 || N2 < 64 || K % BK || M > BM) return cudaErrorInvalidValue;
    const int widths[3] = {128, 192, 256};
    int bn = 256;
    for (int w = 0; w < 3; ++w) {
        const int t = (N1 + widths[w] - 1) / widths[w] + (N2 + widths[w] - 1) / widths[w];
        if (t <= device_sm_count()) {
            bn = widths[w];
            break;
        }
    }
    const int t1 = (N1 + bn - 1) / bn, t2 = (N2 + bn - 1) / bn;
    GemmParams p{};
    p.A = A; p.lda = K; p.B = B1; p.ldb = K;
    p.M = M; p.N = (t1 + t2) * bn; p.K = K; p.batch = 1;  // N: the grid's column tiles
    p.k_splits = 1; p.k_per_split = K; p.c_bf16 = C1; p.ldc = N1;
    TcGemmArgs g{};
    g.M = M; g.N = N1 + N2; g.K = K; g.batch = 1;
    g.k_splits = 1; g.k_per_split = K;
    g.c_bf16 = C1; g.ldc = N1;
    g.err = err;
    g.t1 = t1; g.n1 = N1; g.n2 = N2;
    g.rope_pos = pos;
    g.rope = rope_freqs(theta);
    CUtensorMap ma, mb1, mb2, mc1, mc2;
    if (!map_2d(&ma, A, (uint64_t)K, (uint64_t)M, (uint64_t)K, BM) ||
        !map_2d(&mb1, B1, (uint64_t)K, (uint64_t)N1, (uint64_t)K, bn) ||
        !map_2d(&mb2, B2, (uint64_t)K, (uint64_t)N2, (uint64_t)K, bn) ||
        !map_2d(&mc1, C1, (uint64_t)N1, (uint64_t)M, (uint64_t)N1, BM) ||
        !map_2d(&mc2, C2, (uint64_t)N2, (uint64_t)M, (uint64_t)N2, BM))
        return cudaErrorInvalidValue;
    if (bn == 128) return launch_tile<false, 128, true>(ma, mb1, g, p, stream, &mb2, &mc1, &mc2);
    if (bn == 192) return launch_tile<false, 192, true>(ma, mb1, g, p, stream, &mb2, &mc1, &mc2);
    return launch_tile<false, 256, true>(ma, mb1, g, p, stream, &mb2, &mc1, &mc2);
}

}  // namespace mla
