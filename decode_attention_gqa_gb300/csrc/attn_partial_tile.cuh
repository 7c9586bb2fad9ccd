// attn_partial_tile.cuh -- the split partial kernel (steps a1-a6) for a split
// of at most one tile, arranged for the shortest chain of dependent steps:
// 16x8x16 MMAs with their operands in registers, no tensor memory, no merge
// of warp states.
//
// One block per (split sp, KV head hk, sequence s): the static grid of minfer
// "10 · R4" §2.2 with the KV head in place of the query head, so the whole
// group is served from one K/V read (Red Lite dev35 "Change"). The split is
// one tile of TILE rows (128 at head_dim 128, 96 at 256; the wide tiles, one
// block per SM: 256 at 128, 128 at 256), so the block sees each row once and
// its softmax is one pass with a block-wide maximum (§2.1 with a single step).
// Four warps:
//   1. TMA brings the TILE cache rows that end at hi, K and V on separate
//      mbarriers (128-byte swizzled; rows in front of the sequence arrive as
//      zeros, other rows outside the split are earlier rows of the same
//      sequence: finite data that gets weight 0).
//   2. q of the group becomes a 16-row Q tile: hi parts of the scaled q in
//      rows 0-7, lo parts in rows 8-15 (attn_warp_tc.cuh), so q·k keeps about
//      22 bits of q through 16-bit MMA operands.
//   3. S: warp w takes tile rows [w·TILE/4, (w+1)·TILE/4): Q (16 x head_dim)
//      times those K rows, f32 accumulation in registers; slot g's score is C
//      row g plus C row 8 + g.
//   4. a4: each head's maximum over the block (warp maxima through shared
//      memory, one barrier); p = 2^(s - m + OFF), 0 outside the split, stored
//      as a hi/lo pair into a P tile [16 slots][TILE rows] laid over the Q tile.
//   5. a5: O = P · V split by head dimension: warp w takes dimensions
//      [w·head_dim/4, (w+1)·head_dim/4) over all TILE rows, so every warp ends
//      with the block's final accumulator for its dimensions.
//   6. a6: each warp writes its dimensions of oc for every head; one thread
//      per head writes (mx, S), S from the warps' partial sums.
// A wide tile whose split holds at most half its rows runs steps 3-6 on its
// last half only (half the chain; both paths are compiled, the block picks one
// from its row count).
// By block length (Red Lite dev35 "Change": split sp covers [sp·blk, sp·blk +
// blk)) with blk dividing the tile, a second kernel lets one block serve
// SPB = TILE / blk consecutive splits from one tile: one block-wide maximum as
// every split's reference, the sums per split (over 8-row groups through
// shared memory), O = P · V as one sweep over the tile's k-steps that writes
// each split's accumulator at the split's end.
// Several causal query rows: a third kernel serves 16 (query row, head) slots.
#pragma once

#include <type_traits>

#include "attn_device.cuh"
#include "attn_warp_tc.cuh"
#include "attn_warp_tcmq.cuh"

namespace attn {

// A fragment (16 x 16) of a 16-row operand stored like the Q tile (rows of
// COLS 16-bit elements, 128-byte swizzled chunks): k-step kk covers columns
// [16kk, 16kk + 16); matrices (rows 0-7, low 8 columns), (rows 8-15, low 8),
// (rows 0-7, high 8), (rows 8-15, high 8).
template <int COLS>
__device__ __forceinline__ void ldsm_a16(uint32_t (&a)[4], const uint8_t *base, int kk, int lane)
{
    const int i = lane >> 3;
    const int row = (i & 1) * 8 + (lane & 7);
    ldsm_x4(a, base + tile_unit_offset<COLS, 16>(row, 2 * kk + (i >> 1)));
}

// MQ = false: one query row, the G heads of the group in slots 0..G-1, one
// 16-row Q tile (hi parts in rows 0-7, lo parts in 8-15). MQ = true: several
// causal query rows, 16 (query row, head) slots per block, a 16-row hi tile
// and a 16-row lo tile (attn_warp_tcmq.cuh), and P as a hi and a lo tile.
template <int HD, int G, typename KV, bool MQ = false, bool WIDE = false>
struct TileCfg {
    static_assert(HD == 128 || HD == 256, "the one-tile kernel is built for head_dim 128 and 256");
    static_assert(!MQ || HD == 128, "several query rows: head_dim 128 (two blocks per SM would not fit at 256)");
    // rows per block: 128 at head_dim 128 (three blocks per SM), 96 at 256 (two); the
    // wide tile, one block per SM, takes 256 rows at head_dim 128 and 128 at 256
    static constexpr int TILE = HD == 256 ? (WIDE ? 128 : 96) : (WIDE ? 256 : 128);
    static constexpr int MINB = WIDE ? 1 : HD == 256 ? 2 : 3;   // resident blocks per SM
    static constexpr bool IS_WIDE = WIDE;               // half-tile splits run on the tile's last half
    // warps: S rows and O dimensions split NW ways (8 warps were measured slower, on the
    // 128-row tile and on both wide tiles: each warp reads all of Q and P from shared
    // memory, and more warps meet at each barrier)
    static constexpr int NW = 4;
    static constexpr int THREADS = NW * 32;
    static constexpr int WR = TILE / NW;                // S rows per warp (32 or 24)
    static constexpr int DW = HD / NW;                  // O dimensions per warp (32 or 64)
    static constexpr int NS = WR / 8;                   // S n-tiles (8 rows each) per warp (4 or 3)
    static constexpr int KS = HD / 16;                  // S k-steps
    static constexpr int NO = DW / 8;                   // O n-tiles (8 dimensions each) per warp
    static constexpr int KO = TILE / 16;                // O k-steps
    static constexpr int NCH = HD / 64;                 // 128-byte column chunks per row
    static constexpr int GRANULE = TILE;                // count-mode chunks: whole tiles, or 16 rows
                                                        // near a tile (split_range_tile)
    static constexpr bool Q_REGS = KS <= 8 && !MQ;      // Q fragments held in registers
    using QStage = typename std::conditional<MQ, TcWarpMQ<HD, 16, NW, KV>, TcWarp<HD, G, NW, KV>>::type;
    static constexpr uint32_t Q_AREA = (MQ ? 2u : 1u) * QStage::QT_BYTES;   // Q tiles, before the scales
    static constexpr uint32_t TILE_BYTES = (uint32_t)TILE * HD * 2;
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = TILE_BYTES;
    static constexpr uint32_t OFF_Q = 2 * TILE_BYTES;   // Q tile, then per-head scales
    // P tile(s): 16 rows of TILE elements in 128-byte swizzled chunks of 64 (MQ: hi, then lo),
    // over the Q tile once S is done where they fit there, else after the scales
    static constexpr uint32_t P_TILE = 16u * ((TILE + 63) / 64 * 64) * 2;
    static constexpr uint32_t P_BYTES = (MQ ? 2u : 1u) * P_TILE;
    static constexpr bool P_OVER_Q = P_BYTES <= Q_AREA;
    static constexpr uint32_t OFF_P = P_OVER_Q ? OFF_Q : OFF_Q + (QStage::EXTRA_BYTES + 1023) / 1024 * 1024;
    // maxima per warp; sums per warp, or per 8-row group (the several-split kernel); RSL slots each
    static constexpr int NRED = MQ ? NW : (TILE / 8 > NW ? TILE / 8 : NW);
    static constexpr int RSL = MQ ? 16 : 8;
    static constexpr uint32_t OFF_RED = P_OVER_Q ? OFF_Q + (QStage::EXTRA_BYTES + 15) / 16 * 16
                                                 : OFF_P + P_BYTES;                   // [2][NRED][RSL] floats
    static constexpr uint32_t OFF_BAR = OFF_RED + 2 * NRED * RSL * 4;                   // 2 mbarriers, flags
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 2 * 8 + 16 + 1024;                 // + alignment slack
    static constexpr float OFF = 7.f;                   // p headroom: p <= 2^OFF
    static_assert(TILE % 32 == 0 && WR % 8 == 0 && DW % 16 == 0, "fragment shapes");
    static_assert((TILE * 128) % 1024 == 0, "swizzled chunks stay 1024-aligned");
    static_assert(MINB * (SMEM_BYTES + 1024) <= 233472u, "resident blocks per SM");
};


// a3 for one warp: S = Q · Kᵀ over tile rows r0 .. r0 + WR - 1 (Q fragments in
// registers, K by ldmatrix), even and odd k-steps in separate accumulators;
// head g's score for row r0 + 8j + 2t + e is (c[.][j][e] + c[.][j][2 + e]).
template <class Cfg, int HD, typename KV, int NS = Cfg::NS>
__device__ __forceinline__ void tile_scores(const uint8_t *smem, int r0, int lane, float (&c)[2][NS][4])
{
    constexpr int TILE = Cfg::TILE, KS = Cfg::KS;
    const uint8_t *qt = smem + Cfg::OFF_Q;
    const int i8 = lane >> 3;
    uint32_t qa[Cfg::Q_REGS ? KS : 1][4];
    if constexpr (Cfg::Q_REGS) {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) ldsm_a16<HD>(qa[kk], qt, kk, lane);
    }
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
        uint32_t aq[4];
        if constexpr (Cfg::Q_REGS) {
#pragma unroll
            for (int i = 0; i < 4; ++i) aq[i] = qa[kk][i];
        } else {
            ldsm_a16<HD>(aq, qt, kk, lane);
        }
#pragma unroll
        for (int j = 0; j + 1 < NS; j += 2) {
            // (rows 8j..8j+7, dims lo 8), (.., hi 8), (rows 8j+8.., lo 8), (.., hi 8)
            uint32_t b[4];
            const int krow = r0 + 8 * j + (i8 >> 1) * 8 + (lane & 7);
            ldsm_x4(b, smem + Cfg::OFF_K + tile_unit_offset<HD, TILE>(krow, 2 * kk + (i8 & 1)));
            mma_16816<KV>(c[kk & 1][j], aq, b[0], b[1]);
            mma_16816<KV>(c[kk & 1][j + 1], aq, b[2], b[3]);
        }
        if constexpr (NS % 2 == 1) {
            // the last 8 rows alone: (dims lo 8), (dims hi 8); lanes 16-31 repeat the addresses
            uint32_t b[2];
            const int krow = r0 + 8 * (NS - 1) + (lane & 7);
            ldsm_x2(b, smem + Cfg::OFF_K + tile_unit_offset<HD, TILE>(krow, 2 * kk + (i8 & 1)));
            mma_16816<KV>(c[kk & 1][NS - 1], aq, b[0], b[1]);
        }
    }
}

// p of head g for tile rows (r, r + 1) as a hi/lo pair into the P tile
// [16 slots][TILE rows]: hi in slot row g, lo in slot row 8 + g.
template <class Cfg, typename KV>
__device__ __forceinline__ void store_p_pair(uint8_t *pt, int r, int g, int t, float p0, float p1)
{
    const uint32_t hw = float2_to_kv2<KV>(p0, p1);
    const float2 f = kv2_to_float2<KV>(hw);
    const uint32_t lw = float2_to_kv2<KV>(p0 - f.x, p1 - f.y);
    // row pair (r, r + 1) of unit r / 8, 4 bytes apart per t
    *reinterpret_cast<uint32_t *>(pt + tile_unit_offset<Cfg::TILE, 16>(g, r >> 3) + 4 * t) = hw;
    *reinterpret_cast<uint32_t *>(pt + tile_unit_offset<Cfg::TILE, 16>(8 + g, r >> 3) + 4 * t) = lw;
}

// a5 for one warp, one k-step: o += P · V over tile rows 16kk .. 16kk + 15 for
// dimensions d0 .. d0 + DW - 1.
template <class Cfg, int HD, typename KV>
__device__ __forceinline__ void tile_pv_step(const uint8_t *smem, int d0, int lane, int kk, float (&o)[Cfg::NO][4])
{
    constexpr int TILE = Cfg::TILE, NO = Cfg::NO;
    const int i8 = lane >> 3;
    uint32_t ap[4];                       // P rows (slots) x tile rows 16kk .. 16kk + 15
    ldsm_a16<TILE>(ap, smem + Cfg::OFF_P, kk, lane);
    const int vrow = 16 * kk + (i8 & 1) * 8 + (lane & 7);
#pragma unroll
    for (int j = 0; j < NO; j += 2) {
        // (rows 0-7, dims j), (rows 8-15, dims j), (0-7, j+1), (8-15, j+1)
        uint32_t b[4];
        ldsm_x4_trans(b, smem + Cfg::OFF_V + tile_unit_offset<HD, TILE>(vrow, (d0 >> 3) + j + (i8 >> 1)));
        mma_16816<KV>(o[j], ap, b[0], b[1]);
        mma_16816<KV>(o[j + 1], ap, b[2], b[3]);
    }
}

// o += P · V over k-steps [k0, k1), even and odd k-steps into o[0] and o[1]
// (two independent MMA chains).
template <class Cfg, int HD, typename KV>
__device__ __forceinline__ void tile_pv(const uint8_t *smem, int d0, int lane, int k0, int k1,
                                        float (&o)[2][Cfg::NO][4])
{
    for (int kk = k0; kk < k1; kk += 2) {
        tile_pv_step<Cfg, HD, KV>(smem, d0, lane, kk, o[0]);
        if (kk + 1 < k1) tile_pv_step<Cfg, HD, KV>(smem, d0, lane, kk + 1, o[1]);
    }
}

template <class Cfg, int HD, int G, typename KV>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MINB)
attn_split_partial_tile(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const PartialArgs a)
{
    constexpr int TILE = Cfg::TILE, NS = Cfg::NS, NO = Cfg::NO, KO = Cfg::KO;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);    // [0] K landed, [1] V landed
    volatile int *flags = reinterpret_cast<volatile int *>(bar + 2);     // [0] abort
    float *red_m = reinterpret_cast<float *>(smem + Cfg::OFF_RED);      // [NW][8] warp maxima
    float *red_l = red_m + Cfg::NRED * Cfg::RSL;                        // [NW][8] warp sums

    const int hk = blockIdx.x, sp = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = a.n_splits;
    const size_t heads = (size_t)a.n_head;

    // Dependencies as in attn_partial.cuh: with kv_stable the positions read
    // and the tile copies go ahead of the grid dependency, q waits for it.
    const bool stable = a.kv_stable != 0;
    if (tid == 32)
        prefetch_l2(a.q + ((size_t)s * a.n_head + (size_t)hk * G) * HD, (uint32_t)(G * HD * sizeof(float)));
    if (!stable) pdl_wait();
    pdl_launch_dependents();

    // a1: rows attended and this split's rows; an empty split leaves at once
    bool pos_ok;
    const int64_t nkv = rows_attended(a, s, sp == 0 && hk == 0 && tid == 0, &pos_ok);
    int64_t lo, hi;
    split_range_tile(nkv, sp, P, a.split_len, Cfg::TILE, Cfg::IS_WIDE, lo, hi);
    if (lo >= hi) {
        if (stable) pdl_wait();               // the workspace may still be read by the previous grid
        if (tid < G) a.ws_ml[((size_t)s * heads + (size_t)hk * G + tid) * P + sp] = make_float2(-INFINITY, 0.f);
        return;
    }
    const int n = (int)(hi - lo);             // 1..TILE rows: the tile's last n rows
    const int row_first = (int)(hi - TILE);   // negative near the sequence start: zero rows

    if (tid == 0) {
        mbar_init(bar + 0, 1);
        mbar_init(bar + 1, 1);
        flags[0] = 0;
        fence_barrier_init();
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        mbar_arrive_expect_tx(bar + 0, Cfg::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < Cfg::NCH; ++c)
            tma_load_4d(smem + Cfg::OFF_K + c * (Cfg::TILE_BYTES / Cfg::NCH), &kmap, bar + 0, c * 64, hk, row_first, s);
        mbar_arrive_expect_tx(bar + 1, Cfg::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < Cfg::NCH; ++c)
            tma_load_4d(smem + Cfg::OFF_V + c * (Cfg::TILE_BYTES / Cfg::NCH), &vmap, bar + 1, c * 64, hk, row_first, s);
    }

    // a2, while the tile is in flight: the Q tile and the per-head scales
    if (stable) pdl_wait();
    // Fused append: the split ending at nkv holds the new row nkv - 1 as the
    // tile's last row, which is in the last warp's S rows; that warp fetches it
    // now (one 16-byte unit per lane, issued before q's loads so that both are in
    // flight together) and writes each half into its tile and the cache once that
    // tile has landed (V's before the barrier that precedes any read of V).
    constexpr int NU = HD / 8;                    // 16-byte units per row
    constexpr int NJ = 2 * NU / 32;               // units of the new K and V rows per lane
    static_assert(2 * NU % 32 == 0, "whole units per lane");
    const bool appending = a.k_new != nullptr && pos_ok && hi == nkv && warp == Cfg::NW - 1;
    uint4 newrow[NJ];
    if (appending) {
        const size_t src = ((size_t)s * a.n_kv_head + hk) * HD;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int i = lane + 32 * j;
            newrow[j] = ld_dep(reinterpret_cast<const uint4 *>((i < NU ? a.k_new : a.v_new) + src) + (i % NU));
        }
    }
    Cfg::QStage::template prepare<Cfg::THREADS>(smem + Cfg::OFF_Q, a, s, hk, 0, tid);
    __syncthreads();

    const float inv = reinterpret_cast<const float *>(smem + Cfg::OFF_Q + Cfg::QStage::QT_BYTES)[lane >> 2];
    const int g = lane >> 2, t = lane & 3;
    bool ok = mbar_wait_bounded(bar + 0, 0);
    ok = __all_sync(0xffffffffu, ok);
    // the new row's K half into the K tile and the cache once K has landed (S reads
    // it); its V half waits for V below, so that S does not
    const size_t new_dst = ((size_t)((int64_t)s * a.cap + nkv - 1) * a.n_kv_head + hk) * HD;
    auto put_new_row = [&](bool k_half) {
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int i = lane + 32 * j;
            if ((i < NU) == k_half) {
                *reinterpret_cast<uint4 *>(smem + (k_half ? Cfg::OFF_K : Cfg::OFF_V) +
                                           tile_unit_offset<HD, TILE>(TILE - 1, i % NU)) = newrow[j];
                reinterpret_cast<uint4 *>((k_half ? a.k_w : a.v_w) + new_dst)[i % NU] = newrow[j];
            }
        }
        __syncwarp();
    };
    if (ok && appending) put_new_row(true);
    if (!ok && lane == 0) { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); }

    // a3 .. a6 for NSX S n-tiles per warp from tile row 16 K0 on: the whole tile
    // (NSX = NS, K0 = 0), or, in a wide tile, its last half only when the split has
    // no more rows (NSX = NS / 2, K0 = KO / 2: half the chain)
    auto rows_from = [&](auto nsx_c, auto k0_c) {
        constexpr int NSX = decltype(nsx_c)::value, K0 = decltype(k0_c)::value;
        // ---- a3: S for this warp's rows r0 .. r0 + 8 NSX - 1 ----
        const int r0 = 16 * K0 + warp * 8 * NSX;
        float sc[NSX][2];                         // head g, rows r0 + 8j + 2t + {0, 1}
        {
            float c[2][NSX][4];
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int j = 0; j < NSX; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) c[e][j][i] = 0.f;
            if (ok) tile_scores<Cfg, HD, KV, NSX>(smem, r0, lane, c);
#pragma unroll
            for (int j = 0; j < NSX; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = r0 + 8 * j + 2 * t + e;   // tile row
                    const float v = ((c[0][j][e] + c[1][j][e]) + (c[0][j][2 + e] + c[1][j][2 + e])) * inv;
                    sc[j][e] = r >= TILE - n ? v : -INFINITY;
                }
        }
        // ---- a4: each head's maximum over the block ----
        {
            float m = -INFINITY;
#pragma unroll
            for (int j = 0; j < NSX; ++j) m = fmaxf(m, fmaxf(sc[j][0], sc[j][1]));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            if (t == 0) red_m[warp * 8 + g] = m;
        }
        __syncthreads();                          // the maxima are in; S is done, so Q is dead
        float M = red_m[g];
#pragma unroll
        for (int w = 1; w < Cfg::NW; ++w) M = fmaxf(M, red_m[w * 8 + g]);
        const float base = M - Cfg::OFF;          // M is finite: the split has rows in every block
        {
            float lsum = 0.f;
            uint8_t *pt = smem + Cfg::OFF_P;
#pragma unroll
            for (int j = 0; j < NSX; ++j) {
                const float p0 = ex2(sc[j][0] - base), p1 = ex2(sc[j][1] - base);   // 0 at -inf
                lsum += p0 + p1;
                store_p_pair<Cfg, KV>(pt, r0 + 8 * j, g, t, p0, p1);
            }
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
            lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
            if (t == 0) red_l[warp * 8 + g] = lsum;
        }
        bool vok = ok;
        if (vok) vok = __all_sync(0xffffffffu, mbar_wait_bounded(bar + 1, 0));
        if (vok && appending) put_new_row(false);
        if (ok && !vok && lane == 0) { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); }
        __syncthreads();                          // P and the sums are in; every V wait is done
        // ---- a5: O = P · V for this warp's dimensions d0 .. d0 + DW - 1 ----
        const int d0 = warp * Cfg::DW;
        const bool abort = flags[0] != 0;         // the same for every thread past the barrier
        if (!abort) {
            float o[2][NO][4];
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int j = 0; j < NO; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[e][j][i] = 0.f;
#pragma unroll
            for (int kk = K0; kk < KO; kk += 2) {
                tile_pv_step<Cfg, HD, KV>(smem, d0, lane, kk, o[0]);
                if (kk + 1 < KO) tile_pv_step<Cfg, HD, KV>(smem, d0, lane, kk + 1, o[1]);
            }
            // ---- a6: oc of every head for these dimensions; (mx, S) per head ----
            if (g < G) {
                float *dst = a.ws_o + (((size_t)s * heads + (size_t)hk * G + g) * P + sp) * HD + d0 + 2 * t;
#pragma unroll
                for (int j = 0; j < NO; ++j)
                    *reinterpret_cast<float2 *>(dst + 8 * j) =
                        make_float2((o[0][j][0] + o[1][j][0]) + (o[0][j][2] + o[1][j][2]),
                                    (o[0][j][1] + o[1][j][1]) + (o[0][j][3] + o[1][j][3]));
            }
            if (warp == 0 && t == 0 && g < G) {
                float L = 0.f;
#pragma unroll
                for (int w = 0; w < Cfg::NW; ++w) L += red_l[w * 8 + g];
                a.ws_ml[((size_t)s * heads + (size_t)hk * G + g) * P + sp] = make_float2(base, L);
            }
        } else if (tid == 0) {
            // nothing may still be writing shared memory when the block exits:
            // wait (bounded) for both copies before leaving
            (void)mbar_wait_bounded(bar + 0, 0);
            (void)mbar_wait_bounded(bar + 1, 0);
        }
    };
    if constexpr (Cfg::IS_WIDE) {
        if (n <= TILE / 2) rows_from(std::integral_constant<int, NS / 2>{}, std::integral_constant<int, KO / 2>{});
        else rows_from(std::integral_constant<int, NS>{}, std::integral_constant<int, 0>{});
    } else {
        rows_from(std::integral_constant<int, NS>{}, std::integral_constant<int, 0>{});
    }
}

// By block length with blk = split_len dividing TILE (and a multiple of 16):
// block b serves the SPB = TILE / blk splits b·SPB .. b·SPB + SPB - 1, whose
// rows [b·TILE, b·TILE + TILE) are one tile starting at row b·TILE. Each split's
// (mx, S, oc) is relative to the block's per-head maximum (one reference for the
// block, as in the single-split kernel); the combine rescales them. Cache
// rows of that tile at or past nkv (in the last block only; all within cap,
// and rows past cap arrive as zeros) are read but never used: their scores
// are masked and their V rows are set to zero in shared memory before P · V,
// so whatever the cache holds there cannot reach the result.
template <class Cfg, int HD, int G, typename KV>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MINB)
attn_split_partial_tile_ms(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const PartialArgs a)
{
    constexpr int TILE = Cfg::TILE, NS = Cfg::NS, NO = Cfg::NO;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);    // [0] K landed, [1] V landed
    volatile int *flags = reinterpret_cast<volatile int *>(bar + 2);     // [0] abort
    float *red_m = reinterpret_cast<float *>(smem + Cfg::OFF_RED);      // [NW][8] warp maxima
    float *red_l = red_m + Cfg::NRED * Cfg::RSL;                        // [TILE / 8][8] group sums

    const int hk = blockIdx.x, b = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = a.n_splits, blk = a.split_len, SPB = TILE / blk, GPS = blk / 8;   // 8-row groups per split
    const size_t heads = (size_t)a.n_head;

    const bool stable = a.kv_stable != 0;
    if (tid == 32)
        prefetch_l2(a.q + ((size_t)s * a.n_head + (size_t)hk * G) * HD, (uint32_t)(G * HD * sizeof(float)));
    if (!stable) pdl_wait();
    pdl_launch_dependents();

    // a1: rows attended; this block's rows are [row0, row0 + nv)
    bool pos_ok;
    const int64_t nkv = rows_attended(a, s, b == 0 && hk == 0 && tid == 0, &pos_ok);
    const int64_t row0 = (int64_t)b * TILE;
    const int nv = nkv > row0 ? (int)(nkv - row0 < TILE ? nkv - row0 : TILE) : 0;
    auto write_empty = [&](int j0) {
        // (mx, S) = (-inf, 0) for the splits j0 .. SPB - 1 of this block
        for (int i = tid; i < (SPB - j0) * 8; i += Cfg::THREADS) {
            const int j = j0 + i / 8, gg = i % 8, sp = b * SPB + j;
            if (gg < G && sp < P)
                a.ws_ml[((size_t)s * heads + (size_t)hk * G + gg) * P + sp] = make_float2(-INFINITY, 0.f);
        }
    };
    if (nv == 0) {
        if (stable) pdl_wait();               // the workspace may still be read by the previous grid
        write_empty(0);
        return;
    }
    const int nsplit = (nv + blk - 1) / blk;  // splits of this block with rows (the rest are empty)

    if (tid == 0) {
        mbar_init(bar + 0, 1);
        mbar_init(bar + 1, 1);
        flags[0] = 0;
        fence_barrier_init();
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        mbar_arrive_expect_tx(bar + 0, Cfg::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < Cfg::NCH; ++c)
            tma_load_4d(smem + Cfg::OFF_K + c * (Cfg::TILE_BYTES / Cfg::NCH), &kmap, bar + 0, c * 64, hk, (int)row0, s);
        mbar_arrive_expect_tx(bar + 1, Cfg::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < Cfg::NCH; ++c)
            tma_load_4d(smem + Cfg::OFF_V + c * (Cfg::TILE_BYTES / Cfg::NCH), &vmap, bar + 1, c * 64, hk, (int)row0, s);
    }

    if (stable) pdl_wait();
    Cfg::QStage::template prepare<Cfg::THREADS>(smem + Cfg::OFF_Q, a, s, hk, 0, tid);
    // Fused append: the new row nkv - 1 is tile row nv - 1 of the block that
    // holds it; the warp whose S rows contain it writes it into both tiles and
    // the cache once they have landed, before the barrier that precedes any
    // read of V.
    constexpr int NU = HD / 8;
    constexpr int NJ = 2 * NU / 32;
    static_assert(2 * NU % 32 == 0, "whole units per lane");
    const bool appending = a.k_new != nullptr && pos_ok && row0 + nv == nkv && warp == (nv - 1) / Cfg::WR;
    uint4 newrow[NJ];
    if (appending) {
        const size_t src = ((size_t)s * a.n_kv_head + hk) * HD;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int i = lane + 32 * j;
            newrow[j] = ld_dep(reinterpret_cast<const uint4 *>((i < NU ? a.k_new : a.v_new) + src) + (i % NU));
        }
    }
    if (nsplit < SPB) write_empty(nsplit);    // before the barrier: the workspace is ours past the wait
    __syncthreads();

    const float inv = reinterpret_cast<const float *>(smem + Cfg::OFF_Q + Cfg::QStage::QT_BYTES)[lane >> 2];
    const int g = lane >> 2, t = lane & 3;
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar + 0, 0));
    if (ok && appending) {
        const bool vl = __all_sync(0xffffffffu, mbar_wait_bounded(bar + 1, 0));
        if (vl) {
            const size_t dst = ((size_t)((int64_t)s * a.cap + nkv - 1) * a.n_kv_head + hk) * HD;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int i = lane + 32 * j;
                uint8_t *tile = smem + (i < NU ? Cfg::OFF_K : Cfg::OFF_V);
                *reinterpret_cast<uint4 *>(tile + tile_unit_offset<HD, TILE>(nv - 1, i % NU)) = newrow[j];
                reinterpret_cast<uint4 *>((i < NU ? a.k_w : a.v_w) + dst)[i % NU] = newrow[j];
            }
            __syncwarp();
        }
        ok = vl;
    }
    if (!ok && lane == 0) { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); }

    // ---- a3: S for this warp's rows r0 .. r0 + WR - 1 (rows at or past nv masked) ----
    const int r0 = warp * Cfg::WR;
    float sc[NS][2];
    {
        float c[2][NS][4];
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int j = 0; j < NS; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) c[e][j][i] = 0.f;
        if (ok) tile_scores<Cfg, HD, KV>(smem, r0, lane, c);
#pragma unroll
        for (int j = 0; j < NS; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = r0 + 8 * j + 2 * t + e;
                const float v = ((c[0][j][e] + c[1][j][e]) + (c[0][j][2 + e] + c[1][j][2 + e])) * inv;
                sc[j][e] = r < nv ? v : -INFINITY;
            }
    }
    // ---- a4: each head's maximum over the block's rows, the reference of all of its
    // splits (every split's p = 2^(s - M + OFF) with M >= its own maximum: a split far
    // below M contributes equally little to the combined result), then each head's sum
    // per 8-row group ----
    {
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < NS; ++j) m = fmaxf(m, fmaxf(sc[j][0], sc[j][1]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        if (t == 0) red_m[warp * 8 + g] = m;
    }
    __syncthreads();                          // the maxima are in; S is done, so Q is dead
    float M = red_m[g];
#pragma unroll
    for (int w = 1; w < Cfg::NW; ++w) M = fmaxf(M, red_m[w * 8 + g]);
    const float base = M - Cfg::OFF;          // M is finite: the block has rows before nv
    {
        uint8_t *pt = smem + Cfg::OFF_P;
#pragma unroll
        for (int j = 0; j < NS; ++j) {
            const float p0 = ex2(sc[j][0] - base), p1 = ex2(sc[j][1] - base);
            store_p_pair<Cfg, KV>(pt, r0 + 8 * j, g, t, p0, p1);
            float l = p0 + p1;
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            if (t == 0) red_l[(r0 / 8 + j) * 8 + g] = l;
        }
    }
    bool vok = ok;
    if (vok && !appending) vok = __all_sync(0xffffffffu, mbar_wait_bounded(bar + 1, 0));
    if (ok && !vok && lane == 0) { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); }
    if (vok && nv < TILE) {
        // V rows at or past nkv in this warp's row range: zero, so P = 0 there meets 0
        const int rlo = r0 > nv ? r0 : nv, rhi = r0 + Cfg::WR;
        for (int i = lane; i < (rhi - rlo) * NU; i += 32)
            if (rlo < rhi)
                *reinterpret_cast<uint4 *>(smem + Cfg::OFF_V + tile_unit_offset<HD, TILE>(rlo + i / NU, i % NU)) =
                    make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();                          // P, the sums and the zeroed rows are in
    // ---- a5, a6: per split, O = P · V over its k-steps, oc and (mx, S) written ----
    const int d0 = warp * Cfg::DW;
    const bool abort = flags[0] != 0;
    if (!abort) {
        // one pass over the tile's k-steps, fully unrolled; after each split's
        // KPS k-steps its accumulator is written out and cleared (the splits
        // past nsplit hold P = 0 and are not written)
        const int KPS = blk / 16;             // k-steps per split
        float o[NO][4];
#pragma unroll
        for (int jj = 0; jj < NO; ++jj)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[jj][i] = 0.f;
        int left = KPS, j = 0;
        float *dst = a.ws_o + (((size_t)s * heads + (size_t)hk * G + g) * P + (size_t)b * SPB) * HD + d0 + 2 * t;
#pragma unroll
        for (int kk = 0; kk < Cfg::KO; ++kk) {
            tile_pv_step<Cfg, HD, KV>(smem, d0, lane, kk, o);
            if (--left == 0) {
                if (j < nsplit && g < G && b * SPB + j < P) {
#pragma unroll
                    for (int jj = 0; jj < NO; ++jj)
                        *reinterpret_cast<float2 *>(dst + 8 * jj) =
                            make_float2(o[jj][0] + o[jj][2], o[jj][1] + o[jj][3]);
                }
#pragma unroll
                for (int jj = 0; jj < NO; ++jj)
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[jj][i] = 0.f;
                left = KPS;
                ++j;
                dst += HD;
            }
        }
        // (mx, S) of every non-empty split: thread (j, head); mx is the block's reference
        for (int i = tid; i < nsplit * 8; i += Cfg::THREADS) {
            const int j = i / 8, gg = i % 8, sp = b * SPB + j;
            if (gg < G && sp < P) {
                float Mh = red_m[gg], L = 0.f;
                for (int w = 1; w < Cfg::NW; ++w) Mh = fmaxf(Mh, red_m[w * 8 + gg]);
                for (int k = 0; k < GPS; ++k) L += red_l[(j * GPS + k) * 8 + gg];
                a.ws_ml[((size_t)s * heads + (size_t)hk * G + gg) * P + sp] = make_float2(Mh - Cfg::OFF, L);
            }
        }
    } else if (tid == 0) {
        (void)mbar_wait_bounded(bar + 0, 0);
        (void)mbar_wait_bounded(bar + 1, 0);
    }
}

// Several causal query rows (TileCfg<HD, 16, KV, true>): block (KV head, query
// group qg, split sp) serves 16 (query row, head) slots of one KV head from one
// tile. The slots' q is a hi and a lo Q tile; S accumulates the hi and the lo
// MMA of each step into one fragment, so a thread holds slots g and g + 8 of
// its rows directly. Slot i (query row t) sees cache rows [0, nkv - n_q + t];
// a slot that sees no row of the split writes (-inf, 0). P is a hi and a lo
// tile over the Q tiles, and O = P · V accumulates both into one fragment.
template <class Cfg, int HD, typename KV>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MINB)
attn_split_partial_tile_mq(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const PartialArgs a)
{
    constexpr int TILE = Cfg::TILE, NS = Cfg::NS, NO = Cfg::NO, KS = Cfg::KS, KO = Cfg::KO;
    using QS = typename Cfg::QStage;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);    // [0] K landed, [1] V landed
    volatile int *flags = reinterpret_cast<volatile int *>(bar + 2);     // [0] abort
    float *red_m = reinterpret_cast<float *>(smem + Cfg::OFF_RED);      // [NW][16] warp maxima
    float *red_l = red_m + Cfg::NRED * Cfg::RSL;                        // [NW][16] warp sums

    const int hk = blockIdx.x / a.qgroups, qg = blockIdx.x % a.qgroups, sp = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = a.n_splits;
    const size_t heads = (size_t)a.n_q * a.n_head;         // partial heads per sequence

    const bool stable = a.kv_stable != 0;
    if (tid == 32) {
        // q of this block's slots into L2 (query rows t0..t1 of the group's heads)
        const int G = a.group;
        const int t0 = qg * 16 / G, t1 = min(a.n_q - 1, (qg * 16 + 15) / G);
        for (int t = t0; t <= t1; ++t)
            prefetch_l2(a.q + (((size_t)s * a.n_q + t) * a.n_head + (size_t)hk * G) * HD,
                        (uint32_t)(G * HD * sizeof(float)));
    }
    if (!stable) pdl_wait();
    pdl_launch_dependents();

    bool pos_ok;
    const int64_t nkv = rows_attended(a, s, sp == 0 && blockIdx.x == 0 && tid == 0, &pos_ok);
    int64_t lo, hi;
    split_range_tile(nkv, sp, P, a.split_len, Cfg::TILE, Cfg::IS_WIDE, lo, hi);
    if (lo >= hi) {
        if (stable) pdl_wait();
        if (tid < 16) {
            const int hp = QS::slot_head(a, hk, qg, tid);
            if (hp >= 0) a.ws_ml[((size_t)s * heads + hp) * P + sp] = make_float2(-INFINITY, 0.f);
        }
        return;
    }
    const int n = (int)(hi - lo);
    const int row_first = (int)(hi - TILE);

    if (tid == 0) {
        mbar_init(bar + 0, 1);
        mbar_init(bar + 1, 1);
        flags[0] = 0;
        fence_barrier_init();
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        mbar_arrive_expect_tx(bar + 0, Cfg::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < Cfg::NCH; ++c)
            tma_load_4d(smem + Cfg::OFF_K + c * (Cfg::TILE_BYTES / Cfg::NCH), &kmap, bar + 0, c * 64, hk, row_first, s);
        mbar_arrive_expect_tx(bar + 1, Cfg::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < Cfg::NCH; ++c)
            tma_load_4d(smem + Cfg::OFF_V + c * (Cfg::TILE_BYTES / Cfg::NCH), &vmap, bar + 1, c * 64, hk, row_first, s);
    }

    if (stable) pdl_wait();
    QS::template prepare<Cfg::THREADS>(smem + Cfg::OFF_Q, a, s, hk, qg, tid);
    __syncthreads();

    const uint8_t *qhi = smem + Cfg::OFF_Q, *qlo = qhi + QS::QT_BYTES;
    const float *inv = reinterpret_cast<const float *>(smem + Cfg::OFF_Q + 2 * QS::QT_BYTES);
    const int *qrow = reinterpret_cast<const int *>(inv + 16);
    const int g = lane >> 2, t = lane & 3, i8 = lane >> 3;
    // this thread's slots g and g + 8: scale, and the last cache row each may see
    float isc[2];
    int64_t last[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        isc[k] = inv[g + 8 * k];
        last[k] = qrow[g + 8 * k] >= 0 ? nkv - a.n_q + qrow[g + 8 * k] : -1;
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar + 0, 0));
    if (!ok && lane == 0) { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); }

    // a3 .. a6 for NSX S n-tiles per warp from tile row 16 K0 on: the whole tile, or,
    // in a wide tile, its last half only when the split has no more rows
    auto rows_from = [&](auto nsx_c, auto k0_c) {
        constexpr int NSX = decltype(nsx_c)::value, K0 = decltype(k0_c)::value;
        // ---- a3: S for rows r0 .. r0 + 8 NSX - 1, hi and lo q into one accumulator ----
        const int r0 = 16 * K0 + warp * 8 * NSX;
        float sc[NSX][2][2];                      // [n-tile][slot g, g + 8][row 2t, 2t + 1]
        {
            float c[2][NSX][4];
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int j = 0; j < NSX; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) c[e][j][i] = 0.f;
            if (ok) {
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    uint32_t ah[4], al[4];
                    ldsm_a16<HD>(ah, qhi, kk, lane);
                    ldsm_a16<HD>(al, qlo, kk, lane);
#pragma unroll
                    for (int j = 0; j < NSX; j += 2) {
                        uint32_t b[4];
                        const int krow = r0 + 8 * j + (i8 >> 1) * 8 + (lane & 7);
                        ldsm_x4(b, smem + Cfg::OFF_K + tile_unit_offset<HD, TILE>(krow, 2 * kk + (i8 & 1)));
                        mma_16816<KV>(c[kk & 1][j], ah, b[0], b[1]);
                        mma_16816<KV>(c[kk & 1][j], al, b[0], b[1]);
                        mma_16816<KV>(c[kk & 1][j + 1], ah, b[2], b[3]);
                        mma_16816<KV>(c[kk & 1][j + 1], al, b[2], b[3]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < NSX; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = r0 + 8 * j + 2 * t + e;
                    const int64_t row = hi - TILE + r;              // the cache row
                    const bool in_split = r >= TILE - n;
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const float v = (c[0][j][2 * k + e] + c[1][j][2 * k + e]) * isc[k];
                        sc[j][k][e] = in_split && row <= last[k] ? v : -INFINITY;
                    }
                }
        }
        // ---- a4: each slot's maximum over the block ----
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            float m = -INFINITY;
#pragma unroll
            for (int j = 0; j < NSX; ++j) m = fmaxf(m, fmaxf(sc[j][k][0], sc[j][k][1]));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            if (t == 0) red_m[warp * 16 + g + 8 * k] = m;
        }
        __syncthreads();                          // the maxima are in; S is done, so the Q tiles are dead
        float base[2];
        bool none[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            float M = red_m[g + 8 * k];
#pragma unroll
            for (int w = 1; w < Cfg::NW; ++w) M = fmaxf(M, red_m[w * 16 + g + 8 * k]);
            none[k] = M == -INFINITY;             // the slot sees no row of this split
            base[k] = M - Cfg::OFF;
        }
        {
            uint8_t *phi = smem + Cfg::OFF_P, *plo = phi + Cfg::P_TILE;
            float lsum[2] = {0.f, 0.f};
#pragma unroll
            for (int j = 0; j < NSX; ++j) {
                const int r = r0 + 8 * j;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float p0 = none[k] ? 0.f : ex2(sc[j][k][0] - base[k]);
                    const float p1 = none[k] ? 0.f : ex2(sc[j][k][1] - base[k]);
                    lsum[k] += p0 + p1;
                    const uint32_t hw = float2_to_kv2<KV>(p0, p1);
                    const float2 f = kv2_to_float2<KV>(hw);
                    const uint32_t lw = float2_to_kv2<KV>(p0 - f.x, p1 - f.y);
                    const uint32_t off = tile_unit_offset<TILE, 16>(g + 8 * k, r >> 3) + 4 * t;
                    *reinterpret_cast<uint32_t *>(phi + off) = hw;
                    *reinterpret_cast<uint32_t *>(plo + off) = lw;
                }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float l = lsum[k];
                l += __shfl_xor_sync(0xffffffffu, l, 1);
                l += __shfl_xor_sync(0xffffffffu, l, 2);
                if (t == 0) red_l[warp * 16 + g + 8 * k] = l;
            }
        }
        bool vok = ok;
        if (vok) vok = __all_sync(0xffffffffu, mbar_wait_bounded(bar + 1, 0));
        if (ok && !vok && lane == 0) { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); }
        __syncthreads();                          // P and the sums are in; every V wait is done
        // ---- a5: O = P · V for dimensions d0 .. d0 + DW - 1, hi and lo P into one accumulator ----
        const int d0 = warp * Cfg::DW;
        const bool abort = flags[0] != 0;
        if (!abort) {
            float o[2][NO][4];
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int j = 0; j < NO; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[e][j][i] = 0.f;
            const uint8_t *phi = smem + Cfg::OFF_P, *plo = phi + Cfg::P_TILE;
#pragma unroll
            for (int kk = K0; kk < KO; ++kk) {
                uint32_t ah[4], al[4];
                ldsm_a16<TILE>(ah, phi, kk, lane);
                ldsm_a16<TILE>(al, plo, kk, lane);
                const int vrow = 16 * kk + (i8 & 1) * 8 + (lane & 7);
#pragma unroll
                for (int j = 0; j < NO; j += 2) {
                    uint32_t b[4];
                    ldsm_x4_trans(b, smem + Cfg::OFF_V + tile_unit_offset<HD, TILE>(vrow, (d0 >> 3) + j + (i8 >> 1)));
                    mma_16816<KV>(o[kk & 1][j], ah, b[0], b[1]);
                    mma_16816<KV>(o[kk & 1][j], al, b[0], b[1]);
                    mma_16816<KV>(o[kk & 1][j + 1], ah, b[2], b[3]);
                    mma_16816<KV>(o[kk & 1][j + 1], al, b[2], b[3]);
                }
            }
            // ---- a6: oc of both slots for these dimensions; (mx, S) per slot ----
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int hp = QS::slot_head(a, hk, qg, g + 8 * k);
                if (hp < 0) continue;
                float *dst = a.ws_o + (((size_t)s * heads + hp) * P + sp) * HD + d0 + 2 * t;
#pragma unroll
                for (int j = 0; j < NO; ++j)
                    *reinterpret_cast<float2 *>(dst + 8 * j) =
                        make_float2(o[0][j][2 * k] + o[1][j][2 * k], o[0][j][2 * k + 1] + o[1][j][2 * k + 1]);
            }
            if (warp == 0 && t == 0) {
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int hp = QS::slot_head(a, hk, qg, g + 8 * k);
                    if (hp < 0) continue;
                    float L = 0.f;
#pragma unroll
                    for (int w = 0; w < Cfg::NW; ++w) L += red_l[w * 16 + g + 8 * k];
                    a.ws_ml[((size_t)s * heads + hp) * P + sp] =
                        make_float2(none[k] ? -INFINITY : base[k], none[k] ? 0.f : L);
                }
            }
        } else if (tid == 0) {
            (void)mbar_wait_bounded(bar + 0, 0);
            (void)mbar_wait_bounded(bar + 1, 0);
        }
    };
    if constexpr (Cfg::IS_WIDE) {
        if (n <= TILE / 2) rows_from(std::integral_constant<int, NS / 2>{}, std::integral_constant<int, KO / 2>{});
        else rows_from(std::integral_constant<int, NS>{}, std::integral_constant<int, 0>{});
    } else {
        rows_from(std::integral_constant<int, NS>{}, std::integral_constant<int, 0>{});
    }
}

} // namespace attn
