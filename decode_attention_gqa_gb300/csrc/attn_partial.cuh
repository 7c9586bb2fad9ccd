// attn_partial.cuh -- the split partial kernel (steps a1-a6).
//
// One block per (split sp, KV head hk, sequence s): the static grid of minfer
// "10 · R4" §2.2 with the KV head in place of the query head, so that the
// whole query-head group is served from one K/V read (Red Lite dev35
// "Change"). nkv is read from positions[s] on the device (§2.2).
//
// Block = NWC compute warps + 1 producer warp. The producer streams the
// split's rows through an S-stage ring of shared-memory tiles of TILE rows of
// K and of V (128-byte swizzled), with one mbarrier pair per stage:
//   - a whole tile comes by TMA (cp.async.bulk.tensor);
//   - the split's last tile, when shorter, is loaded as the TILE rows that end
//     at hi (TMA again; the rows in front of the tile's own first row are
//     earlier cache rows, finite data that the compute warps skip), so no
//     cache row at or past nkv is read; when hi < TILE it is copied with
//     cp.async instead, zero-filled in front. In both cases the rows in range
//     are the tile's last nrows rows.
// Compute warp w owns rows [w*WR, (w+1)*WR) of every tile and keeps its own
// online-softmax state (mx, S, oc) for all G heads in registers (§2.1 update,
// §2.4 register accumulator). At the end the NWC states are merged in shared
// memory and the block writes one partial triple per query head (§3.2).
//
// The per-warp arithmetic is a policy class: SimtWarp (attn_warp_simt.cuh,
// CUDA cores, f32), TcWarp (attn_warp_tc.cuh, tensor cores, one query row)
// or TcWarpMQ (attn_warp_tcmq.cuh, tensor cores, several causal query rows).
#pragma once

#include "attn_device.cuh"
#include "attn_warp_simt.cuh"
#include "attn_warp_tc.cuh"
#include "attn_warp_tcmq.cuh"

namespace attn {

template <int HD, int G, template <int, int, int, typename> class W, int NWC_, int S_, int MINB_,
          typename KV>
struct PartialCfg {
    static constexpr int NWC = NWC_;                 // compute warps
    static constexpr int S = S_;                     // pipeline stages
    static constexpr int MIN_BLOCKS = MINB_;         // resident blocks per SM the registers must allow
    using Warp = W<HD, G, NWC, KV>;
    static constexpr int WR = Warp::WR;
    static constexpr int TILE = NWC * WR;            // rows per stage
    static constexpr int GRANULE = Warp::WHOLE_TILE_SPLITS ? TILE : WR;   // count-mode chunk unit
    static constexpr int THREADS = (NWC + 1) * 32;
    static constexpr int NCH = HD >= 64 ? HD / 64 : 1;
    static constexpr int BOX_X = HD >= 64 ? 64 : HD; // TMA box inner extent (elements)
    static constexpr uint32_t TILE_BYTES = (uint32_t)TILE * HD * 2;        // one of K or V
    static constexpr uint32_t STAGE_BYTES = 2 * TILE_BYTES;
    // shared-memory carve-up (byte offsets from a 1024-aligned base)
    static constexpr uint32_t OFF_EXTRA = S * STAGE_BYTES;
    static constexpr uint32_t OFF_BAR = (OFF_EXTRA + Warp::EXTRA_BYTES + 1023) / 1024 * 1024;
    static constexpr uint32_t BAR_BYTES = 2 * S * 8 + 16;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;   // + base alignment slack
    // merge area (reuses the stage buffers after the main loop)
    static constexpr int NQH = Warp::NQH;            // query heads per block
    static constexpr int MS = merge_stride<HD>();    // floats per published accumulator row
    // merge area (floats): (mx, S) pairs, then the accumulator rows from a
    // 16-byte boundary (the merge reads them as float4)
    static constexpr uint32_t OFF_MO = ((uint32_t)2 * NWC * NQH + 3) / 4 * 4;
    static constexpr uint32_t MERGE_BYTES = (OFF_MO + (uint32_t)NWC * NQH * MS) * 4;
    static_assert(OFF_MO % 4 == 0 && MS % 4 == 0, "float4 rows in the merge area");
    static_assert(MERGE_BYTES <= S * STAGE_BYTES, "merge area must fit in the stage buffers");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(HD < 64 || (TILE_BYTES / NCH) % 1024 == 0, "swizzled chunks must stay 1024-aligned");
    // the shared memory must allow MIN_BLOCKS resident blocks (228 KB per SM,
    // 1 KB reserved per block)
    static_assert(MIN_BLOCKS * (SMEM_BYTES + 1024u) <= 233472u, "MIN_BLOCKS exceeds shared memory");
};

template <class Cfg, int HD, int G>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_BLOCKS)
attn_split_partial(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const PartialArgs a)
{
    using Warp = typename Cfg::Warp;
    constexpr int NWC = Cfg::NWC, S = Cfg::S, TILE = Cfg::TILE, WR = Cfg::WR;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *extra = smem + Cfg::OFF_EXTRA;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *empty = full + S;
    volatile int *flags = reinterpret_cast<volatile int *>(empty + S);   // [0] abort, [1] tiles issued

    // grid (KV head x query group, split, sequence): the KV heads vary
    // fastest, so the low splits of every head -- the ones a short context
    // fills -- are dispatched first
    const int sp = blockIdx.y, s = blockIdx.z;
    const int hk = blockIdx.x / a.qgroups, qg = blockIdx.x % a.qgroups;
    constexpr int NQH = Cfg::NQH;
    const size_t heads = (size_t)a.n_q * a.n_head;          // partial heads per sequence
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = a.n_splits;

    // Inputs may be produced by the previous kernel in the stream: wait for it
    // before the first read of them. The next kernel (the combine) may get
    // resident at once; it waits for this grid in turn. With kv_stable the
    // caller has promised that positions and the attended cache rows are not
    // written by anything still running, so the wait moves to just before q
    // is read, after the first K/V copies are in flight.
    const bool stable = a.kv_stable != 0;
    if (tid == NWC * 32) {
        // q of this block's query heads into L2 while the previous grid runs
        // (query rows t0..t1 hold the block's (row, group head) pairs)
        const uint32_t gbytes = (uint32_t)(G * HD * sizeof(float));
        const int t0 = qg * NQH / G, t1 = min(a.n_q - 1, (qg * NQH + NQH - 1) / G);
        for (int t = t0; t <= t1; ++t)
            prefetch_l2(a.q + (((size_t)s * a.n_q + t) * a.n_head + (size_t)hk * G) * HD, gbytes);
    }
    if (!stable) pdl_wait();
    pdl_launch_dependents();

    // a1: rows attended and this split's range; an empty split leaves at once
    bool pos_ok;
    const int64_t nkv = rows_attended(a, s, sp == 0 && blockIdx.x == 0 && tid == 0, &pos_ok);
    int64_t lo, hi;
    split_range(nkv, sp, P, a.split_len, Cfg::GRANULE, lo, hi);
    if (lo >= hi) {                                                      // empty split: mx=-inf, S=0
        if (stable) pdl_wait();               // the workspace may still be read by the previous grid
        if (tid < NQH) {
            const int hp = Warp::slot_head(a, hk, qg, tid);
            if (hp >= 0) a.ws_ml[((size_t)s * heads + hp) * P + sp] = make_float2(-INFINITY, 0.f);
        }
        return;
    }
    const int ntiles = (int)((hi - lo + TILE - 1) / TILE);
    const int64_t seq_row0 = (int64_t)s * a.cap;                          // flat row of (s, 0)

    // Tile t by TMA: rows [first, first + TILE), or the TILE rows ending at hi
    // for a short last tile (needs hi >= TILE, else it goes by cp.async).
    auto tma_tile = [&](int t, int st) {
        const int64_t first = lo + (int64_t)t * TILE;
        const int z = (int)(seq_row0 + (hi - first >= TILE ? first : hi - TILE));
        uint8_t *kst = smem + st * Cfg::STAGE_BYTES;
        uint8_t *vst = kst + Cfg::TILE_BYTES;
        mbar_arrive_expect_tx(full + st, Cfg::STAGE_BYTES);
#pragma unroll
        for (int c = 0; c < Cfg::NCH; ++c) {
            tma_load_3d(kst + c * (Cfg::TILE_BYTES / Cfg::NCH), &kmap, full + st, c * Cfg::BOX_X, hk, z);
            tma_load_3d(vst + c * (Cfg::TILE_BYTES / Cfg::NCH), &vmap, full + st, c * Cfg::BOX_X, hk, z);
        }
    };
    const bool tail_by_tma = hi >= TILE;
    // The same rows into L2 only, for a tile that has no free stage yet.
    auto tma_prefetch_tile = [&](int t) {
        const int64_t first = lo + (int64_t)t * TILE;
        const int z = (int)(seq_row0 + (hi - first >= TILE ? first : hi - TILE));
#pragma unroll
        for (int c = 0; c < Cfg::NCH; ++c) {
            tma_prefetch_3d(&kmap, c * Cfg::BOX_X, hk, z);
            tma_prefetch_3d(&vmap, c * Cfg::BOX_X, hk, z);
        }
    };

    int early = 0;                          // tiles the producer issues before the block syncs
    if (tid == NWC * 32) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, NWC);
        }
        flags[0] = 0;
        fence_barrier_init();
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        for (; early < S && early < ntiles; ++early) {
            const bool whole = hi - (lo + (int64_t)early * TILE) >= TILE;
            if (!whole && !tail_by_tma) break;
            tma_tile(early, early);
        }
        flags[1] = early;
        // the next S tiles into L2, so that a stage freed later refills from L2
        for (int t = early; t < ntiles && t < early + S; ++t) {
            if (hi - (lo + (int64_t)t * TILE) < TILE && !tail_by_tma) break;
            tma_prefetch_tile(t);
        }
    }
    // a2, while the first tiles are in flight
    if (stable) pdl_wait();
    Warp::template prepare<Cfg::THREADS>(extra, a, s, hk, qg, tid);
    __syncthreads();
    early = flags[1];

    if (warp == NWC) {
        // ---------------- producer warp ----------------
        for (int t = early; t < ntiles; ++t) {
            const int st = t % S;
            int ok = 1;
            if (lane == 0) {
                if (t >= S && !mbar_wait_bounded(empty + st, ((t / S) - 1) & 1)) {
                    flags[0] = 1;
                    atomicOr(a.err, kErrPipelineTimeout);
                }
                ok = !flags[0];
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            const int64_t first = lo + (int64_t)t * TILE;
            const int nrows = (int)(hi - first < TILE ? hi - first : TILE);
            if (nrows == TILE || tail_by_tma) {
                if (lane == 0) tma_tile(t, st);
            } else {
                // hi < TILE: rows [first, hi) to tile rows [vs0, TILE), vs0 = TILE - nrows.
                // V rows of the slice holding vs0 that lie before it are zeroed
                // (their p is 0 and must not meet stale non-finite data); slices
                // wholly before vs0 are skipped by the compute warps.
                constexpr int NU = HD / 8;
                uint8_t *kst = smem + st * Cfg::STAGE_BYTES;
                uint8_t *vst = kst + Cfg::TILE_BYTES;
                const int vs0 = TILE - nrows;
                const int zs = vs0 / WR * WR;
                const size_t rstride = (size_t)a.n_kv_head * HD;               // elements per row
                const uint16_t *kg = a.k + (size_t)(seq_row0 + first) * rstride + (size_t)hk * HD;
                const uint16_t *vg = a.v + (size_t)(seq_row0 + first) * rstride + (size_t)hk * HD;
                for (int i = lane; i < (TILE - zs) * NU; i += 32) {
                    const int r = zs + i / NU, U = i % NU;
                    const uint32_t so = tile_unit_offset<HD, TILE>(r, U);
                    if (r >= vs0) {
                        const size_t off = (size_t)(r - vs0) * rstride + (size_t)U * 8;
                        cp_async16(kst + so, kg + off, 16u);
                        cp_async16(vst + so, vg + off, 16u);
                    } else {
                        *reinterpret_cast<uint4 *>(vst + so) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                cp_async_mbar_arrive(full + st);
                __syncwarp();
                if (lane == 0) mbar_arrive(full + st);
            }
            if (lane == 0) flags[1] = t + 1;
        }
    } else {
        // ---------------- compute warps ----------------
        Warp wst;
        wst.init(extra, warp, lane);
        // Fused append: the split ending at nkv holds the new row nkv - 1, and in
        // its last tile that row is always shared-memory row TILE - 1, owned by
        // the last compute warp. That warp puts the new K/V row into the tile
        // (over whatever the cache held there) and into the cache itself; no
        // other block reads this row.
        constexpr int NU = HD / 8;
        constexpr int NJ = (2 * NU + 31) / 32;
        const bool appending = a.k_new != nullptr && pos_ok && hi == nkv && warp == NWC - 1;
        uint4 newrow[NJ];
        if (appending) {
            const size_t src = ((size_t)s * a.n_kv_head + hk) * HD;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int i = lane + 32 * j;
                if (i < 2 * NU)
                    newrow[j] = ld_dep(reinterpret_cast<const uint4 *>((i < NU ? a.k_new : a.v_new) + src) +
                                      (i < NU ? i : i - NU));
            }
        }
        for (int t = 0; t < ntiles; ++t) {
            const int st = t % S;
            const bool landed = mbar_wait_bounded(full + st, (t / S) & 1);
            if (!__all_sync(0xffffffffu, landed)) {
                if (lane == 0) { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); }
                break;
            }
            if (__shfl_sync(0xffffffffu, flags[0], 0)) break;
            const uint8_t *kst = smem + st * Cfg::STAGE_BYTES;
            const uint8_t *vst = kst + Cfg::TILE_BYTES;
            const int64_t first = lo + (int64_t)t * TILE;
            const int nrows = (int)(hi - first < TILE ? hi - first : TILE);
            const int ra = TILE - nrows - warp * WR;      // first in-range row of the slice
            if (appending && t == ntiles - 1) {
                const size_t dst = ((size_t)(seq_row0 + nkv - 1) * a.n_kv_head + hk) * HD;
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int i = lane + 32 * j;
                    if (i < 2 * NU) {
                        const int U = i < NU ? i : i - NU;
                        uint8_t *tile = const_cast<uint8_t *>(i < NU ? kst : vst);
                        *reinterpret_cast<uint4 *>(tile + tile_unit_offset<HD, TILE>(TILE - 1, U)) = newrow[j];
                        reinterpret_cast<uint4 *>((i < NU ? a.k_w : a.v_w) + dst)[U] = newrow[j];
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            const int64_t row0 = nrows == TILE ? first : hi - TILE;   // sequence row of tile row 0
            if (ra < WR)
                wst.template process<TILE>(kst, vst, warp * WR, ra > 0 ? ra : 0, row0, nkv, a, extra,
                                           warp, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + st);
        }
        // the merge area overlaps the stage buffers: every compute warp must be
        // done with the ring before any of them publishes its state
        asm volatile("bar.sync 1, %0;" :: "r"(NWC * 32) : "memory");
        if (!__shfl_sync(0xffffffffu, flags[0], 0))
            wst.publish(reinterpret_cast<float2 *>(smem) + warp * NQH,
                        reinterpret_cast<float *>(smem) + Cfg::OFF_MO + warp * NQH * Cfg::MS, lane);
    }
    __syncthreads();

    // Drain: no copy may still be writing shared memory when the block exits.
    // Without an abort the compute warps have waited for every issued tile.
    if (tid == NWC * 32 && flags[0]) {
        const int issued = flags[1];
        for (int t = issued - S > 0 ? issued - S : 0; t < issued; ++t)
            (void)mbar_wait_bounded(full + (t % S), (t / S) & 1);
    }
    if (flags[0]) return;        // partial left unwritten; the error word says why

    // a6: merge the NWC warp states and write the partial triple of each head
    // (a query head no warp saw a row for -- possible with causal limits --
    // keeps mx = -inf and S = 0). Each thread takes the maximum and the NWC
    // weights of its own head from the published (mx, S) pairs, then scales
    // and adds the accumulators in float4 units; the thread holding a head's
    // first unit also writes its (mx, S).
    const float2 *mm = reinterpret_cast<const float2 *>(smem);
    const float *mo = reinterpret_cast<const float *>(smem) + Cfg::OFF_MO;
    constexpr int D4 = HD / 4;
    for (int i = tid; i < NQH * D4; i += Cfg::THREADS) {
        const int g = i / D4, d = (i % D4) * 4;
        const int hp = Warp::slot_head(a, hk, qg, g);
        if (hp < 0) continue;
        float2 ml[NWC];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NWC; ++w) {
            ml[w] = mm[w * NQH + g];
            M = fmaxf(M, ml[w].x);
        }
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < NWC; ++w) {
            const float wt = ml[w].x == -INFINITY ? 0.f : ex2(ml[w].x - M);
            const float4 v = *reinterpret_cast<const float4 *>(mo + (w * NQH + g) * Cfg::MS + d);
            O.x = fmaf(wt, v.x, O.x);
            O.y = fmaf(wt, v.y, O.y);
            O.z = fmaf(wt, v.z, O.z);
            O.w = fmaf(wt, v.w, O.w);
            L = fmaf(wt, ml[w].y, L);
        }
        const size_t slot = ((size_t)s * heads + hp) * P + sp;
        *reinterpret_cast<float4 *>(a.ws_o + slot * HD + d) = O;
        if (d == 0) a.ws_ml[slot] = make_float2(M, L);
    }
}

} // namespace attn
