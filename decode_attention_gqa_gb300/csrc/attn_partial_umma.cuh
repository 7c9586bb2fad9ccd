// attn_partial_umma.cuh -- the split partial kernel on the fifth-generation
// tensor cores (tcgen05, accumulators in tensor memory): steps a1-a6 for a
// split of at most one tile (128 rows; 96 at head_dim 256), one query row or
// several causal ones, head_dim 128 or 256.
//
// One block per (split sp, KV head hk, sequence s), the static grid of minfer
// "10 · R4" §2.2 with the KV head in place of the query head (Red Lite dev35
// "Change": the whole query-head group from one K/V read). The split is a
// single tile of rows, so the block sees each of its rows once and its softmax
// is one pass over the tile with a block-wide maximum (§2.1 with one step):
//   1. TMA brings the 128 cache rows that end at hi, K and V (128-byte
//      swizzled, as in attn_partial.cuh). The rows of the split are the tile's
//      last n = hi - lo rows; rows in front of the sequence's first row arrive
//      as zeros, all others are earlier rows of the same sequence (finite).
//   2. One thread issues S = K · Qᵀ into tensor memory: M = 128 tile rows,
//      N = 16, K = head_dim. Q's 16 rows are the G query heads' hi parts
//      (rows 0-7) and lo parts (rows 8-15) of the scaled q, as in
//      attn_warp_tc.cuh, so column g plus column 8 + g is head g's score.
//   3. Four warps, one per 32-lane quadrant of tensor memory (one tile row per
//      thread), take each head's maximum over the block, p = 2^(s - m + OFF)
//      (0 outside the split), and store p as a hi/lo pair of 16-bit values:
//      P[row][g] = hi, P[row][8 + g] = lo.
//   4. The same thread issues Oᵀ = Vᵀ · P: M = 128 dimensions per MMA (two
//      halves at head_dim 256), N = 16, K = 128 rows, into tensor-memory
//      accumulators of their own.
//   5. The four warps read Oᵀ back, one dimension per thread, and write the
//      partial triple (mx, S, oc) of every head (§3.2); column g plus column
//      8 + g is head g's accumulator.
// Operand layouts (tcgen05 shared-memory descriptors): K and Q are K-major
// with the 128-byte swizzle (8-row groups 1024 bytes apart); Vᵀ is read from
// the same V tile as an MN-major operand (the two 64-dimension halves
// TILE * 128 bytes apart); P is MN-major without swizzle, in 8 x 8 core
// matrices (16-row blocks of K 512 bytes apart).
#pragma once

#include "attn_device.cuh"
#include "attn_warp_tc.cuh"
#include "attn_warp_tcmq.cuh"

namespace attn {

// ---------------------------------------------------------------------------
// tcgen05 and TMA helpers (inline PTX, sm_100a family).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(slot)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: start address, leading- and stride-dimension
// byte offsets, layout (0: no swizzle, 2: 128-byte swizzle); bit 46 is the
// descriptor version.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)layout << 61;
    return d;
}

// Instruction descriptor of a kind::f16 MMA with f32 accumulation: A and B
// both binary16 or both bfloat16, each K-major (0) or MN-major (1).
template <typename KV>
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N, int a_mn, int b_mn)
{
    constexpr uint32_t fmt = std::is_same<KV, __half>::value ? 0u : 1u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (tensor memory) = A · B, or D += A · B when acc != 0; issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

// One arrival on bar once every MMA this thread has issued is complete.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

// 16 consecutive 32-bit columns of the warp's lane quadrant: thread i gets lane
// (quadrant base + i). Waits for the load before returning.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
                   "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of P[row][n] (n < NCOL) in the MN-major, unswizzled B operand:
// 8 x 8 core matrices of 128 bytes; 8-column groups 128 bytes apart, 8-row
// groups NCOL * 16 bytes apart.
template <int NCOL>
__device__ __forceinline__ uint32_t p_offset(int row, int n)
{
    return (uint32_t)((row >> 3) * (NCOL * 16) + (n >> 3) * 128 + (row & 7) * 16 + (n & 7) * 2);
}

// MQ = false: one query row, the G heads of the group in slots 0..G-1 (q as in
// attn_warp_tc.cuh: one 16-row Q tile, hi parts in rows 0-7, lo in 8-15).
// MQ = true: several causal query rows, 16 (query row, head) slots per block
// (q as in attn_warp_tcmq.cuh: a 16-row hi tile and a 16-row lo tile).
// Either way slot i's score is column i plus column NQH + i of S, and P and Oᵀ
// use the same columns.
template <int HD, int G, typename KV, bool MQ = false>
struct UmmaCfg {
    static_assert(HD == 128 || HD == 256, "the tcgen05 partial kernel is built for head_dim 128 and 256");
    // rows per block: 128 (one MMA M extent); 96 at head_dim 256, so that two
    // blocks fit an SM -- S is still an M = 128 MMA, whose last 32 rows read
    // past the K tile (finite data) and are masked
    static constexpr int TILE = HD == 256 ? 96 : 128;
    static constexpr int MMA_M = 128;
    static constexpr int THREADS = 192;               // TMA/MMA warp, TMEM warp, 4 softmax warps
    static constexpr int NCH = HD / 64;               // 128-byte column chunks per row
    static constexpr int NMO = HD / 128;              // 128-dimension halves of Oᵀ (one MMA M each)
    static constexpr int GRANULE = TILE;              // count-mode chunks are whole tiles
    static constexpr int NQH = MQ ? 16 : 8;           // query-head slots (columns per hi or lo half)
    static constexpr int NSLOT = MQ ? 16 : G;         // slots a block may fill
    static constexpr int NCOL = 2 * NQH;              // MMA N of S, P and Oᵀ
    static constexpr int NQT = MQ ? 2 : 1;            // 16-row Q tiles (B operands of S)
    using QStage = typename std::conditional<MQ, TcWarpMQ<HD, 16, 4, KV>, TcWarp<HD, G, 4, KV>>::type;
    static constexpr uint32_t QT_BYTES = 16u * HD * 2;
    static constexpr uint32_t OFF_INV = NQT * QT_BYTES;           // per-slot scales in the q area
    static constexpr uint32_t TILE_BYTES = (uint32_t)TILE * HD * 2;
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = TILE_BYTES;
    static constexpr uint32_t OFF_Q = 2 * TILE_BYTES;
    static constexpr uint32_t OFF_P = (OFF_Q + QStage::EXTRA_BYTES + 127) / 128 * 128;
    static constexpr uint32_t P_BYTES = (uint32_t)MMA_M * NCOL * 2;
    static constexpr uint32_t OFF_RED = OFF_P + P_BYTES;          // [2][4][NQH] floats: maxima, sums
    static constexpr uint32_t OFF_BAR = OFF_RED + 2 * 4 * NQH * 4; // 4 mbarriers, TMEM slot, flags
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 4 * 8 + 16 + 1024;   // + base alignment slack
    // S in columns 0 .. NCOL-1, Oᵀ half h in NCOL (1 + h) .. ; a power of two >= 32
    static constexpr uint32_t TMEM_NEED = (uint32_t)NCOL * (1 + NMO);
    static constexpr uint32_t TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : 128;
    static constexpr float OFF = 7.f;                 // p headroom: p <= 2^OFF
    static_assert(QStage::QT_BYTES == QT_BYTES, "Q tile layout of the staging policy");
    static_assert(OFF_Q % 1024 == 0 && OFF_V % 1024 == 0 && QT_BYTES % 1024 == 0,
                  "swizzled operands start 1024-aligned");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(TILE % 16 == 0 && TILE <= MMA_M && (TILE * 128) % 1024 == 0, "tile rows");
};

template <class Cfg, int HD, int G, typename KV>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
attn_split_partial_umma(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const PartialArgs a)
{
    constexpr int TILE = Cfg::TILE, NQH = Cfg::NQH, NSLOT = Cfg::NSLOT, NCOL = Cfg::NCOL;
    constexpr bool MQ = Cfg::NQT == 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);   // full, s_done, p_ready, o_done
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 4);
    volatile int *flags = reinterpret_cast<volatile int *>(tslot + 1);   // [0] abort
    float *red = reinterpret_cast<float *>(smem + Cfg::OFF_RED);

    // grid (KV head x query group, split, sequence): KV heads vary fastest
    const int hk = blockIdx.x / a.qgroups, qg = blockIdx.x % a.qgroups, sp = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = a.n_splits;
    const size_t heads = (size_t)a.n_q * a.n_head;       // partial heads per sequence

    // Dependencies as in attn_partial.cuh: with kv_stable the positions read
    // and the tile copy go ahead of the grid dependency, q waits for it.
    const bool stable = a.kv_stable != 0;
    if (tid == 0) {
        // q of this block's slots into L2 (query rows t0..t1 of the group's heads)
        const int gq = MQ ? a.group : G;
        const int t0 = MQ ? qg * NQH / gq : 0;
        const int t1 = MQ ? min(a.n_q - 1, (qg * NQH + NQH - 1) / gq) : 0;
        for (int t = t0; t <= t1; ++t)
            prefetch_l2(a.q + (((size_t)s * a.n_q + t) * a.n_head + (size_t)hk * gq) * HD,
                        (uint32_t)(gq * HD * sizeof(float)));
    }
    if (!stable) pdl_wait();
    pdl_launch_dependents();

    // a1: rows attended and this split's rows; an empty split leaves at once
    bool pos_ok;
    const int64_t nkv = rows_attended(a, s, sp == 0 && blockIdx.x == 0 && tid == 0, &pos_ok);
    int64_t lo, hi;
    split_range(nkv, sp, P, a.split_len, Cfg::GRANULE, lo, hi);
    if (lo >= hi) {
        if (stable) pdl_wait();               // the workspace may still be read by the previous grid
        if (tid < NSLOT) {
            const int hp = Cfg::QStage::slot_head(a, hk, qg, tid);
            if (hp >= 0) a.ws_ml[((size_t)s * heads + hp) * P + sp] = make_float2(-INFINITY, 0.f);
        }
        return;
    }
    const int n = (int)(hi - lo);             // 1..TILE rows: the tile's last n rows
    const int row_first = (int)(hi - TILE);   // negative near the sequence start: zero rows

    if (tid == 0) {
        mbar_init(bar + 0, 1);                // K and V landed
        mbar_init(bar + 1, 1);                // S complete
        mbar_init(bar + 2, 128);              // P written (one arrival per softmax thread)
        mbar_init(bar + 3, 1);                // Oᵀ complete
        flags[0] = 0;
        fence_barrier_init();
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        mbar_arrive_expect_tx(bar + 0, 2 * Cfg::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < Cfg::NCH; ++c) {
            tma_load_4d(smem + Cfg::OFF_K + c * (Cfg::TILE_BYTES / Cfg::NCH), &kmap, bar + 0, c * 64, hk, row_first, s);
            tma_load_4d(smem + Cfg::OFF_V + c * (Cfg::TILE_BYTES / Cfg::NCH), &vmap, bar + 0, c * 64, hk, row_first, s);
        }
    }
    if (warp == 1) tmem_alloc(tslot, Cfg::TMEM_COLS);

    // a2, while the tile is in flight: the Q tile and per-head scales
    if (stable) pdl_wait();
    Cfg::QStage::template prepare<Cfg::THREADS>(smem + Cfg::OFF_Q, a, s, hk, qg, tid);
    // Fused append: the split ending at nkv holds the new row nkv - 1 as the
    // tile's last row. Warp 0 fetches it now (one 16-byte unit per lane) and
    // writes it into the tile and the cache once the copy has landed.
    constexpr int NU = HD / 8;                    // 16-byte units per row
    constexpr int NJ = 2 * NU / 32;               // units of the new K and V rows per lane
    static_assert(2 * NU % 32 == 0, "whole units per lane");
    const bool appending = a.k_new != nullptr && pos_ok && hi == nkv && warp == 0;
    uint4 newrow[NJ];
    if (appending) {
        const size_t src = ((size_t)s * a.n_kv_head + hk) * HD;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int i = lane + 32 * j;
            newrow[j] = ld_dep(reinterpret_cast<const uint4 *>((i < NU ? a.k_new : a.v_new) + src) + (i % NU));
        }
    }
    fence_proxy_async_smem();                 // the Q tile is read by the tensor cores
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tslot;
    const uint32_t tm_s = tm, tm_o = tm + NCOL;

    if (warp == 0) {
        // ---------------- TMA / MMA warp ----------------
        const bool landed = mbar_wait_bounded(bar + 0, 0);
        if (!__all_sync(0xffffffffu, landed)) {
            if (lane == 0) { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); }
        } else {
            if (appending) {
                const size_t dst = ((size_t)((int64_t)s * a.cap + nkv - 1) * a.n_kv_head + hk) * HD;
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int i = lane + 32 * j;
                    uint8_t *tile = smem + (i < NU ? Cfg::OFF_K : Cfg::OFF_V);
                    *reinterpret_cast<uint4 *>(tile + tile_unit_offset<HD, TILE>(TILE - 1, i % NU)) = newrow[j];
                    reinterpret_cast<uint4 *>((i < NU ? a.k_w : a.v_w) + dst)[i % NU] = newrow[j];
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                tc_fence_after();
                const uint32_t sk = smem_u32(smem + Cfg::OFF_K), sq = smem_u32(smem + Cfg::OFF_Q);
                constexpr uint32_t id_s = umma_idesc<KV>(Cfg::MMA_M, 16, 0, 0);
                // Q tile qt (one, or hi and lo) into columns 16qt .. 16qt + 15; k-step kk
                // covers dims [16kk, 16kk + 16): chunk kk / 4, 32 bytes per step within it
#pragma unroll
                for (int qt = 0; qt < Cfg::NQT; ++qt)
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t ok = (kk >> 2) * (TILE * 128) + (kk & 3) * 32;
                        const uint32_t oq = qt * Cfg::QT_BYTES + (kk >> 2) * (16 * 128) + (kk & 3) * 32;
                        umma_f16(tm_s + 16 * qt, umma_desc(sk + ok, 16, 1024, 2), umma_desc(sq + oq, 16, 1024, 2),
                                 id_s, kk > 0);
                    }
                umma_commit(bar + 1);
            }
            __syncwarp();
            const bool pw = mbar_wait_bounded(bar + 2, 0);
            if (!__all_sync(0xffffffffu, pw)) {
                if (lane == 0) { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); }
            } else if (lane == 0) {
                tc_fence_after();
                const uint32_t sv = smem_u32(smem + Cfg::OFF_V), spp = smem_u32(smem + Cfg::OFF_P);
                constexpr uint32_t id_o = umma_idesc<KV>(128, NCOL, 1, 1);
                // half h covers dimensions [128h, 128h + 128): column chunks 2h and 2h + 1;
                // k-step kk covers tile rows [16kk, 16kk + 16): two 8-row groups of V
                // (2048 bytes) and of P (2 * NCOL * 16 bytes)
#pragma unroll
                for (int h = 0; h < Cfg::NMO; ++h)
#pragma unroll
                    for (int kk = 0; kk < TILE / 16; ++kk)
                        umma_f16(tm_o + NCOL * h, umma_desc(sv + h * 2 * (TILE * 128) + kk * 2048, TILE * 128, 1024, 2),
                                 umma_desc(spp + kk * (2 * NCOL * 16), NCOL * 16, 128, 0), id_o, kk > 0);
                umma_commit(bar + 3);
            }
        }
    } else if (warp >= 2) {
        // ---------------- softmax / epilogue warps ----------------
        const int q4 = warp & 3;                       // tensor-memory lane quadrant
        const int r = q4 * 32 + lane;                  // tile row (S) and dimension (Oᵀ)
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const float *inv = reinterpret_cast<const float *>(smem + Cfg::OFF_Q + Cfg::OFF_INV);
        const int *qrow = reinterpret_cast<const int *>(inv + 16);   // several rows: slot -> query row
        // Both named barriers below are passed by all four warps whatever
        // happened before them; a warp whose wait gave up sets the abort flag
        // and the block writes no partial.
        const bool sd = mbar_wait_bounded(bar + 1, 0);
        bool ok = __all_sync(0xffffffffu, sd);
        if (!ok && lane == 0) { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); }
        float sc[NSLOT];
        if (ok) {
            tc_fence_after();
            float c[NCOL];
#pragma unroll
            for (int j = 0; j < NCOL / 16; ++j) {
                float cj[16];
                tmem_ld16(tm_s + 16 * j + lane_base, cj);
#pragma unroll
                for (int i = 0; i < 16; ++i) c[16 * j + i] = cj[i];
            }
            const bool in_split = r >= TILE - n && r < TILE;
            // several query rows: slot i (query row t) sees cache rows [0, nkv - n_q + t]
            const int64_t row = hi - TILE + r;
#pragma unroll
            for (int i = 0; i < NSLOT; ++i) {
                bool valid = in_split;
                if constexpr (MQ) valid = valid && qrow[i] >= 0 && row <= nkv - a.n_q + qrow[i];
                sc[i] = valid ? (c[i] + c[NQH + i]) * inv[i] : -INFINITY;
            }
            // a4: each slot's maximum over the block
#pragma unroll
            for (int i = 0; i < NSLOT; ++i) {
                const float m = warp_max(sc[i]);
                if (lane == 0) red[q4 * NQH + i] = m;
            }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        ok = ok && !flags[0];
        float p[NQH];
        if (ok) {
#pragma unroll
            for (int i = 0; i < NQH; ++i) {
                if (i < NSLOT) {
                    const float M = fmaxf(fmaxf(red[i], red[NQH + i]), fmaxf(red[2 * NQH + i], red[3 * NQH + i]));
                    // 0 outside the split; a slot that sees no row here (several query rows) has M = -inf
                    p[i] = M == -INFINITY ? 0.f : ex2(sc[i] - (M - Cfg::OFF));
                } else {
                    p[i] = 0.f;
                }
            }
            // P row r: hi parts in columns 0 .. NQH-1, lo parts in NQH .. NCOL-1
            uint32_t hw[NQH / 2], lw[NQH / 2];
#pragma unroll
            for (int j = 0; j < NQH / 2; ++j) {
                hw[j] = float2_to_kv2<KV>(p[2 * j], p[2 * j + 1]);
                const float2 f = kv2_to_float2<KV>(hw[j]);
                lw[j] = float2_to_kv2<KV>(p[2 * j] - f.x, p[2 * j + 1] - f.y);
            }
#pragma unroll
            for (int u = 0; u < NQH / 8; ++u) {
                *reinterpret_cast<uint4 *>(smem + Cfg::OFF_P + p_offset<NCOL>(r, 8 * u)) =
                    make_uint4(hw[4 * u], hw[4 * u + 1], hw[4 * u + 2], hw[4 * u + 3]);
                *reinterpret_cast<uint4 *>(smem + Cfg::OFF_P + p_offset<NCOL>(r, NQH + 8 * u)) =
                    make_uint4(lw[4 * u], lw[4 * u + 1], lw[4 * u + 2], lw[4 * u + 3]);
            }
            fence_proxy_async_smem();
        }
        mbar_arrive(bar + 2);
        if (ok) {
            // S of each slot over the block, while the p·V MMAs run
#pragma unroll
            for (int i = 0; i < NSLOT; ++i) {
                const float l = warp_sum(p[i]);
                if (lane == 0) red[4 * NQH + q4 * NQH + i] = l;
            }
            const bool od = mbar_wait_bounded(bar + 3, 0);
            ok = __all_sync(0xffffffffu, od);
            if (!ok && lane == 0) { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); }
        }
        if (ok) {
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < Cfg::NMO; ++h) {
                float c[NCOL];
#pragma unroll
                for (int j = 0; j < NCOL / 16; ++j) {
                    float cj[16];
                    tmem_ld16(tm_o + NCOL * h + 16 * j + lane_base, cj);
#pragma unroll
                    for (int i = 0; i < 16; ++i) c[16 * j + i] = cj[i];
                }
#pragma unroll
                for (int i = 0; i < NSLOT; ++i) {
                    const int hp = Cfg::QStage::slot_head(a, hk, qg, i);
                    if (hp >= 0)
                        a.ws_o[(((size_t)s * heads + hp) * P + sp) * HD + 128 * h + r] = c[i] + c[NQH + i];
                }
            }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (warp == 4 && lane < NSLOT && !flags[0]) {
            const int i = lane;
            const int hp = Cfg::QStage::slot_head(a, hk, qg, i);
            const float M = fmaxf(fmaxf(red[i], red[NQH + i]), fmaxf(red[2 * NQH + i], red[3 * NQH + i]));
            const float L = (red[4 * NQH + i] + red[5 * NQH + i]) + (red[6 * NQH + i] + red[7 * NQH + i]);
            if (hp >= 0)
                a.ws_ml[((size_t)s * heads + hp) * P + sp] = make_float2(M == -INFINITY ? M : M - Cfg::OFF, L);
        }
    }

    // Nothing may still be writing shared or tensor memory when the block
    // exits: after an abort, wait (bounded) for the copy and the MMAs.
    tc_fence_before();
    __syncthreads();
    if (flags[0]) {                           // read after the barrier: the same for every thread
        if (tid == 0) {
            (void)mbar_wait_bounded(bar + 0, 0);
            (void)mbar_wait_bounded(bar + 3, 0, 1000000ull);
        }
        __syncthreads();
    }
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tm, Cfg::TMEM_COLS);
}

} // namespace attn
