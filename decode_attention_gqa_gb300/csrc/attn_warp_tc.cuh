// attn_warp_tc.cuh -- tensor-core per-warp arithmetic of the partial kernel:
// steps a3-a5 for one warp's 16-row slice of a shared-memory tile, with
// 16x8x16 f16 MMAs accumulating in f32.
//
// The dotLLM #199 design (§2) pads the single query row to a 16-row MMA tile
// and wastes 15 rows. Here the 16 rows carry the whole query-head group twice:
// rows 0..7 hold hi = T(x) and rows 8..15 hold lo = T(x - hi) for the G <= 8
// heads, T the cache's element type, so q·k = hi·k + lo·k keeps about 22
// significant bits of q for f16 (16 for bf16; the products are exact in the
// f32 accumulator) instead of the 11 (8) bits of a plain cast (the precision
// risk of "Option B", #199 §0). The softmax weights p
// get the same hi/lo treatment for p·V, and the C fragment of q·Kᵀ is exactly
// the A fragment layout of p·V, so no data moves between lanes.
//
//   scores  C[16 x 8 rows]  = Q[16 x hd] · K[8 rows x hd]ᵀ     (two n-tiles per slice)
//   values  O[16 x hd]     += P[16 x 16 rows] · V[16 rows x hd]
//
// Lane l owns head g = l / 4 and rows {2t, 2t+1, 8+2t, 9+2t} (t = l % 4) of the
// slice's scores, and dims {8n + 2t, 8n + 2t + 1} of head g's accumulator.
//
// q is scaled per head by a power of two (exact) so its largest element lies in
// [2^14, 2^15): no f16 overflow for any finite q and the lo part stays normal.
// Rescaling of the accumulator is lazy: the reference max only moves when a new
// score exceeds it by more than TAU (log2 units), so p <= 2^(TAU + OFF) and the
// final o = acc / S is unchanged (both use the same reference).
#pragma once

#include "attn_device.cuh"

namespace attn {

template <int HD, int G, int NWC, typename KV>
struct TcWarp {
    static_assert(HD % 16 == 0, "tensor-core path needs head_dim % 16 == 0");
    static constexpr int WR = 16;                     // rows per warp slice
    // count-mode splits are whole tiles (head_dim <= 128): a block's rows then
    // fill its stage ring exactly and no split re-reads a neighbour's rows
    static constexpr bool WHOLE_TILE_SPLITS = HD <= 128;
    static constexpr int NQH = G;                     // query heads per block (one query row)

    // Partial-head index of block-local query head i (single query row: the
    // group's heads hk*G .. hk*G+G-1).
    static __device__ __forceinline__ int slot_head(const PartialArgs &a, int hk, int, int i)
    {
        (void)a;
        return hk * G + i;
    }
    static constexpr int KSTEPS = HD / 16;            // k-steps of q·Kᵀ
    static constexpr int NTD = HD / 8;                // n-tiles of p·V
    static constexpr bool Q_REGS = HD <= 128;         // keep q fragments in registers (else smem)
    static constexpr float TAU = 8.f;                 // lazy-rescale threshold
    static constexpr float OFF = 7.f;                 // p headroom: max p in [2^OFF, 2^(OFF+TAU)]
    static constexpr uint32_t QT_BYTES = 16u * HD * 2;  // Q tile, f16, swizzled like K
    static constexpr uint32_t EXTRA_BYTES = QT_BYTES + 8 * 4;

    uint32_t qa[Q_REGS ? KSTEPS : 1][4];
    float o[NTD][4];
    float m_ref, l, inv_sc;

    // a2: Q tile rows g (hi) and 8 + g (lo) for g < G, zero rows for g >= G,
    // and the per-head power-of-two scale. Warp w takes heads w, w + NW, ...;
    // all of a warp's loads are issued before any of its reductions.
    template <int NTHREADS>
    static __device__ __forceinline__ void prepare(uint8_t *extra, const PartialArgs &a, int s,
                                                   int hk, int, int tid)
    {
        const float *qg = a.q + ((size_t)s * a.n_head + (size_t)hk * G) * HD;
        const float qscale = a.qscale;
        constexpr int NW = NTHREADS / 32;
        constexpr int ITER = (8 + NW - 1) / NW;           // heads per warp
        constexpr int PER = (HD + 31) / 32;               // elements per lane per head
        static_assert(PER % 2 == 0 && PER <= 8, "lane owns PER consecutive elements");
        float *inv = reinterpret_cast<float *>(extra + QT_BYTES);
        const int warp = tid >> 5, lane = tid & 31;
        // lane owns elements [lane * PER, lane * PER + PER) of a head: one or
        // two 16-byte loads (8 bytes at head_dim 64) per head row, so the many
        // blocks reading the same q lines send few requests
        // a slot past G loads nothing (warp-uniform): re-reading head 0 for
        // it would pile more requests onto the lines every block of the KV
        // head already reads
        float x[ITER][PER];
#pragma unroll
        for (int it = 0; it < ITER; ++it) {
            const int g = warp + it * NW;
#pragma unroll
            for (int j = 0; j < PER; ++j) x[it][j] = 0.f;
            if (g >= G) continue;
            const float *row = qg + g * HD + lane * PER;
            if constexpr (PER == 2) {
                const float2 u = ld_dep(reinterpret_cast<const float2 *>(row));
                x[it][0] = u.x;
                x[it][1] = u.y;
            } else {
#pragma unroll
                for (int j = 0; j < PER; j += 4) {
                    const float4 u = ld_dep(reinterpret_cast<const float4 *>(row + j));
                    x[it][j] = u.x;
                    x[it][j + 1] = u.y;
                    x[it][j + 2] = u.z;
                    x[it][j + 3] = u.w;
                }
            }
        }
#pragma unroll
        for (int it = 0; it < ITER; ++it)
#pragma unroll
            for (int j = 0; j < PER; ++j) x[it][j] = warp + it * NW < G ? x[it][j] * qscale : 0.f;
#pragma unroll
        for (int it = 0; it < ITER; ++it) {
            const int g = warp + it * NW;
            if (g >= 8) break;                            // warp-uniform
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < PER; ++i) amax = fmaxf(amax, fabsf(x[it][i]));
            amax = warp_max(amax);
            float sc, ig;                                 // scaled max in [2^14, 2^15)
            pow2_scale(amax, sc, ig);
            if (lane == 0) inv[g] = ig;
            // hi = T(v), lo = T(v - hi) element by element, packed in pairs; the
            // lane's PER elements share one 16-byte unit of the swizzled tile
            uint32_t hw[PER / 2], lw[PER / 2];
#pragma unroll
            for (int j = 0; j < PER / 2; ++j) {
                const float v0 = x[it][2 * j] * sc, v1 = x[it][2 * j + 1] * sc;
                hw[j] = float2_to_kv2<KV>(v0, v1);
                const float2 f = kv2_to_float2<KV>(hw[j]);
                lw[j] = float2_to_kv2<KV>(v0 - f.x, v1 - f.y);
            }
            const int d0 = lane * PER;
            const uint32_t off = tile_unit_offset<HD, 16>(g, d0 >> 3) + (d0 & 7) * 2;
            const uint32_t offl = tile_unit_offset<HD, 16>(8 + g, d0 >> 3) + (d0 & 7) * 2;
            if constexpr (PER == 2) {
                *reinterpret_cast<uint32_t *>(extra + off) = hw[0];
                *reinterpret_cast<uint32_t *>(extra + offl) = lw[0];
            } else if constexpr (PER == 4) {
                *reinterpret_cast<uint2 *>(extra + off) = make_uint2(hw[0], hw[1]);
                *reinterpret_cast<uint2 *>(extra + offl) = make_uint2(lw[0], lw[1]);
            } else {
                *reinterpret_cast<uint4 *>(extra + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(extra + offl) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
        }
    }

    // A fragment (16 x 16) of Q for k-step kk: matrices (hi, d 0-7), (lo, d 0-7),
    // (hi, d 8-15), (lo, d 8-15).
    static __device__ __forceinline__ void load_q(uint32_t (&a)[4], const uint8_t *extra, int kk,
                                                  int lane)
    {
        const int i = lane >> 3;
        const int row = (i & 1) * 8 + (lane & 7);
        ldsm_x4(a, extra + tile_unit_offset<HD, 16>(row, 2 * kk + (i >> 1)));
    }

    __device__ __forceinline__ void init(const uint8_t *extra, int, int lane)
    {
        if constexpr (Q_REGS) {
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) load_q(qa[kk], extra, kk, lane);
        }
#pragma unroll
        for (int n = 0; n < NTD; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[n][i] = 0.f;
        m_ref = -INFINITY;
        l = 0.f;
        inv_sc = reinterpret_cast<const float *>(extra + QT_BYTES)[lane >> 2];
    }

    // Rows [r0 + ra, r0 + 16) of a TILE-row stage are in range (0 <= ra < 16);
    // rows before ra hold finite data (zeros or rows already attended).
    template <int TILE>
    __device__ __forceinline__ void process(const uint8_t *ks, const uint8_t *vs, int r0, int ra,
                                            int64_t, int64_t, const PartialArgs &,
                                            uint8_t *extra, int, int lane)
    {
        // a3: scores of the slice's 16 rows for all heads; even and odd
        // k-steps accumulate into separate fragments (two independent MMA
        // chains of half the depth), added at the end
        float c[2][2][4];
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int i = 0; i < 4; ++i) c[e][n][i] = 0.f;
        const int i8 = lane >> 3;
        const int krow = r0 + (i8 >> 1) * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            uint32_t a[4];
            if constexpr (Q_REGS) {
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = qa[kk][i];
            } else {
                load_q(a, extra, kk, lane);
            }
            uint32_t b[4];        // (rows 0-7, d lo8), (rows 0-7, d hi8), (rows 8-15, lo8), (8-15, hi8)
            ldsm_x4(b, ks + tile_unit_offset<HD, TILE>(krow, 2 * kk + (i8 & 1)));
            mma_16816<KV>(c[kk & 1][0], a, b[0], b[1]);
            mma_16816<KV>(c[kk & 1][1], a, b[2], b[3]);
        }
        const int t = lane & 3;
        float s[4];
        s[0] = ((c[0][0][0] + c[1][0][0]) + (c[0][0][2] + c[1][0][2])) * inv_sc;   // row 2t
        s[1] = ((c[0][0][1] + c[1][0][1]) + (c[0][0][3] + c[1][0][3])) * inv_sc;   // row 2t + 1
        s[2] = ((c[0][1][0] + c[1][1][0]) + (c[0][1][2] + c[1][1][2])) * inv_sc;   // row 8 + 2t
        s[3] = ((c[0][1][1] + c[1][1][1]) + (c[0][1][3] + c[1][1][3])) * inv_sc;   // row 9 + 2t
        if (2 * t < ra) s[0] = -INFINITY;
        if (2 * t + 1 < ra) s[1] = -INFINITY;
        if (8 + 2 * t < ra) s[2] = -INFINITY;
        if (9 + 2 * t < ra) s[3] = -INFINITY;
        // a4: slice max of head g (the four lanes of the group), lazy rescale
        float mt = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
        const bool need = mt > m_ref + TAU;
        if (__any_sync(0xffffffffu, need)) {
            const float nr = need ? mt : m_ref;
            const float corr = ex2(m_ref - nr);  // 0 on the first slice (m_ref = -inf)
#pragma unroll
            for (int n = 0; n < NTD; ++n)
#pragma unroll
                for (int i = 0; i < 4; ++i) o[n][i] *= corr;
            l *= corr;
            m_ref = nr;
        }
        const float base = m_ref - OFF;
        float p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) p[i] = ex2(s[i] - base);
        l += (p[0] + p[1]) + (p[2] + p[3]);
        // p as the A fragment of p·V: hi parts in rows 0-7, lo parts in rows 8-15
        uint32_t pa[4];
        {
            pa[0] = float2_to_kv2<KV>(p[0], p[1]);
            pa[2] = float2_to_kv2<KV>(p[2], p[3]);
            const float2 f01 = kv2_to_float2<KV>(pa[0]), f23 = kv2_to_float2<KV>(pa[2]);
            pa[1] = float2_to_kv2<KV>(p[0] - f01.x, p[1] - f01.y);
            pa[3] = float2_to_kv2<KV>(p[2] - f23.x, p[3] - f23.y);
        }
        // a5: O += P · V over the slice's 16 rows
        const int vrow = r0 + (i8 & 1) * 8 + (lane & 7);
#pragma unroll
        for (int n = 0; n < NTD; n += 2) {
            uint32_t b[4];        // (rows 0-7, dims n), (rows 8-15, dims n), (0-7, n+1), (8-15, n+1)
            ldsm_x4_trans(b, vs + tile_unit_offset<HD, TILE>(vrow, n + (i8 >> 1)));
            mma_16816<KV>(o[n], pa, b[0], b[1]);
            mma_16816<KV>(o[n + 1], pa, b[2], b[3]);
        }
    }

    // mm[g] = (mx, S) in the partial's convention (mx is the reference the p's
    // were taken against), mo[g * merge_stride + d] = oc.
    __device__ __forceinline__ void publish(float2 *mm, float *mo, int lane)
    {
        constexpr int MS = merge_stride<HD>();
        float lt = l;
        lt += __shfl_xor_sync(0xffffffffu, lt, 1);
        lt += __shfl_xor_sync(0xffffffffu, lt, 2);
        const int g = lane >> 2, t = lane & 3;
        if (g < G) {
            if (t == 0) mm[g] = make_float2(m_ref - OFF, lt);
#pragma unroll
            for (int n = 0; n < NTD; ++n)
                *reinterpret_cast<float2 *>(mo + g * MS + n * 8 + 2 * t) =
                    make_float2(o[n][0] + o[n][2], o[n][1] + o[n][3]);
        }
    }
};

} // namespace attn
