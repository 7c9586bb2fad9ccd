// attn_warp_tcmq.cuh -- tensor-core per-warp arithmetic for several query rows
// per sequence (causal multi-query decode: speculative drafts, short chunks).
//
// dotLLM #199 §2 gates the decode kernel to one query row and notes that
// more rows need a causal mask whose offset is the query's position
// ("gq = positionOffset"). Here a block serves up to QH = 16 query heads of one
// KV head -- (query row t, group head g) pairs -- against one K/V read. The 16
// MMA rows are those query heads; q is carried as separate hi and lo MMA
// operands (two MMAs per k-step, products exact in f32), and so is p. Query
// row t of a sequence whose last position is positions[s] sits at position
// nkv - n_q + t and sees cache rows [0, nkv - n_q + t].
//
// Lane l owns query heads g = l / 4 and g + 8 (two online-softmax states) and
// rows {2u, 2u+1, 8+2u, 9+2u} (u = l % 4) of the slice's scores.
#pragma once

#include "attn_device.cuh"

namespace attn {

template <int HD, int QH, int NWC, typename KV>
struct TcWarpMQ {
    static_assert(HD % 16 == 0 && QH <= 16, "tensor-core multi-query needs head_dim % 16 == 0");
    static constexpr int WR = 16;
    static constexpr bool WHOLE_TILE_SPLITS = false;      // count-mode splits in warp slices
    static constexpr int NQH = QH;
    static constexpr int KSTEPS = HD / 16;
    static constexpr int NTD = HD / 8;
    static constexpr float TAU = 8.f;                 // lazy-rescale threshold (log2 units)
    static constexpr float OFF = 7.f;                 // p headroom
    static constexpr uint32_t QT_BYTES = 16u * HD * 2;
    static constexpr uint32_t EXTRA_BYTES = 2 * QT_BYTES + 16 * 4 + 16 * 4;

    float o[NTD][4];
    float m_ref[2], l[2], inv_sc[2];
    int qrow[2];                                      // query row t of the lane's heads, -1 if none

    // Block-local query head i -> (t, g) -> partial-head index t * n_head + hk * G + g.
    static __device__ __forceinline__ int slot_head(const PartialArgs &a, int hk, int qg, int i)
    {
        const int G = a.group;
        const int qh = qg * QH + i;
        if (i >= QH || qh >= a.n_q * G) return -1;
        const int t = div_group(a, qh), g = qh - t * G;
        return t * a.n_head + hk * G + g;
    }

    // a2: Q hi and lo tiles (16 rows each), per-head power-of-two scales, and
    // the query row of each block-local head. Warp w takes heads w, w + NW, ...
    template <int NTHREADS>
    static __device__ __forceinline__ void prepare(uint8_t *extra, const PartialArgs &a, int s,
                                                   int hk, int qg, int tid)
    {
        constexpr int NW = NTHREADS / 32;
        constexpr int ITER = (16 + NW - 1) / NW;
        constexpr int PER = (HD + 31) / 32;
        static_assert(PER % 2 == 0 && PER <= 8, "lane owns PER consecutive elements");
        float *inv = reinterpret_cast<float *>(extra + 2 * QT_BYTES);
        int *qr = reinterpret_cast<int *>(inv + 16);
        const int warp = tid >> 5, lane = tid & 31;
        const int G = a.group;
        // lane owns elements [lane * PER, lane * PER + PER) of a head row: one
        // or two 16-byte loads (8 bytes at head_dim 64) per row, few requests
        // for the q lines that every split's block reads
        // Every row's load is issued unconditionally -- a head the block does
        // not have reads the block's first (row, head) pair instead, which
        // always exists, and is zeroed afterwards -- so that all of a lane's
        // loads leave back to back.
        float x[ITER][PER];
        bool have[ITER];
#pragma unroll
        for (int it = 0; it < ITER; ++it) {
            const int i = warp + it * NW;
            const int hp = i < 16 ? slot_head(a, hk, qg, i) : -1;
            have[it] = hp >= 0;
            const int qh = qg * QH + (have[it] ? i : 0);
            const int t = div_group(a, qh);
            const int g = hk * G + qh - t * G;
            const float *qrow_p = a.q + (((size_t)s * a.n_q + t) * a.n_head + g) * HD + lane * PER;
            if constexpr (PER == 2) {
                const float2 u = ld_dep(reinterpret_cast<const float2 *>(qrow_p));
                x[it][0] = u.x;
                x[it][1] = u.y;
            } else {
#pragma unroll
                for (int j = 0; j < PER; j += 4) {
                    const float4 u = ld_dep(reinterpret_cast<const float4 *>(qrow_p + j));
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
            for (int j = 0; j < PER; ++j) x[it][j] = have[it] ? x[it][j] * a.qscale : 0.f;
#pragma unroll
        for (int it = 0; it < ITER; ++it) {
            const int i = warp + it * NW;
            if (i >= 16) break;                                   // warp-uniform
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < PER; ++k) amax = fmaxf(amax, fabsf(x[it][k]));
            amax = warp_max(amax);
            float sc, ig;
            pow2_scale(amax, sc, ig);
            if (lane == 0) {
                inv[i] = ig;
                const int hp = slot_head(a, hk, qg, i);
                qr[i] = hp >= 0 ? div_group(a, qg * QH + i) : -1;
            }
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
            const uint32_t off = tile_unit_offset<HD, 16>(i, d0 >> 3) + (d0 & 7) * 2;
            if constexpr (PER == 2) {
                *reinterpret_cast<uint32_t *>(extra + off) = hw[0];
                *reinterpret_cast<uint32_t *>(extra + QT_BYTES + off) = lw[0];
            } else if constexpr (PER == 4) {
                *reinterpret_cast<uint2 *>(extra + off) = make_uint2(hw[0], hw[1]);
                *reinterpret_cast<uint2 *>(extra + QT_BYTES + off) = make_uint2(lw[0], lw[1]);
            } else {
                *reinterpret_cast<uint4 *>(extra + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(extra + QT_BYTES + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
        }
    }

    // A fragment of a 16-row Q tile (hi or lo) for k-step kk.
    static __device__ __forceinline__ void load_q(uint32_t (&a)[4], const uint8_t *tile, int kk,
                                                  int lane)
    {
        const int i = lane >> 3;
        ldsm_x4(a, tile + tile_unit_offset<HD, 16>((i & 1) * 8 + (lane & 7), 2 * kk + (i >> 1)));
    }

    __device__ __forceinline__ void init(const uint8_t *extra, int, int lane)
    {
#pragma unroll
        for (int n = 0; n < NTD; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[n][i] = 0.f;
        const float *inv = reinterpret_cast<const float *>(extra + 2 * QT_BYTES);
        const int *qr = reinterpret_cast<const int *>(inv + 16);
        const int g = lane >> 2;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            m_ref[k] = -INFINITY;
            l[k] = 0.f;
            inv_sc[k] = inv[g + 8 * k];
            qrow[k] = qr[g + 8 * k];
        }
    }

    // Rows [r0 + ra, r0 + 16) of the tile are in range; tile row r is cache row
    // row0 + r of the sequence, which has nkv rows.
    template <int TILE>
    __device__ __forceinline__ void process(const uint8_t *ks, const uint8_t *vs, int r0, int ra,
                                            int64_t row0, int64_t nkv, const PartialArgs &a,
                                            uint8_t *extra, int, int lane)
    {
        // a3: scores, C rows = query heads, C columns = the slice's rows; the
        // hi and lo parts of q accumulate separately (two independent MMA
        // chains) and are added at the end
        float ch[2][4], cl[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) ch[n][i] = cl[n][i] = 0.f;
        const int i8 = lane >> 3;
        const int krow = r0 + (i8 >> 1) * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            uint32_t ah[4], al[4], b[4];
            load_q(ah, extra, kk, lane);
            load_q(al, extra + QT_BYTES, kk, lane);
            ldsm_x4(b, ks + tile_unit_offset<HD, TILE>(krow, 2 * kk + (i8 & 1)));
            mma_16816<KV>(ch[0], ah, b[0], b[1]);
            mma_16816<KV>(cl[0], al, b[0], b[1]);
            mma_16816<KV>(ch[1], ah, b[2], b[3]);
            mma_16816<KV>(cl[1], al, b[2], b[3]);
        }
        float c[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) c[n][i] = ch[n][i] + cl[n][i];
        const int u = lane & 3;
        const int cols[4] = {2 * u, 2 * u + 1, 8 + 2 * u, 9 + 2 * u};
        float sc[2][4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            // causal limit: cache rows <= nkv - n_q + t; slice row -> tile row r0 + col
            const int64_t last = qrow[k] >= 0 ? nkv - a.n_q + qrow[k] : (int64_t)-1;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float raw = (j < 2 ? c[0][2 * k + j] : c[1][2 * k + j - 2]) * inv_sc[k];
                const int col = cols[j];
                const bool ok = col >= ra && row0 + r0 + col <= last;
                sc[k][j] = ok ? raw : -INFINITY;
            }
        }
        // a4: per head: slice max over the four lanes of the group, lazy rescale
        float mt[2];
        bool need[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            float m = fmaxf(fmaxf(sc[k][0], sc[k][1]), fmaxf(sc[k][2], sc[k][3]));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            mt[k] = m;
            need[k] = m > m_ref[k] + TAU;
        }
        if (__any_sync(0xffffffffu, need[0] || need[1])) {
            float corr[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float nr = need[k] ? mt[k] : m_ref[k];
                corr[k] = need[k] ? ex2(m_ref[k] - nr) : 1.f;    // 0 when m_ref was -inf
                l[k] *= corr[k];
                m_ref[k] = nr;
            }
#pragma unroll
            for (int n = 0; n < NTD; ++n) {
                o[n][0] *= corr[0]; o[n][1] *= corr[0];
                o[n][2] *= corr[1]; o[n][3] *= corr[1];
            }
        }
        float p[2][4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float base = m_ref[k] == -INFINITY ? 0.f : m_ref[k] - OFF;   // no row seen yet
#pragma unroll
            for (int j = 0; j < 4; ++j) p[k][j] = ex2(sc[k][j] - base);
            l[k] += (p[k][0] + p[k][1]) + (p[k][2] + p[k][3]);
        }
        // p as A fragments (rows g / g + 8 = the two heads), hi and lo parts
        uint32_t ph[4], pl[4];
        ph[0] = float2_to_kv2<KV>(p[0][0], p[0][1]);
        ph[1] = float2_to_kv2<KV>(p[1][0], p[1][1]);
        ph[2] = float2_to_kv2<KV>(p[0][2], p[0][3]);
        ph[3] = float2_to_kv2<KV>(p[1][2], p[1][3]);
        {
            const float2 f0 = kv2_to_float2<KV>(ph[0]), f1 = kv2_to_float2<KV>(ph[1]);
            const float2 f2 = kv2_to_float2<KV>(ph[2]), f3 = kv2_to_float2<KV>(ph[3]);
            pl[0] = float2_to_kv2<KV>(p[0][0] - f0.x, p[0][1] - f0.y);
            pl[1] = float2_to_kv2<KV>(p[1][0] - f1.x, p[1][1] - f1.y);
            pl[2] = float2_to_kv2<KV>(p[0][2] - f2.x, p[0][3] - f2.y);
            pl[3] = float2_to_kv2<KV>(p[1][2] - f3.x, p[1][3] - f3.y);
        }
        // a5: O += P · V
        const int vrow = r0 + (i8 & 1) * 8 + (lane & 7);
#pragma unroll
        for (int n = 0; n < NTD; n += 2) {
            uint32_t b[4];
            ldsm_x4_trans(b, vs + tile_unit_offset<HD, TILE>(vrow, n + (i8 >> 1)));
            mma_16816<KV>(o[n], ph, b[0], b[1]);
            mma_16816<KV>(o[n], pl, b[0], b[1]);
            mma_16816<KV>(o[n + 1], ph, b[2], b[3]);
            mma_16816<KV>(o[n + 1], pl, b[2], b[3]);
        }
    }

    // mm[h] = (mx, S) and mo[h * merge_stride + d] = oc for the block-local
    // heads h = g and g + 8 of lane group g.
    __device__ __forceinline__ void publish(float2 *mm, float *mo, int lane)
    {
        const int g = lane >> 2, u = lane & 3;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            float lt = l[k];
            lt += __shfl_xor_sync(0xffffffffu, lt, 1);
            lt += __shfl_xor_sync(0xffffffffu, lt, 2);
            const int h = g + 8 * k;
            if (h < QH) {
                if (u == 0) mm[h] = make_float2(m_ref[k] - OFF, lt);
#pragma unroll
                for (int n = 0; n < NTD; ++n)
                    *reinterpret_cast<float2 *>(mo + h * merge_stride<HD>() + n * 8 + 2 * u) =
                        make_float2(o[n][2 * k], o[n][2 * k + 1]);
            }
        }
    }
};

} // namespace attn
