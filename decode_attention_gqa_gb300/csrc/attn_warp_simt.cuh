// attn_warp_simt.cuh -- CUDA-core (f32) per-warp arithmetic of the partial
// kernel: steps a3-a5 for one warp's slice of a shared-memory tile.
//
// Scores: one lane per cache row, all G heads, q broadcast from shared memory
// (Red Lite dev35 "Change": one thread per position). Values: lanes own
// head_dim slices and walk the rows (one thread per dimension; minfer
// "10 · R4" §2.4 lane<->dim binding), p broadcast from shared memory. The
// online-softmax state (mx, S, oc) of all G heads stays in registers (§2.4,
// §6 lesson 1: compile-time extents, no local memory).
#pragma once

#include "attn_device.cuh"

namespace attn {

template <int HD, int G, int NWC, typename KV>
struct SimtWarp {
    static constexpr int WR = 32;                          // rows per warp slice
    static constexpr bool WHOLE_TILE_SPLITS = false;      // count-mode splits in warp slices
    static constexpr int NQH = G;                     // query heads per block (one query row)

    // Partial-head index of block-local query head i (single query row: the
    // group's heads hk*G .. hk*G+G-1).
    static __device__ __forceinline__ int slot_head(const PartialArgs &a, int hk, int, int i)
    {
        (void)a;
        return hk * G + i;
    }
    static constexpr int NU = HD / 8;                      // 16-byte units per row
    static constexpr int DPL = HD >= 64 ? HD / 32 : 2;     // dims per lane, value phase
    static constexpr int LPRV = HD / DPL;                  // lanes per row, value phase
    static constexpr int RGV = 32 / LPRV;                  // rows per value step
    static constexpr int GP = (G + 3) / 4 * 4;             // padded p row
    static constexpr uint32_t Q_BYTES = (uint32_t)G * HD * 4;
    static constexpr uint32_t PS_BYTES = (uint32_t)NWC * WR * GP * 4;
    static constexpr uint32_t EXTRA_BYTES = Q_BYTES + PS_BYTES;

    float m[G], l[G], o[G][DPL];

    // a2: the group's G query rows (f32), pre-multiplied by scale*log2(e),
    // into shared memory. All threads of the block take part.
    template <int NTHREADS>
    static __device__ __forceinline__ void prepare(uint8_t *extra, const PartialArgs &a, int s,
                                                   int hk, int, int tid)
    {
        const float *qg = a.q + ((size_t)s * a.n_head + (size_t)hk * G) * HD;
        const float qscale = a.qscale;
        constexpr int N4 = G * HD / 4;                    // float4s of the group's q
        constexpr int ITER = (N4 + NTHREADS - 1) / NTHREADS;
        const float4 *src = reinterpret_cast<const float4 *>(qg);
        float4 *dst = reinterpret_cast<float4 *>(extra);
        float4 t[ITER];
#pragma unroll
        for (int it = 0; it < ITER; ++it) {
            const int i = tid + it * NTHREADS;
            if (i < N4) t[it] = ld_dep(src + i);
        }
#pragma unroll
        for (int it = 0; it < ITER; ++it) {
            const int i = tid + it * NTHREADS;
            if (i < N4) {
                float4 u = t[it];
                u.x *= qscale; u.y *= qscale; u.z *= qscale; u.w *= qscale;
                dst[i] = u;
            }
        }
    }

    __device__ __forceinline__ void init(const uint8_t *, int, int)
    {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int d = 0; d < DPL; ++d) o[g][d] = 0.f;
        }
    }

    // Rows [r0 + ra, r0 + WR) of a TILE-row stage are in range (0 <= ra < WR).
    template <int TILE>
    __device__ __forceinline__ void process(const uint8_t *ks, const uint8_t *vs, int r0, int ra,
                                            int64_t, int64_t, const PartialArgs &,
                                            uint8_t *extra, int warp, int lane)
    {
        const float *qs = reinterpret_cast<const float *>(extra);
        float *ps = reinterpret_cast<float *>(extra + Q_BYTES) + warp * WR * GP;
        // a3: scores for row r0 + lane, all heads (log2 units)
        float acc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = 0.f;
        const int r = r0 + lane;
        constexpr int UNROLL = (HD >= 256 && G >= 7) ? 1 : 2;   // register budget of the largest shapes
#pragma unroll UNROLL
        for (int U = 0; U < NU; ++U) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(ks + tile_unit_offset<HD, TILE>(r, U));
            float kf[8];
            unpack8<KV>(raw, kf);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float4 qa = *reinterpret_cast<const float4 *>(qs + g * HD + U * 8);
                const float4 qb = *reinterpret_cast<const float4 *>(qs + g * HD + U * 8 + 4);
                float t = acc[g];
                t = fmaf(qa.x, kf[0], t); t = fmaf(qa.y, kf[1], t);
                t = fmaf(qa.z, kf[2], t); t = fmaf(qa.w, kf[3], t);
                t = fmaf(qb.x, kf[4], t); t = fmaf(qb.y, kf[5], t);
                t = fmaf(qb.z, kf[6], t); t = fmaf(qb.w, kf[7], t);
                acc[g] = t;
            }
        }
        // a4: online softmax, warp-uniform per head ("10 · R4" §2.1 update,
        // applied per slice: slice max first, then one rescale)
        float corr[G];
        const bool valid = lane >= ra;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float sg = valid ? acc[g] : -INFINITY;
            const float mn = fmaxf(m[g], warp_max(sg));
            corr[g] = ex2(m[g] - mn);
            const float p = ex2(sg - mn);
            l[g] = fmaf(l[g], corr[g], p);       // per-lane piece of S
            m[g] = mn;
            ps[lane * GP + g] = p;
        }
        __syncwarp();
        // a5: rescale, then accumulate p * V over the lane's head_dim slice
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int d = 0; d < DPL; ++d) o[g][d] *= corr[g];
        const int rg = lane / LPRV, dl = lane % LPRV;
        const int d0 = dl * DPL;
        const uint32_t vbyte = (d0 & 7) * 2;
        const int j0 = rg + (ra > rg ? (ra - rg + RGV - 1) / RGV * RGV : 0);
#pragma unroll 2
        for (int j = j0; j < WR; j += RGV) {
            const uint8_t *vp = vs + tile_unit_offset<HD, TILE>(r0 + j, d0 >> 3) + vbyte;
            float v[DPL];
            if constexpr (DPL == 8) {
                unpack8<KV>(*reinterpret_cast<const uint4 *>(vp), v);
            } else if constexpr (DPL == 4) {
                const uint2 raw = *reinterpret_cast<const uint2 *>(vp);
                const float2 a = kv2_to_float2<KV>(raw.x);
                const float2 b = kv2_to_float2<KV>(raw.y);
                v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
            } else {
                const float2 a = kv2_to_float2<KV>(*reinterpret_cast<const uint32_t *>(vp));
                v[0] = a.x; v[1] = a.y;
            }
            float p[GP];
#pragma unroll
            for (int i = 0; i < GP; i += 4) {
                const float4 t = *reinterpret_cast<const float4 *>(ps + j * GP + i);
                p[i] = t.x; p[i + 1] = t.y; p[i + 2] = t.z; p[i + 3] = t.w;
            }
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int d = 0; d < DPL; ++d) o[g][d] = fmaf(p[g], v[d], o[g][d]);
        }
        __syncwarp();
    }

    // Reduce the per-lane pieces and publish (mx, S) and oc of every head:
    // mm[g] = (mx, S), mo[g * merge_stride + d] = oc.
    __device__ __forceinline__ void publish(float2 *mm, float *mo, int lane)
    {
#pragma unroll
        for (int g = 0; g < G; ++g) l[g] = warp_sum(l[g]);
        if constexpr (RGV > 1) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int d = 0; d < DPL; ++d)
#pragma unroll
                    for (int off = LPRV; off < 32; off <<= 1)
                        o[g][d] += __shfl_xor_sync(0xffffffffu, o[g][d], off);
        }
        if (lane == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) mm[g] = make_float2(m[g], l[g]);
        }
        if (lane < LPRV) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int d = 0; d < DPL; ++d) mo[g * merge_stride<HD>() + lane * DPL + d] = o[g][d];
        }
    }
};

} // namespace attn
