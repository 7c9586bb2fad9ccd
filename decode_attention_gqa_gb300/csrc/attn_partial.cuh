// attn_partial.cuh -- the split partial kernel (steps a1-a6).
//
// One block per (split sp, KV head hk, sequence s) -- the static grid of
// minfer "10 · R4" §2.2 with the KV head replacing the query head, so that the
// whole query-head group is served from one K/V read (Red Lite dev35 "Change").
//
// Block = NWC compute warps + 1 producer warp. The producer streams the
// split's rows through an S-stage ring of shared-memory tiles with TMA
// (cp.async.bulk.tensor, 128-byte swizzle); tile t holds rows
// [lo + t*TILE, lo + (t+1)*TILE) of K and of V. Compute warp w owns rows
// [w*WR, (w+1)*WR) of every tile and keeps its own online-softmax state
// (mx, S, oc) for all G heads in registers (§2.1 update, §2.4 register
// accumulator); at the end the NWC states are merged in shared memory and the
// block writes one partial triple per query head (§3.2 "partial write-out").
//
// The per-warp arithmetic is a policy class (Warp): SimtWarp here (CUDA cores,
// f32), TcWarp in attn_partial_tc.cuh (tensor cores).
#pragma once

#include "attn_device.cuh"

namespace attn {

// ---------------------------------------------------------------------------
// CUDA-core policy. Scores: one lane per cache row, all G heads, q broadcast
// from shared memory (Red Lite dev35 "Change": one thread per position).
// Values: lanes own head_dim slices and walk the rows (one thread per
// dimension; R4 §2.4 lane<->dim binding), p broadcast from shared memory.
// ---------------------------------------------------------------------------
template <int HD, int G>
struct SimtWarp {
    static constexpr int WR = 32;                          // rows per warp slice
    static constexpr int NU = HD / 8;                      // 16-byte units per row
    static constexpr int DPL = HD >= 64 ? HD / 32 : 2;     // dims per lane, value phase
    static constexpr int LPRV = HD / DPL;                  // lanes per row, value phase
    static constexpr int RGV = 32 / LPRV;                  // rows per value step
    static constexpr int GP = (G + 3) / 4 * 4;             // padded p row
    static constexpr int PS_FLOATS = WR * GP;              // per-warp p scratch
    static constexpr bool Q_IN_SMEM = true;

    float m[G], l[G], o[G][DPL];

    __device__ __forceinline__ void init()
    {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int d = 0; d < DPL; ++d) o[g][d] = 0.f;
        }
    }

    // Process rows [r0, r0 + nvalid) of a TILE-row stage (nvalid >= 1).
    template <int TILE>
    __device__ __forceinline__ void process(const uint8_t *ks, const uint8_t *vs, int r0, int nvalid,
                                            const float *qs, float *ps, int lane)
    {
        // a3: scores for row r0 + lane, all heads (log2 units: q carries scale*log2 e)
        float acc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = 0.f;
        const int r = r0 + lane;
#pragma unroll 2
        for (int U = 0; U < NU; ++U) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(ks + tile_unit_offset<HD, TILE>(r, U));
            float kf[8];
            unpack8(raw, kf);
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
        // a4: online softmax, warp-uniform per head (R4 §2.1 update rule,
        // applied once per WR-row slice: tile max first, then the rescale)
        float corr[G];
        const bool valid = lane < nvalid;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float sg = valid ? acc[g] : -INFINITY;
            const float mn = fmaxf(m[g], warp_max(sg));
            corr[g] = ex2(m[g] - mn);
            const float p = ex2(sg - mn);
            l[g] = fmaf(l[g], corr[g], p);       // per-lane partial of S
            m[g] = mn;
            ps[lane * GP + g] = p;
        }
        __syncwarp();
        // a5: rescale and accumulate p * V for the lane's head_dim slice
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int d = 0; d < DPL; ++d) o[g][d] *= corr[g];
        const int rg = lane / LPRV, dl = lane % LPRV;
        const int d0 = dl * DPL;
        const uint32_t vbyte = ((d0 & 7) * 2);
#pragma unroll 2
        for (int j = rg; j < nvalid; j += RGV) {
            const uint8_t *vp = vs + tile_unit_offset<HD, TILE>(r0 + j, d0 >> 3) + vbyte;
            float v[DPL];
            if constexpr (DPL == 8) {
                unpack8(*reinterpret_cast<const uint4 *>(vp), v);
            } else if constexpr (DPL == 4) {
                const uint2 raw = *reinterpret_cast<const uint2 *>(vp);
                const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
                const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
                v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
            } else {
                const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(vp));
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

    // Reduce the per-lane pieces and publish (mx, S) and oc for the merge.
    // mm: [G] float2 for this warp, mo: [G][HD] floats for this warp.
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
                for (int d = 0; d < DPL; ++d) mo[g * HD + lane * DPL + d] = o[g][d];
        }
    }
};

// ---------------------------------------------------------------------------
// Block configuration per policy.
// ---------------------------------------------------------------------------
template <int HD, int G, template <int, int> class W, int NWC_, int S_>
struct PartialCfg {
    using Warp = W<HD, G>;
    static constexpr int NWC = NWC_;                 // compute warps
    static constexpr int S = S_;                     // pipeline stages
    static constexpr int WR = Warp::WR;
    static constexpr int TILE = NWC * WR;            // rows per stage
    static constexpr int THREADS = (NWC + 1) * 32;
    static constexpr int NCH = HD >= 64 ? HD / 64 : 1;
    static constexpr int BOX_X = HD >= 64 ? 64 : HD; // TMA box inner extent (elements)
    static constexpr uint32_t TILE_BYTES = (uint32_t)TILE * HD * 2;        // one of K or V
    static constexpr uint32_t STAGE_BYTES = 2 * TILE_BYTES;
    // shared-memory carve-up (byte offsets; stage buffers first, 1024-aligned)
    static constexpr uint32_t OFF_STAGES = 0;
    static constexpr uint32_t OFF_Q = S * STAGE_BYTES;
    static constexpr uint32_t Q_BYTES = Warp::Q_IN_SMEM ? (uint32_t)G * HD * 4 : 0;
    static constexpr uint32_t OFF_PS = OFF_Q + Q_BYTES;
    static constexpr uint32_t PS_BYTES = (uint32_t)NWC * Warp::PS_FLOATS * 4;
    static constexpr uint32_t OFF_BAR = (OFF_PS + PS_BYTES + 15) / 16 * 16;
    static constexpr uint32_t BAR_BYTES = 2 * S * 8 + 16;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;   // + alignment slack
    // merge area (reuses the stage buffers after the main loop)
    static constexpr uint32_t MERGE_BYTES = (uint32_t)NWC * G * (HD + 2) * 4;
    static_assert(MERGE_BYTES <= S * STAGE_BYTES, "merge area must fit in the stage buffers");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert((TILE_BYTES / NCH) % 1024 == 0 || HD < 64, "swizzled chunks must stay 1024-aligned");
};

template <class Cfg, int HD, int G>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
attn_split_partial(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const PartialArgs a)
{
    using Warp = typename Cfg::Warp;
    constexpr int NWC = Cfg::NWC, S = Cfg::S, TILE = Cfg::TILE, WR = Cfg::WR;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *qs = reinterpret_cast<float *>(smem + Cfg::OFF_Q);
    float *ps = reinterpret_cast<float *>(smem + Cfg::OFF_PS);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *empty = full + S;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + S);

    const int sp = blockIdx.x, hk = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = a.n_splits;

    // Inputs may be produced by the previous kernel in the stream: wait for it
    // before the first read, then let the combine kernel get scheduled.
    pdl_wait();
    pdl_launch_dependents();

    // a1: rows attended and this split's range
    const int64_t nkv = rows_attended(a, s, sp == 0 && hk == 0 && tid == 0);
    int64_t lo, hi;
    split_range(nkv, sp, P, a.split_len, lo, hi);
    const size_t head0 = (size_t)s * a.n_head + (size_t)hk * G;          // first query head of the group
    if (lo >= hi) {                                                      // empty split: mx=-inf, S=0
        if (tid < G) a.ws_ml[(head0 + tid) * P + sp] = make_float2(-INFINITY, 0.f);
        return;
    }
    const int ntiles = (int)((hi - lo + TILE - 1) / TILE);
    const int row0 = (int)((int64_t)s * a.cap + lo);                      // first cache row (flat)

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, NWC);
        }
        abort_flag[0] = 0;           // set when a bounded wait gives up
        abort_flag[1] = 0;           // tiles issued by the producer (for the drain)
        fence_barrier_init();
    }
    // a2: the group's query rows, pre-multiplied by scale*log2(e)
    if constexpr (Warp::Q_IN_SMEM) {
        const float4 *qsrc = reinterpret_cast<const float4 *>(a.q + head0 * HD);
        for (int i = tid; i < G * HD / 4; i += Cfg::THREADS) {
            float4 t = __ldg(qsrc + i);
            t.x *= a.qscale; t.y *= a.qscale; t.z *= a.qscale; t.w *= a.qscale;
            reinterpret_cast<float4 *>(qs)[i] = t;
        }
    }
    __syncthreads();

    if (warp == NWC) {
        // ---------------- producer warp ----------------
        // Full tiles arrive by TMA. The last tile of the split, when it holds
        // fewer than TILE rows, is copied by the warp with plain 16-byte loads
        // of exactly the rows in range and zeros after them, so no row at or
        // past hi is ever read from the cache.
        if (lane == 0) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
        }
        for (int t = 0; t < ntiles; ++t) {
            const int st = t % S;
            int ok = 1;
            if (lane == 0) {
                if (t >= S && !mbar_wait_bounded(empty + st, ((t / S) - 1) & 1)) {
                    *abort_flag = 1;
                    atomicOr(a.err, kErrPipelineTimeout);
                }
                ok = !*abort_flag;
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            uint8_t *kst = smem + Cfg::OFF_STAGES + st * Cfg::STAGE_BYTES;
            uint8_t *vst = kst + Cfg::TILE_BYTES;
            const int64_t first = lo + (int64_t)t * TILE;
            const int nrows = (int)(hi - first < TILE ? hi - first : TILE);
            if (nrows == TILE) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(full + st, Cfg::STAGE_BYTES);
#pragma unroll
                    for (int c = 0; c < Cfg::NCH; ++c) {
                        tma_load_3d(kst + c * (Cfg::TILE_BYTES / Cfg::NCH), &kmap, full + st,
                                    c * Cfg::BOX_X, hk, row0 + t * TILE);
                        tma_load_3d(vst + c * (Cfg::TILE_BYTES / Cfg::NCH), &vmap, full + st,
                                    c * Cfg::BOX_X, hk, row0 + t * TILE);
                    }
                }
            } else {
                constexpr int NU = HD / 8;
                const size_t rstride = (size_t)a.n_kv_head * HD;                // elements per cache row
                const __half *kg = a.k + ((size_t)(row0 + t * TILE)) * rstride + (size_t)hk * HD;
                const __half *vg = a.v + ((size_t)(row0 + t * TILE)) * rstride + (size_t)hk * HD;
                for (int i = lane; i < TILE * NU; i += 32) {
                    const int r = i / NU, U = i % NU;
                    uint4 kv4 = make_uint4(0, 0, 0, 0), vv4 = make_uint4(0, 0, 0, 0);
                    if (r < nrows) {
                        kv4 = __ldg(reinterpret_cast<const uint4 *>(kg + (size_t)r * rstride) + U);
                        vv4 = __ldg(reinterpret_cast<const uint4 *>(vg + (size_t)r * rstride) + U);
                    }
                    const uint32_t off = tile_unit_offset<HD, TILE>(r, U);
                    *reinterpret_cast<uint4 *>(kst + off) = kv4;
                    *reinterpret_cast<uint4 *>(vst + off) = vv4;
                }
                __threadfence_block();
                __syncwarp();
                if (lane == 0) mbar_arrive(full + st);
            }
            if (lane == 0) abort_flag[1] = t + 1;
        }
    } else {
        // ---------------- compute warps ----------------
        Warp wst;
        wst.init();
        float *myps = ps + warp * Warp::PS_FLOATS;
        for (int t = 0; t < ntiles; ++t) {
            const int st = t % S;
            const bool landed = mbar_wait_bounded(full + st, (t / S) & 1);
            if (!__all_sync(0xffffffffu, landed)) {
                if (lane == 0) { *abort_flag = 1; atomicOr(a.err, kErrPipelineTimeout); }
                break;
            }
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const uint8_t *kst = smem + Cfg::OFF_STAGES + st * Cfg::STAGE_BYTES;
            const uint8_t *vst = kst + Cfg::TILE_BYTES;
            const int64_t first = lo + (int64_t)t * TILE + warp * WR;
            const int nvalid = (int)(hi - first < WR ? hi - first : WR);
            if (nvalid > 0) wst.template process<TILE>(kst, vst, warp * WR, nvalid, qs, myps, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + st);
        }
        // the merge area overlaps the stage buffers: every compute warp must be
        // done with the ring before any of them publishes its state
        asm volatile("bar.sync 1, %0;" :: "r"(NWC * 32) : "memory");
        if (!__shfl_sync(0xffffffffu, *abort_flag, 0))
            wst.publish(reinterpret_cast<float2 *>(smem) + warp * G,
                        reinterpret_cast<float *>(smem) + 2 * NWC * G + warp * G * HD, lane);
    }
    __syncthreads();

    // Drain: no TMA copy may still be writing shared memory when the block exits.
    if (tid == NWC * 32) {
        const int issued = abort_flag[1];
        for (int t = issued - S > 0 ? issued - S : 0; t < issued; ++t)
            (void)mbar_wait_bounded(full + (t % S), (t / S) & 1);
    }
    if (*abort_flag) return;     // partial left unwritten; the error word says why

    // a6: merge the NWC warp states and write the partial triple of each head
    const float2 *mm = reinterpret_cast<const float2 *>(smem);
    const float *mo = reinterpret_cast<const float *>(smem) + 2 * NWC * G;
    for (int i = tid; i < G * HD; i += Cfg::THREADS) {
        const int g = i / HD, d = i % HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NWC; ++w) M = fmaxf(M, mm[w * G + g].x);
        float O = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < NWC; ++w) {
            const float2 ml = mm[w * G + g];
            const float wt = ex2(ml.x - M);                 // 0 for a warp that saw no rows
            O = fmaf(wt, mo[(w * G + g) * HD + d], O);
            L = fmaf(wt, ml.y, L);
        }
        const size_t slot = (head0 + g) * P + sp;
        a.ws_o[slot * HD + d] = O;
        if (d == 0) a.ws_ml[slot] = make_float2(M, L);
    }
}

} // namespace attn
