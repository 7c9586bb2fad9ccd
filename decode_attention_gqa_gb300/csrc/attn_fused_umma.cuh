// attn_fused_umma.cuh -- partial and combine in one kernel (steps a1-a7):
// the tcgen05 tile arithmetic of attn_partial_umma.cuh, with all splits of a
// (sequence, KV head) in one thread-block cluster that merges them through
// distributed shared memory and writes o itself.
//
// Grid (16, n_kv_head, n_seq), cluster (16, 1, 1) (a launch attribute; 16 is a
// non-portable cluster size the host opts into): block sp of a cluster takes
// split sp of that (sequence hk, KV head) pair -- the static grid of minfer
// "10 · R4" §2.2 with the KV head in place of the query head and P = 16 --
// and its chunk ceil(nkv / 16) rounded up to whole 128-row tiles, at most 4
// (nkv <= 8192). Per block:
//   - a producer thread streams the tiles' K and V rows by TMA through rings
//     of three K and three V stages (the first three tiles before the grid
//     dependency when the caller allows it; the fourth into L2 at once and
//     into a stage when S of tile 0 (K) and Oᵀ of tile 0 (V) are done);
//   - one thread issues S_t = K_t · Qᵀ for every tile into its own tensor-memory
//     accumulator, another Oᵀ_t = V_tᵀ · P_t once P_t is written;
//   - two groups of four softmax warps take alternate tiles: each tile gets its
//     own block-wide maximum m_t, sum l_t and accumulator Oᵀ_t (§2.1 with one
//     step per tile, no rescaling);
//   - the first group folds the tiles (§3.2's rule within the block) into the
//     block's state (m_b, l_b, o_b) in shared memory;
//   - after a cluster barrier, block r folds head r / 2, half r % 2 of the
//     head dimensions, over the 16 blocks' states read from their shared
//     memory (§2.1: gmx = max m_b, weights 2^(m_b - gmx)), and writes o.
// The combine kernel and its launch disappear; a second cluster barrier keeps
// every block's shared memory alive until the others have read it.
#pragma once

#include "attn_partial_umma.cuh"

namespace attn {

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of the same variable in block `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void *p, int rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

template <int HD, int G, typename KV>
struct FusedCfg {
    static_assert(HD == 128, "the cluster-fused kernel is built for head_dim 128");
    static constexpr int CLUSTER = 16;                // splits per (sequence, KV head)
    static constexpr int TILE = 128;
    static constexpr int NT_MAX = 4;                  // tiles per block: nkv <= 16 * 4 * 128
    static constexpr int STAGES = 3;                  // K and V ring depth
    static constexpr int NCH = HD / 64;
    static constexpr int THREADS = 352;               // S warp, Oᵀ/TMEM warp, producer, 2 x 4 softmax warps
    using QStage = TcWarp<HD, G, 4, KV>;
    static constexpr uint32_t TILE_BYTES = (uint32_t)TILE * HD * 2;       // one of K or V
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = STAGES * TILE_BYTES;
    static constexpr uint32_t OFF_Q = 2 * STAGES * TILE_BYTES;
    static constexpr uint32_t OFF_P = (OFF_Q + QStage::EXTRA_BYTES + 127) / 128 * 128;
    static constexpr uint32_t P_BYTES = (uint32_t)TILE * 16 * 2;          // one tile's P
    static constexpr uint32_t OFF_RED = OFF_P + NT_MAX * P_BYTES;          // [tile][max | sum][4][8]
    static constexpr uint32_t OFF_BAR = OFF_RED + NT_MAX * 2 * 4 * 8 * 4;
    static constexpr int NBAR = 3 * 4 + 2 * NT_MAX + 1;                   // k/v full/empty, s_done, p_ready, o_done
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 1024;
    // the block state exchanged through the cluster, over the K ring once it is idle:
    // (m_b, l_b) per head, then o_b[head][HD]
    static constexpr uint32_t OFF_XCH = 0;
    static constexpr uint32_t TMEM_COLS = 128;        // S_t at 16t, Oᵀ_t at 64 + 16t
    static constexpr float OFF = 7.f;
    static_assert(OFF_Q % 1024 == 0 && OFF_V % 1024 == 0, "swizzled operands start 1024-aligned");
    static_assert((2 * 8 + 8 * HD) * 4 <= STAGES * TILE_BYTES, "exchange area fits the K ring");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

template <class Cfg, int HD, int G, typename KV>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
attn_fused_umma(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                const PartialArgs a, float *__restrict__ out)
{
    constexpr int TILE = Cfg::TILE, NS = Cfg::STAGES, NTM = Cfg::NT_MAX;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *kfull = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *vfull = kfull + NS, *kempty = vfull + NS, *vempty = kempty + NS;
    uint64_t *s_done = vempty + NS, *p_ready = s_done + NTM, *o_done = p_ready + NTM;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(o_done + 1);
    volatile int *flags = reinterpret_cast<volatile int *>(tslot + 1);    // [0] abort
    float *red = reinterpret_cast<float *>(smem + Cfg::OFF_RED);
    float *xch = reinterpret_cast<float *>(smem + Cfg::OFF_XCH);          // [m_b x8][l_b x8][o_b 8 x HD]

    const int sp = blockIdx.x, hk = blockIdx.y, s = blockIdx.z;           // sp = rank in the cluster
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool stable = a.kv_stable != 0;
    if (tid == 0)
        prefetch_l2(a.q + ((size_t)s * a.n_head + (size_t)hk * G) * HD, (uint32_t)(G * HD * sizeof(float)));
    if (!stable) pdl_wait();
    pdl_launch_dependents();

    // a1: this block's rows: chunks of whole tiles, tile t the rows from lo + 128t
    // (the last one the 128 rows that end at hi)
    bool pos_ok;
    const int64_t nkv = rows_attended(a, s, sp == 0 && hk == 0 && tid == 0, &pos_ok);
    int64_t lo, hi;
    split_range(nkv, sp, Cfg::CLUSTER, 0, TILE, lo, hi);
    // (the host keeps nkv <= 16 * 4 * 128; the bound only guards the tile arrays)
    int NT = lo < hi ? (int)((hi - lo + TILE - 1) / TILE) : 0;
    if (NT > NTM) NT = NTM;
    auto box_first = [&](int t) -> int { return t < NT - 1 ? (int)(lo + (int64_t)t * TILE) : (int)(hi - TILE); };

    if (warp == 2 && lane == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(kfull + i, 1);
            mbar_init(vfull + i, 1);
            mbar_init(kempty + i, 1);
            mbar_init(vempty + i, 1);
        }
        for (int t = 0; t < NTM; ++t) {
            mbar_init(s_done + t, 1);
            mbar_init(p_ready + t, 128);
        }
        mbar_init(o_done, 1);
        flags[0] = 0;
        fence_barrier_init();
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        for (int t = 0; t < NT && t < NS; ++t) {
            const int z = box_first(t);
            mbar_arrive_expect_tx(kfull + t, Cfg::TILE_BYTES);
            mbar_arrive_expect_tx(vfull + t, Cfg::TILE_BYTES);
#pragma unroll
            for (int c = 0; c < Cfg::NCH; ++c) {
                tma_load_4d(smem + Cfg::OFF_K + t * Cfg::TILE_BYTES + c * (Cfg::TILE_BYTES / Cfg::NCH), &kmap,
                            kfull + t, c * 64, hk, z, s);
                tma_load_4d(smem + Cfg::OFF_V + t * Cfg::TILE_BYTES + c * (Cfg::TILE_BYTES / Cfg::NCH), &vmap,
                            vfull + t, c * 64, hk, z, s);
            }
        }
        for (int t = NS; t < NT; ++t)
#pragma unroll
            for (int c = 0; c < Cfg::NCH; ++c) {
                tma_prefetch_4d(&kmap, c * 64, hk, box_first(t), s);
                tma_prefetch_4d(&vmap, c * 64, hk, box_first(t), s);
            }
    }
    if (warp == 1) tmem_alloc(tslot, Cfg::TMEM_COLS);
    if (stable) pdl_wait();
    Cfg::QStage::template prepare<Cfg::THREADS>(smem + Cfg::OFF_Q, a, s, hk, 0, tid);
    // Fused append: the block whose split ends at nkv holds the new row nkv - 1 as
    // row TILE - 1 of its last tile. Lanes 0-15 of warp 0 fetch the new K row and
    // write it into that tile before its S; lanes 0-15 of warp 1 do the same for
    // V before its Oᵀ; both also write it into the cache.
    constexpr int NU = HD / 8;
    static_assert(NU <= 32, "one unit of the new row per lane");
    const bool appending = a.k_new != nullptr && pos_ok && hi == nkv && NT > 0 && warp < 2 && lane < NU;
    uint4 newrow = make_uint4(0u, 0u, 0u, 0u);
    const size_t new_dst = ((size_t)((int64_t)s * a.cap + nkv - 1) * a.n_kv_head + hk) * HD;
    if (appending)
        newrow = ld_dep(reinterpret_cast<const uint4 *>((warp == 0 ? a.k_new : a.v_new) +
                                                        ((size_t)s * a.n_kv_head + hk) * HD) + lane);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tslot;

    auto fail = [&]() { flags[0] = 1; atomicOr(a.err, kErrPipelineTimeout); };
    if (warp == 0) {
        // ---------------- S_t = K_t · Qᵀ ----------------
        const uint32_t sq = smem_u32(smem + Cfg::OFF_Q);
        constexpr uint32_t id_s = umma_idesc<KV>(TILE, 16, 0, 0);
        for (int t = 0; t < NT; ++t) {
            const bool landed = mbar_wait_bounded(kfull + t % NS, (t / NS) & 1);
            if (!__all_sync(0xffffffffu, landed)) { if (lane == 0) fail(); break; }
            uint8_t *kst = smem + Cfg::OFF_K + (t % NS) * Cfg::TILE_BYTES;
            if (t == NT - 1 && a.k_new != nullptr && pos_ok && hi == nkv) {
                if (lane < NU) {
                    *reinterpret_cast<uint4 *>(kst + tile_unit_offset<HD, TILE>(TILE - 1, lane)) = newrow;
                    reinterpret_cast<uint4 *>(a.k_w + new_dst)[lane] = newrow;
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                tc_fence_after();
                const uint32_t sk = smem_u32(kst);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t ok = (kk >> 2) * (TILE * 128) + (kk & 3) * 32;
                    const uint32_t oq = (kk >> 2) * (16 * 128) + (kk & 3) * 32;
                    umma_f16(tm + 16 * t, umma_desc(sk + ok, 16, 1024, 2), umma_desc(sq + oq, 16, 1024, 2),
                             id_s, kk > 0);
                }
                umma_commit(kempty + t % NS);
                umma_commit(s_done + t);
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        // ---------------- Oᵀ_t = V_tᵀ · P_t ----------------
        if (NT > 0) {
            constexpr uint32_t id_o = umma_idesc<KV>(128, 16, 1, 1);
            bool all_ok = true;
            for (int t = 0; t < NT; ++t) {
                const bool ready = mbar_wait_bounded(p_ready + t, 0) && mbar_wait_bounded(vfull + t % NS, (t / NS) & 1);
                if (!__all_sync(0xffffffffu, ready)) { if (lane == 0) fail(); all_ok = false; break; }
                uint8_t *vst = smem + Cfg::OFF_V + (t % NS) * Cfg::TILE_BYTES;
                if (t == NT - 1 && a.k_new != nullptr && pos_ok && hi == nkv) {
                    if (lane < NU) {
                        *reinterpret_cast<uint4 *>(vst + tile_unit_offset<HD, TILE>(TILE - 1, lane)) = newrow;
                        reinterpret_cast<uint4 *>(a.v_w + new_dst)[lane] = newrow;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (lane == 0) {
                    tc_fence_after();
                    const uint32_t sv = smem_u32(vst);
                    const uint32_t spp = smem_u32(smem + Cfg::OFF_P + t * Cfg::P_BYTES);
#pragma unroll
                    for (int kk = 0; kk < TILE / 16; ++kk)
                        umma_f16(tm + 64 + 16 * t, umma_desc(sv + kk * 2048, TILE * 128, 1024, 2),
                                 umma_desc(spp + kk * 512, 256, 128, 0), id_o, kk > 0);
                    umma_commit(vempty + t % NS);
                }
                __syncwarp();
            }
            if (lane == 0 && all_ok) umma_commit(o_done);
        }
    } else if (warp == 2) {
        // ---------------- producer: tiles past the ring ----------------
        if (lane == 0) {
            for (int t = NS; t < NT; ++t) {
                const int st = t % NS, ph = ((t / NS) - 1) & 1;
                const int z = box_first(t);
                if (!mbar_wait_bounded(kempty + st, ph)) { fail(); break; }
                mbar_arrive_expect_tx(kfull + st, Cfg::TILE_BYTES);
#pragma unroll
                for (int c = 0; c < Cfg::NCH; ++c)
                    tma_load_4d(smem + Cfg::OFF_K + st * Cfg::TILE_BYTES + c * (Cfg::TILE_BYTES / Cfg::NCH), &kmap,
                                kfull + st, c * 64, hk, z, s);
                if (!mbar_wait_bounded(vempty + st, ph)) { fail(); break; }
                mbar_arrive_expect_tx(vfull + st, Cfg::TILE_BYTES);
#pragma unroll
                for (int c = 0; c < Cfg::NCH; ++c)
                    tma_load_4d(smem + Cfg::OFF_V + st * Cfg::TILE_BYTES + c * (Cfg::TILE_BYTES / Cfg::NCH), &vmap,
                                vfull + st, c * 64, hk, z, s);
            }
        }
    } else {
        // ---------------- softmax groups: tiles gi, gi + 2 ----------------
        const int gi = (warp - 3) >> 2;                // 0: warps 3-6, 1: warps 7-10
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;                  // tile row
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const float *inv = reinterpret_cast<const float *>(smem + Cfg::OFF_Q + Cfg::QStage::QT_BYTES);
        for (int t = gi; t < NT; t += 2) {
            float *rmax = red + t * 64, *rsum = rmax + 32;
            const bool sd = mbar_wait_bounded(s_done + t, 0);
            const bool ok = __all_sync(0xffffffffu, sd) && !flags[0];
            if (!sd && lane == 0) fail();
            float sc[G];
            if (ok) {
                tc_fence_after();
                float c[16];
                tmem_ld16(tm + 16 * t + lane_base, c);
                const int64_t first = lo + (int64_t)t * TILE;
                const bool valid = (int64_t)box_first(t) + r >= first;
#pragma unroll
                for (int g = 0; g < G; ++g) sc[g] = valid ? (c[g] + c[8 + g]) * inv[g] : -INFINITY;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float m = warp_max(sc[g]);
                    if (lane == 0) rmax[q4 * 8 + g] = m;
                }
            }
            asm volatile("bar.sync %0, 128;" :: "r"(1 + gi) : "memory");
            float p[8];
            if (ok) {
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    if (g < G) {
                        const float M = fmaxf(fmaxf(rmax[g], rmax[8 + g]), fmaxf(rmax[16 + g], rmax[24 + g]));
                        p[g] = ex2(sc[g] - (M - Cfg::OFF));
                    } else {
                        p[g] = 0.f;
                    }
                }
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    hw[j] = float2_to_kv2<KV>(p[2 * j], p[2 * j + 1]);
                    const float2 f = kv2_to_float2<KV>(hw[j]);
                    lw[j] = float2_to_kv2<KV>(p[2 * j] - f.x, p[2 * j + 1] - f.y);
                }
                uint8_t *pt = smem + Cfg::OFF_P + t * Cfg::P_BYTES;
                *reinterpret_cast<uint4 *>(pt + p_offset<16>(r, 0)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(pt + p_offset<16>(r, 8)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                fence_proxy_async_smem();
            }
            mbar_arrive(p_ready + t);
            if (ok) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float l = warp_sum(p[g]);
                    if (lane == 0) rsum[q4 * 8 + g] = l;
                }
            }
        }
        // both groups' per-tile maxima and sums are in shared memory past this barrier
        asm volatile("bar.sync 3, 256;" ::: "memory");
        if (gi == 0) {
            // a6 within the block: fold the tiles into (m_b, l_b, o_b); thread r = dimension r
            float acc[G], Lb[G], Mb[G];
#pragma unroll
            for (int g = 0; g < G; ++g) { acc[g] = 0.f; Lb[g] = 0.f; Mb[g] = -INFINITY; }
            bool ok = !flags[0];
            if (NT > 0 && ok) {
                const bool od = mbar_wait_bounded(o_done, 0);
                ok = __all_sync(0xffffffffu, od);
                if (!od && lane == 0) fail();
            }
            if (NT > 0 && ok) {
                tc_fence_after();
                float Mt[NTM][G];
#pragma unroll
                for (int t = 0; t < NTM; ++t)
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float *rm = red + t * 64;
                        Mt[t][g] = t < NT ? fmaxf(fmaxf(rm[g], rm[8 + g]), fmaxf(rm[16 + g], rm[24 + g])) : -INFINITY;
                        Mb[g] = fmaxf(Mb[g], Mt[t][g]);
                    }
#pragma unroll
                for (int t = 0; t < NTM; ++t) {
                    if (t < NT) {
                        float c[16];
                        tmem_ld16(tm + 64 + 16 * t + lane_base, c);
                        const float *rs = red + t * 64 + 32;
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float w = ex2(Mt[t][g] - Mb[g]);
                            acc[g] = fmaf(w, c[g] + c[8 + g], acc[g]);
                            Lb[g] = fmaf(w, (rs[g] + rs[8 + g]) + (rs[16 + g] + rs[24 + g]), Lb[g]);
                        }
                    }
                }
            }
            // m_b in the partial convention (the reference the p's were taken against)
#pragma unroll
            for (int g = 0; g < G; ++g) {
                xch[16 + g * HD + r] = acc[g];
                if (r == g) {
                    xch[g] = Mb[g] == -INFINITY ? -INFINITY : Mb[g] - Cfg::OFF;
                    xch[8 + g] = Lb[g];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();

    // a7 across the cluster: block sp folds head sp / 2, dimensions (sp % 2) * 64 .. + 64
    {
        const int g = sp >> 1, d = (sp & 1) * 64 + tid;
        if (g < G && tid < 64) {
            float mb[Cfg::CLUSTER], lb[Cfg::CLUSTER], ob[Cfg::CLUSTER];
#pragma unroll
            for (int b = 0; b < Cfg::CLUSTER; ++b) {
                mb[b] = ld_cluster_f32(cluster_map(xch + g, b));
                lb[b] = ld_cluster_f32(cluster_map(xch + 8 + g, b));
                ob[b] = ld_cluster_f32(cluster_map(xch + 16 + g * HD + d, b));
            }
            float M = -INFINITY;
#pragma unroll
            for (int b = 0; b < Cfg::CLUSTER; ++b) M = fmaxf(M, mb[b]);
            float num = 0.f, den = 0.f;
#pragma unroll
            for (int b = 0; b < Cfg::CLUSTER; ++b) {
                const float w = mb[b] == -INFINITY ? 0.f : ex2(mb[b] - M);
                num = fmaf(w, ob[b], num);
                den = fmaf(w, lb[b], den);
            }
            out[((size_t)s * a.n_head + (size_t)hk * G + g) * HD + d] = den > 0.f ? num / den : 0.f;
        }
    }
    // no block may leave while another still reads its shared memory; then,
    // after an abort, wait (bounded) for this block's copies and MMAs
    cluster_sync_all();
    if (flags[0] && tid == 64) {
        for (int i = 0; i < NS; ++i) {
            (void)mbar_wait_bounded(kfull + i, 0, 1000000ull);
            (void)mbar_wait_bounded(vfull + i, 0, 1000000ull);
        }
        (void)mbar_wait_bounded(o_done, 0, 1000000ull);
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tm, Cfg::TMEM_COLS);
}

} // namespace attn
