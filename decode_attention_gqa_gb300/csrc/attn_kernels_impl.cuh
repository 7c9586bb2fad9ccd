// attn_kernels_impl.cuh -- kernel instantiation and launch per (head_dim,
// cache element type). Each attn_kernels_hd<N>_<type>.cu includes this once
// with its own pair, so the instantiations compile in parallel.
#pragma once

#include "attn_combine.cuh"
#include "attn_launch.h"
#include "attn_partial.cuh"
#include "attn_partial_umma.cuh"
#include "attn_fused_umma.cuh"
#include "attn_partial_tile.cuh"

namespace attn {

// Pipeline shape per (policy, head_dim): compute warps and stages, sized so
// the stage ring fits the 227 KB shared-memory budget with enough bytes in
// flight per SM (about two stages ahead of the compute warps).
// MINB is the number of resident blocks per SM the register budget is sized
// for (the shared memory must allow as many).
template <int HD> struct SimtShape;
template <> struct SimtShape<8>   { static constexpr int NWC = 4, S = 4, MINB = 1; };
template <> struct SimtShape<64>  { static constexpr int NWC = 4, S = 3, MINB = 1; };
template <> struct SimtShape<128> { static constexpr int NWC = 4, S = 3, MINB = 1; };
template <> struct SimtShape<256> { static constexpr int NWC = 2, S = 3, MINB = 1; };

template <int HD> struct TcShape  { static constexpr int NWC = 4, S = 3, MINB = 2; };
template <> struct TcShape<64>    { static constexpr int NWC = 4, S = 4, MINB = 2; };
template <> struct TcShape<256>   { static constexpr int NWC = 4, S = 3, MINB = 1; };

// Multi-query tensor-core blocks: 16 query heads each.
template <int HD> struct TcMqShape { static constexpr int NWC = 4, S = 3, MINB = 2; };
template <> struct TcMqShape<256>  { static constexpr int NWC = 4, S = 3, MINB = 1; };
constexpr int kMqHeads = 16;

template <int HD, int G, typename KV>
using SimtCfg = PartialCfg<HD, G, SimtWarp, SimtShape<HD>::NWC, SimtShape<HD>::S, SimtShape<HD>::MINB, KV>;
template <int HD, int G, typename KV>
using TcCfg = PartialCfg<HD, G, TcWarp, TcShape<HD>::NWC, TcShape<HD>::S, TcShape<HD>::MINB, KV>;

template <int HD, typename KV>
using TcMqCfg = PartialCfg<HD, kMqHeads, TcWarpMQ, TcMqShape<HD>::NWC, TcMqShape<HD>::S,
                           TcMqShape<HD>::MINB, KV>;

template <typename KV> constexpr int kv_dtype_code() { return std::is_same<KV, __half>::value ? kKvF16 : kKvBf16; }

// Resident blocks per SM for a configuration: 228 KB of shared memory per SM
// with 1 KB reserved per block, 64 K registers, at most 32 blocks.
template <class Cfg>
constexpr int blocks_per_sm()
{
    const int by_smem = (int)(233472u / (Cfg::SMEM_BYTES + 1024u));
    return by_smem < 1 ? 1 : (by_smem > 32 ? 32 : by_smem);
}

template <class Cfg, int HD, int G, typename KV>
cudaError_t launch_partial(const LaunchRequest &r)
{
    alignas(64) CUtensorMap kmap, vmap;
    const int64_t rows = (int64_t)r.n_seq * r.pa.cap;
    const int dt = kv_dtype_code<KV>();
    cudaError_t e = encode_kv_map(&kmap, r.k_cache, rows, r.pa.n_kv_head, HD, Cfg::BOX_X, Cfg::TILE, dt);
    if (e != cudaSuccess) return e;
    e = encode_kv_map(&vmap, r.v_cache, rows, r.pa.n_kv_head, HD, Cfg::BOX_X, Cfg::TILE, dt);
    if (e != cudaSuccess) return e;
    const void *fn = reinterpret_cast<const void *>(&attn_split_partial<Cfg, HD, G>);
    e = ensure_smem_attr(fn, (int)Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    PartialArgs pa = r.pa;
    void *args[] = {&kmap, &vmap, &pa};
    return launch_pdl(fn, dim3(pa.n_kv_head * pa.qgroups, pa.n_splits, r.n_seq), dim3(Cfg::THREADS),
                      Cfg::SMEM_BYTES, r.stream, args);
}

// The tcgen05 kernel: one block per (KV head x query group, split, sequence),
// one 128-row tile each; MQ: several causal query rows, 16 slots per block.
template <int HD, int G, typename KV, bool MQ = false>
cudaError_t launch_partial_umma(const LaunchRequest &r)
{
    using C = UmmaCfg<HD, G, KV, MQ>;
    alignas(64) CUtensorMap kmap, vmap;
    const int dt = kv_dtype_code<KV>();
    cudaError_t e = encode_kv_map4(&kmap, r.k_cache, r.n_seq, r.pa.cap, r.pa.n_kv_head, HD, 64, C::TILE, dt);
    if (e != cudaSuccess) return e;
    e = encode_kv_map4(&vmap, r.v_cache, r.n_seq, r.pa.cap, r.pa.n_kv_head, HD, 64, C::TILE, dt);
    if (e != cudaSuccess) return e;
    const void *fn = reinterpret_cast<const void *>(&attn_split_partial_umma<C, HD, G, KV>);
    e = ensure_smem_attr(fn, (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    PartialArgs pa = r.pa;
    void *args[] = {&kmap, &vmap, &pa};
    return launch_pdl(fn, dim3(pa.n_kv_head * pa.qgroups, pa.n_splits, r.n_seq), dim3(C::THREADS),
                      C::SMEM_BYTES, r.stream, args);
}

// The one-tile mma.sync kernel: one block per (KV head, split, sequence), one
// tile of TileCfg::TILE rows each, one query row (WIDE: 128-row tiles at
// head_dim 256).
template <int HD, int G, typename KV, bool WIDE = false>
cudaError_t launch_partial_tile(const LaunchRequest &r)
{
    using C = TileCfg<HD, G, KV, false, WIDE>;
    alignas(64) CUtensorMap kmap, vmap;
    const int dt = kv_dtype_code<KV>();
    cudaError_t e = encode_kv_map4(&kmap, r.k_cache, r.n_seq, r.pa.cap, r.pa.n_kv_head, HD, 64, C::TILE, dt);
    if (e != cudaSuccess) return e;
    e = encode_kv_map4(&vmap, r.v_cache, r.n_seq, r.pa.cap, r.pa.n_kv_head, HD, 64, C::TILE, dt);
    if (e != cudaSuccess) return e;
    // by block length with blk dividing the tile: one block per SPB = TILE / blk splits
    const int blk = r.pa.split_len;
    const void *fn = reinterpret_cast<const void *>(&attn_split_partial_tile<C, HD, G, KV>);
    bool ms = false;
    if constexpr (!WIDE) {              // the wide tile takes splits longer than 96 rows only
        ms = tile_serves_splits(C::TILE, blk);
        if (ms) fn = reinterpret_cast<const void *>(&attn_split_partial_tile_ms<C, HD, G, KV>);
    }
    e = ensure_smem_attr(fn, (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    PartialArgs pa = r.pa;
    void *args[] = {&kmap, &vmap, &pa};
    const int spb = ms ? C::TILE / blk : 1;
    return launch_pdl(fn, dim3(pa.n_kv_head, (pa.n_splits + spb - 1) / spb, r.n_seq), dim3(C::THREADS),
                      C::SMEM_BYTES, r.stream, args);
}

// The one-tile mma.sync kernel for several causal query rows: 16 (row, head)
// slots per block, grid (KV head x query group, split, sequence); WIDE:
// 256-row tiles, one block per SM.
template <int HD, typename KV, bool WIDE = false>
cudaError_t launch_partial_tile_mq(const LaunchRequest &r)
{
    using C = TileCfg<HD, kMqHeads, KV, true, WIDE>;
    alignas(64) CUtensorMap kmap, vmap;
    const int dt = kv_dtype_code<KV>();
    cudaError_t e = encode_kv_map4(&kmap, r.k_cache, r.n_seq, r.pa.cap, r.pa.n_kv_head, HD, 64, C::TILE, dt);
    if (e != cudaSuccess) return e;
    e = encode_kv_map4(&vmap, r.v_cache, r.n_seq, r.pa.cap, r.pa.n_kv_head, HD, 64, C::TILE, dt);
    if (e != cudaSuccess) return e;
    const void *fn = reinterpret_cast<const void *>(&attn_split_partial_tile_mq<C, HD, KV>);
    e = ensure_smem_attr(fn, (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    PartialArgs pa = r.pa;
    void *args[] = {&kmap, &vmap, &pa};
    return launch_pdl(fn, dim3(pa.n_kv_head * pa.qgroups, pa.n_splits, r.n_seq), dim3(C::THREADS),
                      C::SMEM_BYTES, r.stream, args);
}

// The cluster-fused tcgen05 kernel: partial and combine in one launch, o written directly.
template <int HD, int G, typename KV>
cudaError_t launch_fused_umma(const LaunchRequest &r)
{
    using C = FusedCfg<HD, G, KV>;
    alignas(64) CUtensorMap kmap, vmap;
    const int dt = kv_dtype_code<KV>();
    cudaError_t e = encode_kv_map4(&kmap, r.k_cache, r.n_seq, r.pa.cap, r.pa.n_kv_head, HD, 64, C::TILE, dt);
    if (e != cudaSuccess) return e;
    e = encode_kv_map4(&vmap, r.v_cache, r.n_seq, r.pa.cap, r.pa.n_kv_head, HD, 64, C::TILE, dt);
    if (e != cudaSuccess) return e;
    const void *fn = reinterpret_cast<const void *>(&attn_fused_umma<C, HD, G, KV>);
    e = ensure_smem_attr(fn, (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    PartialArgs pa = r.pa;
    float *o = r.out;
    void *args[] = {&kmap, &vmap, &pa, &o};
    return launch_pdl_cluster(fn, dim3(C::CLUSTER, pa.n_kv_head, r.n_seq), dim3(C::THREADS), C::SMEM_BYTES,
                              r.stream, args, C::CLUSTER);
}

// Whether the current device can hold a cluster of the fused kernel (16 blocks
// of one SM each). Host only; takes no library lock.
template <int HD>
bool fused_cluster_fits()
{
    if constexpr (HD == 128) {
        using C = FusedCfg<HD, 8, __half>;
        const void *fn = reinterpret_cast<const void *>(&attn_fused_umma<C, HD, 8, __half>);
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        return cluster_slots(fn, dim3(C::THREADS), C::SMEM_BYTES, C::CLUSTER) > 0;
    } else {
        return false;
    }
}

template <int HD>
cudaError_t launch_combine(const LaunchRequest &r)
{
    CombineArgs ca;
    ca.ws_o = r.pa.ws_o;
    ca.ws_ml = r.pa.ws_ml;
    ca.out = r.out;
    ca.n_head = r.pa.n_head * (r.pa.n_q > 0 ? r.pa.n_q : 1);   // partial heads per sequence
    ca.n_splits = r.pa.n_splits;
    // the smallest batch that puts every split of a lane group in one round of loads
    const int ng = CombineCfg<HD>::NG;
    const void *fn = ca.n_splits <= ng * 8    ? reinterpret_cast<const void *>(&attn_combine<HD, 8>)
                     : ca.n_splits <= ng * 16 ? reinterpret_cast<const void *>(&attn_combine<HD, 16>)
                                              : reinterpret_cast<const void *>(&attn_combine<HD, 24>);
    const cudaError_t e = ensure_smem_attr(fn, 0);
    if (e != cudaSuccess) return e;
    void *args[] = {&ca};
    return launch_pdl(fn, dim3(ca.n_head, r.n_seq, CombineCfg<HD>::NCHUNK),
                      dim3(CombineCfg<HD>::THREADS), 0, r.stream, args);
}

template <int HD, int G, typename KV>
cudaError_t launch_group(const LaunchRequest &r)
{
    cudaError_t e = cudaSuccess;
    if (r.stages & kStagePartial) {
        if constexpr (HD % 16 == 0) {
            if (r.variant == kVariantFused) {
                // partial and combine in one launch
                if constexpr (HD == 128) return launch_fused_umma<HD, G, KV>(r);
                else return cudaErrorInvalidValue;
            } else if (r.variant == kVariantUmma) {
                if constexpr (HD == 128 || HD == 256) e = launch_partial_umma<HD, G, KV>(r);
                else return cudaErrorInvalidValue;
            } else if (r.variant == kVariantTile) {
                if constexpr (HD == 128 || HD == 256) e = launch_partial_tile<HD, G, KV>(r);
                else return cudaErrorInvalidValue;
            } else if (r.variant == kVariantTileWide) {
                if constexpr (HD == 128 || HD == 256) e = launch_partial_tile<HD, G, KV, true>(r);
                else return cudaErrorInvalidValue;
            } else if (r.variant == kVariantTc) {
                e = launch_partial<TcCfg<HD, G, KV>, HD, G, KV>(r);
            } else {
                e = launch_partial<SimtCfg<HD, G, KV>, HD, G, KV>(r);
            }
        } else {
            if (r.variant != kVariantSimt) return cudaErrorInvalidValue;
            e = launch_partial<SimtCfg<HD, G, KV>, HD, G, KV>(r);
        }
        if (e != cudaSuccess) return e;
    }
    if (r.stages & kStageCombine) e = launch_combine<HD>(r);
    return e;
}

template <int HD, typename KV>
cudaError_t launch_for_hd(const LaunchRequest &r)
{
    if (r.pa.n_q > 1) {                     // several causal query rows: tensor cores only
        if constexpr (HD % 16 == 0) {
            cudaError_t e = cudaSuccess;
            if (r.stages & kStagePartial) {
                if (r.variant == kVariantUmma) {
                    if constexpr (HD == 128 || HD == 256) e = launch_partial_umma<HD, kMqHeads, KV, true>(r);
                    else return cudaErrorInvalidValue;
                } else if (r.variant == kVariantTile) {
                    if constexpr (HD == 128) e = launch_partial_tile_mq<HD, KV>(r);
                    else return cudaErrorInvalidValue;
                } else if (r.variant == kVariantTileWide) {
                    if constexpr (HD == 128) e = launch_partial_tile_mq<HD, KV, true>(r);
                    else return cudaErrorInvalidValue;
                } else {
                    e = launch_partial<TcMqCfg<HD, KV>, HD, kMqHeads, KV>(r);
                }
                if (e != cudaSuccess) return e;
            }
            if (r.stages & kStageCombine) e = launch_combine<HD>(r);
            return e;
        } else {
            return cudaErrorInvalidValue;
        }
    }
    switch (r.group) {
    case 1: return launch_group<HD, 1, KV>(r);
    case 2: return launch_group<HD, 2, KV>(r);
    case 3: return launch_group<HD, 3, KV>(r);
    case 4: return launch_group<HD, 4, KV>(r);
    case 5: return launch_group<HD, 5, KV>(r);
    case 6: return launch_group<HD, 6, KV>(r);
    case 7: return launch_group<HD, 7, KV>(r);
    case 8: return launch_group<HD, 8, KV>(r);
    default: return cudaErrorInvalidValue;
    }
}

template <int HD>
KernelInfo kernel_info_for_hd(int group, int variant, bool multi)
{
    KernelInfo k{0, 0, 0, false, 0, 0};
    if (group < 1 || group > 8) return k;
    if (variant == kVariantFused) {
        if constexpr (HD == 128) {
            if (multi) return k;
            using C = FusedCfg<HD, 8, __half>;
            k.tile_rows = C::TILE;
            k.granule = C::TILE;
            k.stages = C::STAGES;
            k.blocks_per_sm = 1;
            k.max_chunk = C::TILE * C::NT_MAX;
            k.available = true;
        }
        return k;
    }
    if (variant == kVariantUmma) {
        if constexpr (HD == 128 || HD == 256) {
            // one query row (the largest group sets the shared-memory need) or 16 slots
            const uint32_t smem = multi ? UmmaCfg<HD, kMqHeads, __half, true>::SMEM_BYTES
                                        : UmmaCfg<HD, 8, __half>::SMEM_BYTES;
            using C = UmmaCfg<HD, 8, __half>;     // tile and granule are the same for both
            k.tile_rows = C::TILE;
            k.granule = C::GRANULE;
            k.stages = 1;
            k.blocks_per_sm = (int)(233472u / (smem + 1024u));
            k.max_chunk = C::TILE;
            k.available = true;
        }
        return k;
    }
    if (variant == kVariantTile) {
        if constexpr (HD == 128 || HD == 256) {
            if (multi && HD != 128) return k;   // several query rows: head_dim 128 only
            using C = TileCfg<HD, 8, __half>;   // the shapes do not depend on the group
            k.tile_rows = C::TILE;
            k.granule = C::GRANULE;
            k.stages = 1;
            const uint32_t smem = multi ? TileCfg<128, kMqHeads, __half, true>::SMEM_BYTES : C::SMEM_BYTES;
            k.blocks_per_sm = (int)(233472u / (smem + 1024u));
            k.max_chunk = C::TILE;
            // balanced counts measured slower here: two query rows 7.61 -> 7.72 us; one row
            // 5.89 -> 5.75 us at full context but 4.40 -> 4.72 / 3.67 -> 3.86 / 3.59 -> 3.74 us
            // at contexts 2048 / 512 / 128 of the same capacity (more splits, all empty there)
            k.balanced = false;
            k.available = true;
        }
        return k;
    }
    if (variant == kVariantTileWide) {
        if constexpr (HD == 128 || HD == 256) {
            if (multi && HD != 128) return k;   // several query rows: head_dim 128 only
            using C = TileCfg<HD, 8, __half, false, true>;
            k.tile_rows = C::TILE;
            k.granule = C::GRANULE;
            k.stages = 1;
            const uint32_t smem = multi ? TileCfg<128, kMqHeads, __half, true, true>::SMEM_BYTES : C::SMEM_BYTES;
            k.blocks_per_sm = (int)(233472u / (smem + 1024u));
            k.max_chunk = C::TILE;
            k.balanced = true;
            k.available = true;
        }
        return k;
    }
    if (variant == kVariantSimt) {
        if (multi) return k;
        using C = SimtCfg<HD, 8, __half>;   // the largest group sets the shared-memory need
        k.tile_rows = C::TILE;
        k.granule = C::GRANULE;
        k.stages = C::S;
        k.blocks_per_sm = blocks_per_sm<C>();
        k.available = true;
    } else if (variant == kVariantTc) {
        if constexpr (HD % 16 == 0) {
            if (multi) {
                using C = TcMqCfg<HD, __half>;
                k.tile_rows = C::TILE;
                k.granule = C::GRANULE;
                k.stages = C::S;
                k.blocks_per_sm = blocks_per_sm<C>();
            } else {
                using C = TcCfg<HD, 8, __half>;
                k.tile_rows = C::TILE;
                k.granule = C::GRANULE;
                k.stages = C::S;
                k.blocks_per_sm = blocks_per_sm<C>();
            }
            k.available = true;
        }
    }
    return k;
}

} // namespace attn
