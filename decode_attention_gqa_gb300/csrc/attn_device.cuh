// attn_device.cuh -- device-side helpers shared by the decode-attention kernels:
// the argument block, the split rule, mbarriers with bounded waits, TMA tile
// loads, programmatic-dependent-launch controls and small math wrappers.
// sm_103a only (inline PTX for mbarrier, cp.async.bulk.tensor, griddepcontrol,
// redux.sync.f32, ex2.approx).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;

// Error bits, the same values as ATTN_DEVERR_* in include/attn_decode.h.
constexpr unsigned kErrPositionClamped = 0x1u;
constexpr unsigned kErrPipelineTimeout = 0x2u;

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// The host heuristic never makes a split shorter than this at full capacity.
constexpr int kSplitGranule = 16;

// ---------------------------------------------------------------------------
// Loads of inputs that the previous kernel in the stream may have written (q,
// positions, the appended rows, the partials). They go through L2 (.cg), the
// point of coherence, and are volatile with a memory clobber, so the compiler
// keeps them after griddepcontrol.wait. The read-only path (__ldg) is not
// used for these: its loads may be hoisted above the wait and may return
// lines cached before the other grid wrote them.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ld_dep(const float *p)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_dep(const int *p)
{
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float2 ld_dep(const float2 *p)
{
    float2 v;
    asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_dep(const float4 *p)
{
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint4 ld_dep(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
    return v;
}

struct PartialArgs {
    const float *q;           // [n_seq][n_head][HD] f32
    const uint16_t *k;        // [n_seq][cap][n_kv_head][HD] 16-bit elements (tail tiles read directly)
    const uint16_t *v;
    const int32_t *positions; // [n_seq]
    float *ws_o;              // [n_seq][n_head][P][HD]   unnormalised partial accumulators
    float2 *ws_ml;            // [n_seq][n_head][P]       (mx, S), mx in log2 units
    unsigned *err;            // sticky device error word
    int n_head;
    int n_kv_head;
    int n_splits;             // P
    int split_len;            // 0 = by count
    int64_t cap;              // cache rows per sequence
    float qscale;             // scale * log2(e): scores come out in log2 units
    int n_q;                  // query rows per sequence (1: decode; > 1: causal multi-query)
    int qgroups;              // blocks per (split, KV head) along the query heads
    // Fused append (optional): the new token's rows [n_seq][n_kv_head][HD],
    // written into cache row positions[s] and attended in the same launch.
    const uint16_t *k_new;    // null: no append
    const uint16_t *v_new;
    uint16_t *k_w;            // the caches again, writable, when appending
    uint16_t *v_w;
    int kv_stable;            // 1: positions and cache rows may be read before the grid dependency
    int group;                // G = n_head / n_kv_head
    unsigned group_magic;     // ceil(2^16 / G): x / G == (x * group_magic) >> 16 for 0 <= x < 8192
};

// x / G for a (query row, group head) index x < 8192 without an integer
// division (exact for every G in 1..8 over that range).
__device__ __forceinline__ int div_group(const PartialArgs &a, int x)
{
    return (int)(((unsigned)x * a.group_magic) >> 16);
}

struct CombineArgs {
    const float *ws_o;
    const float2 *ws_ml;
    float *out;               // [n_seq][n_head][HD]
    int n_head;
    int n_splits;
};

// ---------------------------------------------------------------------------
// a1: rows attended and the split's row range. nkv = positions[s] + 1 clamped
// to [0, cap] ("10 · R4" §2.2). By count: chunk = ceil(nkv / P) rounded up to
// kSplitGranule rows; by block (Red Lite dev35 "Change"): chunk = split_len.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int64_t rows_attended(const PartialArgs &a, int s, bool report,
                                                 bool *in_range = nullptr)
{
    int64_t n = (int64_t)ld_dep(a.positions + s) + 1;
    const bool ok = n >= 0 && n <= a.cap;
    if (!ok) {
        if (report) atomicOr(a.err, kErrPositionClamped);
        n = n < 0 ? 0 : a.cap;
    }
    if (in_range) *in_range = ok;
    return n;
}

// By count the chunk is rounded up to a whole number of the kernel's tiles
// (`tile` rows), so that only the last split of a sequence ends in a partial tile.
__device__ __forceinline__ void split_range(int64_t nkv, int sp, int n_splits, int split_len,
                                            int tile, int64_t &lo, int64_t &hi)
{
    int64_t chunk;
    if (split_len > 0) {
        chunk = split_len;
    } else {
        chunk = (nkv + n_splits - 1) / n_splits;
        chunk = (chunk + tile - 1) / tile * tile;
    }
    lo = (int64_t)sp * chunk;
    hi = lo + chunk < nkv ? lo + chunk : nkv;
}

// split_range for the one-tile kernel (tile rows per block, count mode): a
// chunk that would fill more than three quarters of a tile is rounded up to 16
// rows only, so that a split count sized for one block per SM balances the
// rows over the blocks (the 7b layer at full context on 256-row tiles: 38
// splits of 216 -> 224 rows on 152 SMs); shorter chunks are rounded up to whole
// tiles (few, full blocks for short contexts), or, on a wide tile (halves) while
// the context fits in four tiles, to half tiles, which that kernel runs on the
// tile's last half only (twice the blocks, each with half the chain).
__device__ __forceinline__ void split_range_tile(int64_t nkv, int sp, int n_splits, int split_len,
                                                 int tile, bool halves, int64_t &lo, int64_t &hi)
{
    if (split_len > 0) {
        split_range(nkv, sp, n_splits, split_len, tile, lo, hi);
        return;
    }
    int64_t chunk = (nkv + n_splits - 1) / n_splits;
    chunk = 4 * chunk > 3 * (int64_t)tile ? (chunk + 15) / 16 * 16
          : halves && nkv <= 4 * (int64_t)tile && 2 * chunk <= (int64_t)tile ? (int64_t)tile / 2
          : (chunk + tile - 1) / tile * tile;
    lo = (int64_t)sp * chunk;
    hi = lo + chunk < nkv ? lo + chunk : nkv;
}

// Row stride (floats) of a warp's published accumulators in the merge area:
// 8 floats of padding put the rows of consecutive heads 8 banks apart, so
// that the tensor-core fragments (lanes 4 apart hold the same dims of
// different heads) store without bank conflicts.
template <int HD> __host__ __device__ constexpr int merge_stride() { return HD + 8; }

// Warm L2 with [p, p + bytes) (p and bytes multiples of 16). A hint with no
// effect on what any load returns: L2 is coherent, so it may be issued before
// the data's producer has finished.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Shared-memory addresses and mbarriers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity)
{
    unsigned ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete. Gives up after
// kWaitLimitNs and returns false; never spins forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, unsigned parity,
                                                  unsigned long long limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------------------
// TMA: one 3-D tile (x = element within the row, y = KV head, z = cache row)
// into shared memory, completion counted on an mbarrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
           "r"(smem_u32(bar))
        : "memory");
}

// The same box into L2 only (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// TMA: one 4-D tile (x = element, y = KV head, z = row within the sequence,
// w = sequence). z may be negative: rows outside the tensor arrive as zeros.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z, int w)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w),
           "r"(smem_u32(bar))
        : "memory");
}

// The same 4-D box into L2 only (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *map, int x, int y, int z, int w)
{
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// cp.async (16 bytes, zero-filled when src_bytes == 0) with completion tracked
// by an mbarrier: the arrive below fires once every cp.async this thread has
// issued so far has landed, without changing the phase's expected count.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void *dst, const void *src, unsigned src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" :: "r"(smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core primitives (16x8x16 f16 MMA with f32 accumulation,
// 8x8 matrix loads from shared memory).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}

// D = A x B + D, 16x8x16, A and B of the cache element type KV (both operands
// always the same type), f32 accumulation.
template <typename KV>
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1)
{
    if constexpr (std::is_same<KV, __half>::value) {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                     "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                     "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// Two cache elements (one 32-bit word) to f32, and two f32 to a packed pair of
// cache elements (round to nearest even), for KV = __half or __nv_bfloat16.
template <typename KV>
__device__ __forceinline__ float2 kv2_to_float2(uint32_t w)
{
    if constexpr (std::is_same<KV, __half>::value)
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    else
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}

template <typename KV>
__device__ __forceinline__ uint32_t float2_to_kv2(float lo, float hi)
{
    if constexpr (std::is_same<KV, __half>::value) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

// ---------------------------------------------------------------------------
// Math.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Power-of-two scale for a row of q whose largest magnitude is amax >= 0:
// sc = 2^s brings amax into [2^14, 2^15) (amax in [2^(e-1), 2^e) gives
// s = 15 - e, read off the exponent field, no library call), and inv = 2^-s
// undoes it; both are exact. s is capped at 126 so that both stay normal
// floats (rows below 2^-113 then scale to less than 2^14, still far from the
// 16-bit types' limits); a zero row gets sc = inv = 1.
__device__ __forceinline__ void pow2_scale(float amax, float &sc, float &inv)
{
    const int E = (int)((__float_as_uint(amax) >> 23) & 0xFFu);   // biased exponent
    const int s = min(141 - E, 126);                              // 15 - e with e = E - 126
    sc = amax > 0.f ? __uint_as_float((unsigned)(127 + s) << 23) : 1.f;
    inv = amax > 0.f ? __uint_as_float((unsigned)(127 - s) << 23) : 1.f;
}

__device__ __forceinline__ float warp_max(float x)
{
    float y;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Eight cache elements (one 16-byte unit) to f32.
template <typename KV>
__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = kv2_to_float2<KV>(w[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// ---------------------------------------------------------------------------
// Shared-memory tile layout written by TMA. A tile of R rows x HD f16 is stored
// as HD/64 column chunks; chunk c is R rows of 128 bytes, with the 16-byte
// units of row r permuted by r & 7 (the 128-byte swizzle). head_dim 8 rows
// (16 bytes) are stored densely. Returns the byte offset of 16-byte unit U of
// row r.
// ---------------------------------------------------------------------------
template <int HD, int R>
__device__ __forceinline__ uint32_t tile_unit_offset(int r, int U)
{
    if constexpr (HD >= 64) {
        const int c = U >> 3, u = U & 7;
        return (uint32_t)(c * R * 128 + r * 128 + ((u ^ (r & 7)) << 4));
    } else {
        return (uint32_t)(r * (HD * 2) + U * 16);
    }
}

} // namespace attn
