// attn_api.cu -- the C ABI of include/attn_decode.h: argument validation, the
// split-count heuristic, workspace sizing and ownership, tensor-map encoding,
// the device error word, and dispatch to the per-head_dim kernel units.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <set>
#include <utility>

#include "attn_decode.h"
#include "attn_launch.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 4096;                  // combine keeps P weights in shared memory
constexpr int64_t kMaxFlatRows = (int64_t)1 << 31; // TMA row coordinates are int32
constexpr int64_t kUnknownCap = kMaxFlatRows - 1024;
constexpr int kFusedSplits = 16;                   // blocks per cluster of the fused tcgen05 kernel
constexpr int kStableTiles = 4;                    // "short call": <= 4 tiles per block at one per SM

thread_local int t_last_cuda_error = 0;

std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::set<std::pair<const void *, int>> g_smem_done;

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    unsigned *err_word = nullptr;                 // device address of g_attn_error_word
    void *ws = nullptr;                           // library-owned workspace
    size_t ws_bytes = 0;
    int fused_ok = -1;                            // the device holds a fused kernel's cluster (-1: not asked yet)
};
DeviceState g_dev[kMaxDevices];

} // namespace

// One sticky error word per device, set by the kernels with atomicOr.
__device__ unsigned g_attn_error_word;

// Self-test of the bounded wait: one warp waits on an mbarrier that nothing
// arrives on, through the same helper the kernels use, and reports the
// timeout in the error word as they do.
__global__ void attn_selftest_wait_kernel(unsigned *err, unsigned long long limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        attn::mbar_init(&bar, 1);
        attn::fence_barrier_init();
    }
    __syncthreads();
    const bool landed = attn::mbar_wait_bounded(&bar, 0, limit_ns);   // phase 0 never completes
    if (!__all_sync(0xffffffffu, landed) && threadIdx.x == 0) atomicOr(err, attn::kErrPipelineTimeout);
}

namespace {

attn_status cuda_fail(cudaError_t e)
{
    t_last_cuda_error = (int)e;
    return ATTN_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device state; called with g_mu held and the device current.
cudaError_t device_state(int dev, DeviceState **out)
{
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        cudaError_t e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_error_word);
        if (e != cudaSuccess) return e;
        d.err_word = static_cast<unsigned *>(p);
        d.ready = true;
    }
    *out = &d;
    return cudaSuccess;
}

attn::KernelInfo kernel_info(int head_dim, int group, int variant, bool multi = false)
{
    switch (head_dim) {
    case 8: return attn::kernel_info_hd8(group, variant, multi);
    case 64: return attn::kernel_info_hd64(group, variant, multi);
    case 128: return attn::kernel_info_hd128(group, variant, multi);
    case 256: return attn::kernel_info_hd256(group, variant, multi);
    default: return attn::KernelInfo{0, 0, 0, false, 0, 0};
    }
}

bool head_dim_supported(int hd) { return hd == 8 || hd == 64 || hd == 128 || hd == 256; }

// The ATTN_VARIANT_* value that names an internal kernel form: the one-tile
// kernel's 128-row tiles at head_dim 256 are the one-tile kernel.
int public_variant(int v) { return v == attn::kVariantTileWide ? ATTN_VARIANT_TC_TILE : v; }

// ATTN_VARIANT_AUTO, first choice: the mma.sync tensor-core kernel wherever it
// is compiled (head_dim % 16 == 0); it was measured faster than the CUDA-core
// kernel for every group size. head_dim 8 runs on CUDA cores.
int resolve_variant(int variant, int head_dim, int group)
{
    (void)group;
    if (variant == ATTN_VARIANT_AUTO)
        return head_dim % 16 == 0 ? attn::kVariantTc : attn::kVariantSimt;
    return variant;
}

// Static split count P (the host never sees nkv). With the capacity known,
// size the chunk so that at full capacity the (sequence, KV head) units fill
// `waves` waves of resident blocks -- one wave for a single sequence, eight for
// a batch whose lengths may be ragged, so blocks of unequal work still balance
// -- round it up to the kernel's row granule and take P = ceil(cap / chunk).
// Without it: one wave. A unit is one (sequence, KV head, query group) block
// column. With kv_stable, one sequence and a short call (at one block per SM
// each block's rows fit in a few tiles, so the launch is bound by latency
// rather than bandwidth) the wave is one block per SM, leaving room for the
// next flagged call's blocks.
int heuristic(int n_seq, int n_kv_head, int qgroups, int64_t cap, int sm_count,
              const attn::KernelInfo &ki, bool kv_stable)
{
    const int64_t units = (int64_t)n_seq * n_kv_head * (qgroups > 0 ? qgroups : 1);
    int per_sm = ki.blocks_per_sm > 0 ? ki.blocks_per_sm : 1;
    const bool short_stable = kv_stable && n_seq == 1 && cap > 0 && sm_count > 0 &&
        (cap * units + sm_count - 1) / sm_count <= (int64_t)kStableTiles * ki.tile_rows;
    if (short_stable) per_sm = 1;
    const int64_t slots = (int64_t)sm_count * per_sm;
    const int64_t gran = ki.granule > 0 ? ki.granule : attn::kSplitGranule;
    int64_t P;
    if (cap > 0) {
        const int64_t waves = n_seq > 1 ? 8 : 1;
        int64_t chunk = (cap * units + waves * slots - 1) / (waves * slots);
        chunk = (chunk + gran - 1) / gran * gran;
        // a short early-start block takes no more rows than its stage ring
        // holds, so that all of its copies start before the grid dependency
        const int64_t ring = (int64_t)ki.stages * ki.tile_rows;
        if (short_stable && ring >= gran && chunk > ring) chunk = ring / gran * gran;
        P = (cap + chunk - 1) / chunk;
    } else {
        P = slots / (units > 0 ? units : 1);
    }
    // a kernel whose block takes at most max_chunk rows needs enough splits
    // to cover the capacity
    if (ki.max_chunk > 0 && cap > 0) {
        const int64_t need = (cap + ki.max_chunk - 1) / ki.max_chunk;
        if (P < need) P = need;
    }
    // Balanced chunks (the one-tile kernel's wide tiles, one block per SM): where a
    // count that gives each SM one block makes chunks of more than three quarters
    // of a tile at full capacity, take it; the device rounds such chunks to 16
    // rows, not to whole tiles (the 7b layer: 38 splits of 224 rows, the long
    // layer: 76 of 112, on all 152 SMs). Shorter contexts run whole tiles.
    if (ki.balanced && cap > 0 && sm_count > 0 && ki.max_chunk > 0) {
        const int per_sm2 = ki.blocks_per_sm >= 3 ? 2 : ki.blocks_per_sm == 1 ? 1 : 0;
        const int64_t P2 = per_sm2 > 0 ? (int64_t)sm_count * per_sm2 / units : 0;
        const int64_t c2 = P2 > 0 ? (cap + P2 - 1) / P2 : 0;
        if (P2 > 0 && 4 * c2 > 3 * (int64_t)ki.max_chunk && c2 <= ki.max_chunk) P = P2;
    }
    if (P < 1) P = 1;
    if (P > kMaxSplits) P = kMaxSplits;
    return (int)P;
}

// Whether a one-tile kernel (max_chunk rows per block) can take the call:
// head_dim 128 or 256 (several query rows: the one-tile mma.sync kernel at 128,
// ceil(n_q * group / 16) blocks per split and KV head; tcgen05 when a KV head's
// (row, head) slots fit one 16-slot block); a known capacity; splits of at most one tile
// each; and one wave of its blocks (at full capacity at most blocks_per_sm
// tiles per SM, so a short call, bound by its chain of dependent steps rather
// than by bandwidth). On success `ku` holds the kernel's info.
bool one_tile_fits(int variant, int head_dim, int group, int n_q, int n_seq, int n_kv_head, int64_t cap,
                   int sm_count, int n_splits, int split_len, bool kv_stable, attn::KernelInfo &ku)
{
    const int qgroups = (n_q * group + attn::kMqHeadsPerBlock - 1) / attn::kMqHeadsPerBlock;
    // the tcgen05 kernel takes one query group per KV head; the one-tile mma.sync
    // kernel as many as fit one wave
    if ((head_dim != 128 && head_dim != 256) || (variant == attn::kVariantUmma && n_q > 1 && qgroups != 1) ||
        cap <= 0 || sm_count <= 0)
        return false;
    ku = kernel_info(head_dim, group, variant, n_q > 1);
    if (!ku.available) return false;
    const bool fits = split_len > 0 ? split_len <= ku.max_chunk
                                    : n_splits == 0 || (int64_t)n_splits * ku.max_chunk >= cap;
    const int64_t pu = n_splits > 0 ? n_splits
                       : split_len > 0 ? (cap + split_len - 1) / split_len
                                       : heuristic(n_seq, n_kv_head, n_q > 1 ? qgroups : 1, cap, sm_count, ku,
                                                   kv_stable);
    // the one-tile mma.sync kernel serves several block-length splits per block
    const int64_t spb = variant == attn::kVariantTile && n_q == 1 && attn::tile_serves_splits(ku.tile_rows, split_len)
                            ? ku.tile_rows / split_len : 1;
    const int64_t qb = n_q > 1 ? qgroups : 1;
    return fits && (pu + spb - 1) / spb * n_kv_head * n_seq * qb <= (int64_t)sm_count * ku.blocks_per_sm;
}

// ATTN_VARIANT_AUTO for short calls (one_tile_fits): one query row runs the
// one-tile mma.sync kernel (operands in registers, no tensor-memory round
// trips; measured faster than the tcgen05 kernel at every context of the
// 7b-like layer -- 3.7 against 4.5 us per call at context 128, 5.8 against
// 6.0 at 8192 -- and on the head_dim-256 layer, 6.3 against 7.2 us); so do
// several query rows at head_dim 128 (two rows of the 7b-like layer at context
// 8192: 7.6 us against 8.7 on tcgen05); several rows at head_dim 256 run the
// tcgen05 kernel. Long caches and batches keep the mma.sync streaming kernel
// (0: no short-call kernel).
// The call path and the planning entry points share this rule, so that they
// report the kernel and split count a call uses.
int auto_short_kernel(int head_dim, int group, int n_q, int n_seq, int n_kv_head, int64_t cap,
                      int sm_count, int n_splits, int split_len, bool kv_stable, attn::KernelInfo &ku)
{
    // By count: where one block per SM makes chunks of more than three quarters of the
    // wide tile (256 rows at head_dim 128, 128 at 256), the wide tile with balanced
    // chunks, one block per SM (the 7b layer: 38 splits of 224 rows, 5.89 -> 5.51 us per
    // layer at full context; the long layer: 76 splits of 112 rows, 6.32 -> 6.00 us);
    // several query rows too at head_dim 128 with one query group per KV head
    const int qgroups1 = (n_q * group + attn::kMqHeadsPerBlock - 1) / attn::kMqHeadsPerBlock;
    if ((n_q == 1 ? head_dim == 128 || head_dim == 256 : head_dim == 128 && qgroups1 == 1) && n_splits == 0 &&
        split_len == 0 && cap > 0 && sm_count > 0) {
        const int64_t wide = head_dim == 256 ? 128 : 256;      // the wide tile's rows
        const int64_t P1 = (int64_t)sm_count / ((int64_t)n_seq * n_kv_head);
        const int64_t c1 = P1 > 0 ? (cap + P1 - 1) / P1 : 0;
        if (P1 > 0 && 4 * c1 > 3 * wide && c1 <= wide &&
            one_tile_fits(attn::kVariantTileWide, head_dim, group, n_q, n_seq, n_kv_head, cap, sm_count, n_splits,
                          split_len, kv_stable, ku))
            return attn::kVariantTileWide;
    }
    if ((n_q == 1 || head_dim == 128) &&
        one_tile_fits(attn::kVariantTile, head_dim, group, n_q, n_seq, n_kv_head, cap, sm_count, n_splits,
                      split_len, kv_stable, ku))
        return attn::kVariantTile;
    // splits longer than a tile (block length 128 at head_dim 256, 256 at 128): the wide
    // tile, one block per SM
    if ((n_q == 1 || head_dim == 128) &&
        one_tile_fits(attn::kVariantTileWide, head_dim, group, n_q, n_seq, n_kv_head, cap, sm_count, n_splits,
                      split_len, kv_stable, ku))
        return attn::kVariantTileWide;
    if (one_tile_fits(attn::kVariantUmma, head_dim, group, n_q, n_seq, n_kv_head, cap, sm_count, n_splits,
                      split_len, kv_stable, ku))
        return attn::kVariantUmma;
    return 0;
}

// The plan of a call: which partial kernel runs, how many splits, how many
// workspace bytes, and the facts the launch needs besides.
struct CallPlan {
    int variant = 0;                  // resolved kernel (attn::kVariant*), never auto
    attn::KernelInfo ki{};
    int n_splits = 0;
    size_t workspace = 0;             // bytes of partials (0: the fused form keeps them on chip)
    int group = 0;
    int qgroups = 1;
    int kv_dtype = attn::kKvF16;
    int kv_stable = 0;
};

// Checks of everything but the pointers, done before the device is touched.
attn_status check_shape(int n_seq, int n_head, int n_kv_head, int head_dim, int64_t cap,
                        int n_splits, int split_len, int variant, int n_q, bool appending,
                        CallPlan &pl)
{
    pl.kv_dtype = (variant & ATTN_KV_BF16) ? attn::kKvBf16 : attn::kKvF16;
    pl.kv_stable = (variant & ATTN_KV_STABLE) ? 1 : 0;
    variant &= ~(ATTN_KV_BF16 | ATTN_KV_STABLE);
    if (n_seq < 0 || n_head <= 0 || n_kv_head <= 0 || head_dim <= 0) return ATTN_ERR_INVALID_ARG;
    if (n_head % n_kv_head != 0) return ATTN_ERR_INVALID_ARG;
    if (cap < 1) return ATTN_ERR_INVALID_ARG;
    if (n_splits < 0 || n_splits > kMaxSplits || split_len < 0) return ATTN_ERR_INVALID_ARG;
    if (variant != ATTN_VARIANT_AUTO && variant != ATTN_VARIANT_SIMT && variant != ATTN_VARIANT_TC &&
        variant != ATTN_VARIANT_TCGEN05 && variant != ATTN_VARIANT_TCGEN05_CLUSTER &&
        variant != ATTN_VARIANT_TC_TILE)
        return ATTN_ERR_INVALID_ARG;
    if (n_seq > 65535 || n_kv_head > 65535) return ATTN_ERR_INVALID_ARG;   // grid z limit; heads kept as before
    if ((int64_t)n_seq * cap > kMaxFlatRows - 1024) return ATTN_ERR_INVALID_ARG;
    pl.group = n_head / n_kv_head;
    // n_q * G <= 8192 also keeps the kernels' multiply-shift division by G exact
    if (n_q < 1 || n_q > 1024) return ATTN_ERR_INVALID_ARG;
    if (n_q > 1 && appending) return ATTN_ERR_INVALID_ARG;
    if (!head_dim_supported(head_dim) || pl.group > 8) return ATTN_ERR_UNSUPPORTED;
    if (n_q > 1 && (head_dim % 16 != 0 || variant == ATTN_VARIANT_SIMT)) return ATTN_ERR_UNSUPPORTED;
    pl.variant = resolve_variant(variant, head_dim, pl.group);
    const int qg = (n_q * pl.group + attn::kMqHeadsPerBlock - 1) / attn::kMqHeadsPerBlock;
    if (n_q > 1 && (int64_t)n_kv_head * qg > 65535) return ATTN_ERR_INVALID_ARG;
    pl.qgroups = n_q > 1 ? qg : 1;
    pl.ki = kernel_info(head_dim, pl.group, pl.variant, n_q > 1);
    if (!pl.ki.available) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// The rest of the plan, which needs the device (its SM count; for the fused
// form whether it holds the cluster). Called with g_mu held, after
// check_shape, for n_seq > 0.
attn_status finish_plan(DeviceState *ds, int n_seq, int n_head, int n_kv_head, int head_dim,
                        int64_t cap, bool cap_known, int n_splits, int split_len, int variant,
                        int stages, int n_q, CallPlan &pl)
{
    variant &= ~(ATTN_KV_BF16 | ATTN_KV_STABLE);
    if (variant == ATTN_VARIANT_AUTO) {
        attn::KernelInfo ku{};
        const int vs = auto_short_kernel(head_dim, pl.group, n_q, n_seq, n_kv_head, cap_known ? cap : 0,
                                         ds->sm_count, n_splits, split_len, pl.kv_stable != 0, ku);
        if (vs) {
            pl.variant = vs;
            pl.ki = ku;
        }
    }
    // The cluster-fused form of the tcgen05 kernel (partial and combine in one launch,
    // 16 splits per (sequence, KV head) merged through distributed shared memory),
    // on request only: a whole call, one query row, head_dim 128, splits by count with
    // P = 16 (n_splits 0 or 16), a capacity of at most 16 blocks of 4 tiles, and a
    // device that holds the 16-block cluster. Variant 0 does not take it: on one box it
    // was 1 % faster than the plain tcgen05 kernel at context 2048 and 7-13 % slower at
    // 512 and 128 (capacity 2048), and 20 % slower at the 7b capacity of 8192.
    if (pl.variant == attn::kVariantFused) {
        const attn::KernelInfo kf = kernel_info(head_dim, pl.group, attn::kVariantFused, n_q > 1);
        bool ok = kf.available && n_q == 1 && stages == (attn::kStagePartial | attn::kStageCombine) &&
                  split_len == 0 && (n_splits == 0 || n_splits == kFusedSplits) && cap_known &&
                  cap <= (int64_t)kFusedSplits * kf.max_chunk;
        if (!ok) return ATTN_ERR_INVALID_ARG;
        if (ds->fused_ok < 0) ds->fused_ok = attn::fused_fits_hd128() ? 1 : 0;   // asked once per device
        if (ds->fused_ok != 1) return ATTN_ERR_UNSUPPORTED;
        pl.ki = kf;
    }
    // by block length with no split count: one split per block of rows of the
    // capacity (Red Lite dev35 "Change": P = ceil(positions / block))
    const int64_t P_blk = split_len > 0 && n_splits == 0 ? (cap + split_len - 1) / split_len : 0;
    if (P_blk > kMaxSplits) return ATTN_ERR_INVALID_ARG;
    const int P = pl.variant == attn::kVariantFused ? kFusedSplits
                : n_splits > 0 ? n_splits
                : P_blk > 0    ? (int)P_blk
                               : heuristic(n_seq, n_kv_head, pl.qgroups, cap_known ? cap : 0,
                                           ds->sm_count, pl.ki, pl.kv_stable != 0);
    if (split_len > 0 && (int64_t)P * split_len < cap) return ATTN_ERR_INVALID_ARG;
    // the one-tile kernel at head_dim 256 takes splits longer than its 96-row tile
    // in 128-row tiles
    if (pl.variant == attn::kVariantTile && (n_q == 1 || head_dim == 128) &&
        (split_len > 0 ? split_len > pl.ki.max_chunk : (cap_known && (int64_t)P * pl.ki.max_chunk < cap))) {
        const attn::KernelInfo kw = kernel_info(head_dim, pl.group, attn::kVariantTileWide);
        if (kw.available) {
            pl.variant = attn::kVariantTileWide;
            pl.ki = kw;
        }
    }
    // one tile per block: every split must fit in max_chunk rows at any nkv <= cap
    if (pl.ki.max_chunk > 0 && (split_len > 0 ? split_len > pl.ki.max_chunk
                                              : (!cap_known || (int64_t)P * pl.ki.max_chunk < cap)))
        return ATTN_ERR_INVALID_ARG;
    pl.n_splits = P;
    // the fused form keeps its partial states on chip: no workspace
    pl.workspace = pl.variant == attn::kVariantFused ? 0 : attn_workspace_size(n_seq, n_q * n_head, head_dim, P);
    return ATTN_OK;
}

attn_status decode_impl(const float *q, const void *k_cache, const void *v_cache,
                        const int32_t *positions, float *out, int n_seq, int n_head,
                        int n_kv_head, int head_dim, float scale, int64_t cap, bool cap_known,
                        int n_splits, int split_len, int variant, void *workspace,
                        size_t workspace_bytes, int stages, cudaStream_t stream,
                        const void *k_new = nullptr, const void *v_new = nullptr, int n_q = 1)
{
    // ---- synchronous argument checks, nothing launched yet ----
    // (every check that answers ATTN_ERR_INVALID_ARG for the pointers and the
    // scale comes before the shape checks that can answer ATTN_ERR_UNSUPPORTED)
    if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (n_seq > 0 && (!q || !k_cache || !v_cache || !positions)) return ATTN_ERR_INVALID_ARG;
    if (n_seq > 0 && (stages & attn::kStageCombine) && !out) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(positions) ||
        !aligned16(out) || !aligned16(k_new) || !aligned16(v_new))
        return ATTN_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return ATTN_ERR_INVALID_ARG;
    CallPlan pl;
    attn_status st = check_shape(n_seq, n_head, n_kv_head, head_dim, cap, n_splits, split_len, variant,
                                 n_q, k_new != nullptr, pl);
    if (st != ATTN_OK) return st;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTN_ERR_INVALID_ARG;
    if (n_seq == 0) return ATTN_OK;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);

    std::unique_lock<std::mutex> lock(g_mu);
    DeviceState *ds = nullptr;
    e = device_state(dev, &ds);
    if (e != cudaSuccess) return cuda_fail(e);
    st = finish_plan(ds, n_seq, n_head, n_kv_head, head_dim, cap, cap_known, n_splits, split_len, variant,
                     stages, n_q, pl);
    if (st != ATTN_OK) return st;
    const int v = pl.variant, P = pl.n_splits, group = pl.group, qgroups = pl.qgroups;
    const int kv_dtype = pl.kv_dtype, kv_stable = pl.kv_stable;
    const size_t need = pl.workspace;

    if (!workspace && need > 0) {
        if (stages != (attn::kStagePartial | attn::kStageCombine)) return ATTN_ERR_INVALID_ARG;
        if (ds->ws_bytes < need) {
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            e = cudaStreamIsCapturing(stream, &cs);
            if (e != cudaSuccess) return cuda_fail(e);
            if (cs != cudaStreamCaptureStatusNone) return ATTN_ERR_WORKSPACE;
            if (ds->ws) {
                e = cudaFree(ds->ws);                 // synchronises with work using it
                ds->ws = nullptr;
                ds->ws_bytes = 0;
                if (e != cudaSuccess) return cuda_fail(e);
            }
            e = cudaMalloc(&ds->ws, need);
            if (e != cudaSuccess) return cuda_fail(e);
            ds->ws_bytes = need;
        }
        workspace = ds->ws;
    } else if (workspace_bytes < need) {
        return ATTN_ERR_WORKSPACE;
    }
    unsigned *err_word = ds->err_word;
    lock.unlock();

    attn::LaunchRequest r{};
    r.pa.q = q;
    r.pa.k = static_cast<const uint16_t *>(k_cache);
    r.pa.v = static_cast<const uint16_t *>(v_cache);
    r.pa.positions = positions;
    const size_t o_bytes = align256((size_t)n_seq * n_q * n_head * P * head_dim * sizeof(float));
    r.pa.ws_o = need > 0 ? static_cast<float *>(workspace) : nullptr;
    r.pa.ws_ml = need > 0 ? reinterpret_cast<float2 *>(static_cast<uint8_t *>(workspace) + o_bytes) : nullptr;
    r.pa.err = err_word;
    r.pa.n_head = n_head;
    r.pa.n_kv_head = n_kv_head;
    r.pa.n_splits = P;
    r.pa.split_len = split_len;
    r.pa.cap = cap;
    r.pa.qscale = (float)((double)scale * 1.4426950408889634);
    r.pa.n_q = n_q;
    r.pa.qgroups = n_q > 1 ? qgroups : 1;
    r.pa.kv_stable = kv_stable;
    r.pa.group = group;
    r.pa.group_magic = (65536u + (unsigned)group - 1u) / (unsigned)group;
    if (k_new) {
        r.pa.k_new = static_cast<const uint16_t *>(k_new);
        r.pa.v_new = static_cast<const uint16_t *>(v_new);
        r.pa.k_w = static_cast<uint16_t *>(const_cast<void *>(k_cache));
        r.pa.v_w = static_cast<uint16_t *>(const_cast<void *>(v_cache));
    }
    r.k_cache = k_cache;
    r.v_cache = v_cache;
    r.out = out;
    r.n_seq = n_seq;
    r.head_dim = head_dim;
    r.group = group;
    r.variant = v;
    r.stages = stages;
    r.kv_dtype = kv_dtype;
    r.stream = stream;

    e = attn::launch_any(r);
    if (e != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
}

} // namespace

// ---------------------------------------------------------------------------
// Internal helpers used by the kernel translation units.
// ---------------------------------------------------------------------------
namespace attn {

// The driver's tensor-map encoder, looked up once.
static cudaError_t load_encoder()
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult qr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &qr);
        if (e != cudaSuccess) return e;
        if (qr != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return cudaSuccess;
}

cudaError_t encode_kv_map(CUtensorMap *map, const void *base, int64_t rows, int n_kv_head,
                          int head_dim, int box_x, int box_rows, int kv_dtype)
{
    const cudaError_t le = load_encoder();
    if (le != cudaSuccess) return le;
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_kv_head, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_kv_head * head_dim * 2};
    const cuuint32_t box[3] = {(cuuint32_t)box_x, 1u, (cuuint32_t)box_rows};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUtensorMapSwizzle sw = (box_x * 2 == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
    const CUtensorMapDataType dt = kv_dtype == kKvBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = g_encode(map, dt, 3, const_cast<void *>(base), dims,
                                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_kv_map4(CUtensorMap *map, const void *base, int n_seq, int64_t cap, int n_kv_head,
                           int head_dim, int box_x, int box_rows, int kv_dtype)
{
    const cudaError_t le = load_encoder();
    if (le != cudaSuccess) return le;
    const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)n_kv_head, (cuuint64_t)cap,
                                (cuuint64_t)n_seq};
    const cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_kv_head * head_dim * 2,
                                   (cuuint64_t)cap * n_kv_head * head_dim * 2};
    const cuuint32_t box[4] = {(cuuint32_t)box_x, 1u, (cuuint32_t)box_rows, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUtensorMapSwizzle sw = (box_x * 2 == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
    const CUtensorMapDataType dt = kv_dtype == kKvBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = g_encode(map, dt, 4, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t ensure_smem_attr(const void *func, int bytes)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_smem_done.count({func, dev})) return cudaSuccess;
    if (bytes > 48 * 1024) {
        e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
    }
    // All of the unified L1/shared array as shared memory, for every kernel of
    // the library (the combine too, although it needs 1 KB): an SM holds one
    // carve-out at a time, so a kernel that preferred a small one would keep
    // the next layer's partial blocks off the SMs it occupies.
    e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) g_smem_done.insert({func, dev});
    return e;
}

cudaError_t launch_pdl(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void **args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, func, args);
}

cudaError_t launch_pdl_cluster(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               void **args, unsigned cluster_x)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelExC(&cfg, func, args);
}

int cluster_slots(const void *func, dim3 block, size_t smem, unsigned cluster_x)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster_x, 1, 1);
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster_x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

} // namespace attn

// ---------------------------------------------------------------------------
// Public C ABI.
// ---------------------------------------------------------------------------
extern "C" {

attn_status attn_decode(const float *q, const void *k_cache, const void *v_cache,
                        const int32_t *positions, float *out, int n_seq, int n_head,
                        int n_kv_head, int head_dim, float scale, attn_stream_t stream)
{
    if (n_seq != 1) return ATTN_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, positions, out, n_seq, n_head, n_kv_head, head_dim,
                       scale, kUnknownCap, false, 0, 0, ATTN_VARIANT_AUTO, nullptr, 0,
                       attn::kStagePartial | attn::kStageCombine,
                       reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_decode_ex(const float *q, const void *k_cache, const void *v_cache,
                           const int32_t *positions, float *out, int n_seq, int n_head,
                           int n_kv_head, int head_dim, float scale, int64_t cap,
                           int n_splits, int split_len, int variant, void *workspace,
                           size_t workspace_bytes, attn_stream_t stream)
{
    return decode_impl(q, k_cache, v_cache, positions, out, n_seq, n_head, n_kv_head, head_dim,
                       scale, cap, true, n_splits, split_len, variant, workspace, workspace_bytes,
                       attn::kStagePartial | attn::kStageCombine,
                       reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_decode_append(const float *q, const void *k_new, const void *v_new,
                               void *k_cache, void *v_cache, const int32_t *positions, float *out,
                               int n_seq, int n_head, int n_kv_head, int head_dim, float scale,
                               int64_t cap, int n_splits, int split_len, int variant,
                               void *workspace, size_t workspace_bytes, attn_stream_t stream)
{
    if (n_seq > 0 && (!k_new || !v_new)) return ATTN_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, positions, out, n_seq, n_head, n_kv_head, head_dim,
                       scale, cap, true, n_splits, split_len, variant, workspace, workspace_bytes,
                       attn::kStagePartial | attn::kStageCombine,
                       reinterpret_cast<cudaStream_t>(stream), k_new, v_new);
}

attn_status attn_decode_multi(const float *q, const void *k_cache, const void *v_cache,
                              const int32_t *positions, float *out, int n_seq, int n_q, int n_head,
                              int n_kv_head, int head_dim, float scale, int64_t cap, int n_splits,
                              int split_len, int variant, void *workspace, size_t workspace_bytes,
                              attn_stream_t stream)
{
    return decode_impl(q, k_cache, v_cache, positions, out, n_seq, n_head, n_kv_head, head_dim,
                       scale, cap, true, n_splits, split_len, variant, workspace, workspace_bytes,
                       attn::kStagePartial | attn::kStageCombine,
                       reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, n_q);
}

attn_status attn_decode_partial(const float *q, const void *k_cache, const void *v_cache,
                                const int32_t *positions, int n_seq, int n_head, int n_kv_head,
                                int head_dim, float scale, int64_t cap, int n_splits,
                                int split_len, int variant, void *workspace,
                                size_t workspace_bytes, attn_stream_t stream)
{
    if (n_splits <= 0 || !workspace) return ATTN_ERR_INVALID_ARG;
    return decode_impl(q, k_cache, v_cache, positions, nullptr, n_seq, n_head, n_kv_head,
                       head_dim, scale, cap, true, n_splits, split_len, variant, workspace,
                       workspace_bytes, attn::kStagePartial, reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_decode_combine(const void *workspace, size_t workspace_bytes, float *out,
                                int n_seq, int n_head, int head_dim, int n_splits,
                                attn_stream_t stream)
{
    if (n_seq < 0 || n_head <= 0 || n_splits <= 0 || n_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
    if (n_seq > 65535) return ATTN_ERR_INVALID_ARG;
    if (!head_dim_supported(head_dim)) return ATTN_ERR_UNSUPPORTED;
    if (n_seq == 0) return ATTN_OK;
    if (!workspace || !out || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return ATTN_ERR_INVALID_ARG;
    if (workspace_bytes < attn_workspace_size(n_seq, n_head, head_dim, n_splits))
        return ATTN_ERR_WORKSPACE;
    attn::LaunchRequest r{};
    const size_t o_bytes = align256((size_t)n_seq * n_head * n_splits * head_dim * sizeof(float));
    r.pa.ws_o = static_cast<float *>(const_cast<void *>(workspace));
    r.pa.ws_ml = reinterpret_cast<float2 *>(static_cast<uint8_t *>(const_cast<void *>(workspace)) + o_bytes);
    r.pa.n_head = n_head;
    r.pa.n_splits = n_splits;
    r.out = out;
    r.n_seq = n_seq;
    r.head_dim = head_dim;
    r.group = 1;
    r.variant = attn::kVariantSimt;
    r.stages = attn::kStageCombine;
    r.stream = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = attn::launch_any(r);
    if (e != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
}

} // extern "C"

namespace {

// The kernel a call with the heuristic's split count runs (and that kernel's
// properties), or 0 when the shape is not supported. sm_count <= 0: the
// current device's.
int plan_variant(int n_seq, int n_q, int n_head, int n_kv_head, int head_dim, int64_t cap,
                 int &sm_count, int variant, attn::KernelInfo &ki)
{
    const bool kv_stable = (variant & ATTN_KV_STABLE) != 0;
    variant &= ~(ATTN_KV_BF16 | ATTN_KV_STABLE);
    if (variant != ATTN_VARIANT_AUTO && variant != ATTN_VARIANT_SIMT && variant != ATTN_VARIANT_TC &&
        variant != ATTN_VARIANT_TCGEN05 && variant != ATTN_VARIANT_TCGEN05_CLUSTER &&
        variant != ATTN_VARIANT_TC_TILE)
        return 0;
    if (n_seq <= 0 || n_q < 1 || n_q > 1024 || n_head <= 0 || n_kv_head <= 0 ||
        n_head % n_kv_head != 0)
        return 0;
    const int group = n_head / n_kv_head;
    if (!head_dim_supported(head_dim) || group > 8) return 0;
    if (sm_count <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return 0;
        if (cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
    }
    int v = resolve_variant(variant, head_dim, group);
    attn::KernelInfo ku{};
    if (variant == ATTN_VARIANT_AUTO) {
        const int vs = auto_short_kernel(head_dim, group, n_q, n_seq, n_kv_head, cap, sm_count, 0, 0,
                                         kv_stable, ku);
        if (vs) v = vs;
    }
    ki = kernel_info(head_dim, group, v, n_q > 1);
    return ki.available ? v : 0;
}

} // namespace

extern "C" {

int attn_split_heuristic_ex(int n_seq, int n_q, int n_head, int n_kv_head, int head_dim,
                            int64_t cap, int sm_count, int variant)
{
    attn::KernelInfo ki{};
    const int v = plan_variant(n_seq, n_q, n_head, n_kv_head, head_dim, cap, sm_count, variant, ki);
    if (!v) return 0;
    if (v == attn::kVariantFused) return kFusedSplits;
    const int group = n_head / n_kv_head;
    const int qgroups = n_q > 1 ? (n_q * group + attn::kMqHeadsPerBlock - 1) / attn::kMqHeadsPerBlock : 1;
    return heuristic(n_seq, n_kv_head, qgroups, cap, sm_count, ki, (variant & ATTN_KV_STABLE) != 0);
}

int attn_resolve_variant(int n_seq, int n_q, int n_head, int n_kv_head, int head_dim, int64_t cap,
                         int sm_count, int variant)
{
    attn::KernelInfo ki{};
    return public_variant(plan_variant(n_seq, n_q, n_head, n_kv_head, head_dim, cap, sm_count, variant, ki));
}

attn_status attn_plan_call(int n_seq, int n_q, int n_head, int n_kv_head, int head_dim, int64_t cap,
                           int n_splits, int split_len, int variant, int *variant_out,
                           int *n_splits_out, size_t *workspace_bytes_out)
{
    CallPlan pl;
    attn_status st = check_shape(n_seq, n_head, n_kv_head, head_dim, cap, n_splits, split_len, variant,
                                 n_q, false, pl);
    if (st != ATTN_OK) return st;
    if (n_seq == 0) return ATTN_ERR_INVALID_ARG;          // nothing to plan
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState *ds = nullptr;
        e = device_state(dev, &ds);
        if (e != cudaSuccess) return cuda_fail(e);
        st = finish_plan(ds, n_seq, n_head, n_kv_head, head_dim, cap, true, n_splits, split_len, variant,
                         attn::kStagePartial | attn::kStageCombine, n_q, pl);
    }
    if (st != ATTN_OK) return st;
    if (variant_out) *variant_out = public_variant(pl.variant);
    if (n_splits_out) *n_splits_out = pl.n_splits;
    if (workspace_bytes_out) *workspace_bytes_out = pl.workspace;
    return ATTN_OK;
}

int attn_split_heuristic(int n_seq, int n_head, int n_kv_head, int head_dim, int64_t cap,
                         int sm_count)
{
    return attn_split_heuristic_ex(n_seq, 1, n_head, n_kv_head, head_dim, cap, sm_count,
                                   ATTN_VARIANT_AUTO);
}

size_t attn_workspace_size(int n_seq, int n_head, int head_dim, int n_splits)
{
    if (n_seq <= 0 || n_head <= 0 || head_dim <= 0 || n_splits <= 0) return 0;
    const size_t slots = (size_t)n_seq * n_head * n_splits;
    return align256(slots * head_dim * sizeof(float)) + align256(slots * 2 * sizeof(float));
}

attn_status attn_read_device_error(attn_stream_t stream, unsigned int *flags)
{
    if (!flags) return ATTN_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned v = 0;
    e = cudaMemcpyFromSymbol(&v, g_attn_error_word, sizeof(v));
    if (e != cudaSuccess) return cuda_fail(e);
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_attn_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e);
    *flags = v;
    return ATTN_OK;
}

const char *attn_status_string(attn_status status)
{
    switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    default: return "ATTN_ERR_UNKNOWN";
    }
}

attn_status attn_selftest_bounded_wait(unsigned long long limit_ns, attn_stream_t stream)
{
    if (limit_ns == 0 || limit_ns > attn::kWaitLimitNs) return ATTN_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    DeviceState *ds = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        e = device_state(dev, &ds);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    attn_selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ds->err_word,
                                                                                    limit_ns);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
}

int attn_last_cuda_error(void) { return t_last_cuda_error; }

int attn_version(void) { return 10000; }

} // extern "C"
