// attn_launch.h -- internal host interface between the C-ABI layer
// (attn_api.cu) and the per-head_dim kernel translation units
// (attn_kernels_hd*.cu). Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_device.cuh"

namespace attn {

constexpr int kVariantSimt = 1;
constexpr int kVariantTc = 2;
constexpr int kVariantUmma = 3;             // tcgen05 kernel (attn_partial_umma.cuh)
constexpr int kVariantFused = 4;            // tcgen05 + cluster combine (attn_fused_umma.cuh)
constexpr int kVariantTile = 5;             // one-tile mma.sync kernel (attn_partial_tile.cuh)
constexpr int kVariantTileWide = 6;         // the same with 128-row tiles at head_dim 256 (internal:
                                            // reported as the one-tile kernel)
constexpr int kMqHeadsPerBlock = 16;        // query heads per multi-query block
constexpr int kKvF16 = 0;
constexpr int kKvBf16 = 1;
constexpr int kStagePartial = 1;
constexpr int kStageCombine = 2;

struct LaunchRequest {
    PartialArgs pa;          // partial-kernel arguments (ws pointers, qscale, P, ...)
    const void *k_cache;
    const void *v_cache;
    float *out;
    int n_seq;
    int head_dim;
    int group;               // G = n_head / n_kv_head
    int variant;             // kVariantSimt / kVariantTc / kVariantUmma / kVariantFused / kVariantTile(Wide) (resolved, never auto)
    int stages;              // kStagePartial | kStageCombine
    int kv_dtype;            // kKvF16 / kKvBf16
    cudaStream_t stream;
};

// Static properties of the partial kernel chosen for (head_dim, variant).
struct KernelInfo {
    int tile_rows;           // rows per pipeline stage
    int granule;             // split chunks (by count) are rounded up to this many rows
    int blocks_per_sm;       // resident blocks per SM (from its shared-memory need)
    bool available;          // compiled for this (head_dim, group)
    int stages;              // pipeline stages (tiles in flight per block)
    int max_chunk;           // rows one block can take (0: any; the tcgen05 kernel: one tile)
    bool balanced = false;   // count-mode chunks near a tile are rounded to 16 rows (one-tile kernel)
};

// Whether the one-tile kernel serves several block-length splits per block:
// split_len divides the tile (tile_rows rows) into at least two whole 16-row
// parts (SPB = tile_rows / split_len splits per block).
inline bool tile_serves_splits(int tile_rows, int split_len)
{
    return split_len > 0 && split_len < tile_rows && split_len % 16 == 0 && tile_rows % split_len == 0;
}

// Implemented in attn_api.cu.
// Build a 3-D tensor map over a [rows][n_kv_head][head_dim] 16-bit cache
// (kv_dtype kKvF16 / kKvBf16) with a box of (box_x, 1, box_rows); 128-byte
// swizzle when box_x * 2 == 128.
cudaError_t encode_kv_map(CUtensorMap *map, const void *base, int64_t rows, int n_kv_head,
                          int head_dim, int box_x, int box_rows, int kv_dtype);
// The same cache as a 4-D tensor [n_seq][cap][n_kv_head][head_dim] with a box
// of (box_x, 1, box_rows, 1): a box that starts before a sequence's first row
// reads zeros there instead of the previous sequence's rows.
cudaError_t encode_kv_map4(CUtensorMap *map, const void *base, int n_seq, int64_t cap, int n_kv_head,
                           int head_dim, int box_x, int box_rows, int kv_dtype);
// Opt a kernel into `bytes` of dynamic shared memory (when above 48 KB) and the
// largest shared-memory carve-out (once per device).
cudaError_t ensure_smem_attr(const void *func, int bytes);
// Launch with the programmatic-stream-serialisation attribute set.
cudaError_t launch_pdl(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void **args);

// The same with a thread-block cluster of cluster_x blocks along x.
cudaError_t launch_pdl_cluster(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               void **args, unsigned cluster_x);
// How many clusters of cluster_x blocks of `func` the device can hold at once
// (0: none, or the query failed).
int cluster_slots(const void *func, dim3 block, size_t smem, unsigned cluster_x);

// Implemented in attn_kernels_hd{8,64,128,256}_{f16,bf16}.cu (kernel_info in
// the f16 units: the shapes do not depend on the element type).
KernelInfo kernel_info_hd8(int group, int variant, bool multi);
KernelInfo kernel_info_hd64(int group, int variant, bool multi);
KernelInfo kernel_info_hd128(int group, int variant, bool multi);
KernelInfo kernel_info_hd256(int group, int variant, bool multi);
// Whether the current device holds a cluster of the fused head_dim-128 kernel.
bool fused_fits_hd128();
cudaError_t launch_hd8_f16(const LaunchRequest &r);
cudaError_t launch_hd64_f16(const LaunchRequest &r);
cudaError_t launch_hd128_f16(const LaunchRequest &r);
cudaError_t launch_hd256_f16(const LaunchRequest &r);
cudaError_t launch_hd8_bf16(const LaunchRequest &r);
cudaError_t launch_hd64_bf16(const LaunchRequest &r);
cudaError_t launch_hd128_bf16(const LaunchRequest &r);
cudaError_t launch_hd256_bf16(const LaunchRequest &r);

// Dispatch on (head_dim, kv_dtype).
inline cudaError_t launch_any(const LaunchRequest &r)
{
    const bool bf = r.kv_dtype == kKvBf16;
    switch (r.head_dim) {
    case 8: return bf ? launch_hd8_bf16(r) : launch_hd8_f16(r);
    case 64: return bf ? launch_hd64_bf16(r) : launch_hd64_f16(r);
    case 128: return bf ? launch_hd128_bf16(r) : launch_hd128_f16(r);
    case 256: return bf ? launch_hd256_bf16(r) : launch_hd256_f16(r);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace attn
