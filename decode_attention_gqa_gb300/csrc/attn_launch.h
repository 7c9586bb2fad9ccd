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
    int variant;             // kVariantSimt / kVariantTc (resolved, never auto)
    int stages;              // kStagePartial | kStageCombine
    cudaStream_t stream;
};

// Static properties of the partial kernel chosen for (head_dim, variant).
struct KernelInfo {
    int tile_rows;           // rows per pipeline stage
    int granule;             // split chunks (by count) are rounded up to this many rows
    int blocks_per_sm;       // resident blocks per SM (from its shared-memory need)
    bool available;          // compiled for this (head_dim, group)
};

// Implemented in attn_api.cu.
// Build a 3-D tensor map over a [rows][n_kv_head][head_dim] f16 cache with a
// box of (box_x, 1, box_rows); 128-byte swizzle when box_x * 2 == 128.
cudaError_t encode_kv_map(CUtensorMap *map, const void *base, int64_t rows, int n_kv_head,
                          int head_dim, int box_x, int box_rows);
// Opt a kernel into more than 48 KB of dynamic shared memory (once per device).
cudaError_t ensure_smem_attr(const void *func, int bytes);
// Launch with the programmatic-stream-serialisation attribute set.
cudaError_t launch_pdl(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void **args);

// Implemented in attn_kernels_hd{8,64,128,256}.cu.
KernelInfo kernel_info_hd8(int group, int variant);
KernelInfo kernel_info_hd64(int group, int variant);
KernelInfo kernel_info_hd128(int group, int variant);
KernelInfo kernel_info_hd256(int group, int variant);
cudaError_t launch_hd8(const LaunchRequest &r);
cudaError_t launch_hd64(const LaunchRequest &r);
cudaError_t launch_hd128(const LaunchRequest &r);
cudaError_t launch_hd256(const LaunchRequest &r);

} // namespace attn
