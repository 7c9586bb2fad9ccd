// attn_noalloc.cu -- attn_decode_static: the decode-attention call for callers
// that cannot allocate device memory when they call it.
//
// Who: an engine step that runs while a CUDA stream is being captured (device
// allocation is not allowed during capture), a plugin whose host framework
// owns every device allocation and forbids them in its enqueue callback, or a
// process whose device-memory budget is fixed at start-up. Such callers can
// pass inputs and outputs but no workspace, and the library-owned workspace
// of attn_decode may need a cudaMalloc to grow.
//
// The partial triples (the kernels' only scratch) live instead in a fixed
// file-scope device array that every GPU loading this library holds until
// the process exits. Host code cannot use the array's name as a device
// address, so the address is looked up once per device with
// cudaGetSymbolAddress (on the first call made with that device current) and
// handed to the same kernels attn_decode_ex launches.
#include <cuda_runtime.h>

#include <mutex>

#include "attn_decode.h"

namespace {

constexpr int kMaxDevices = 64;

// The scratch: partial accumulators and (mx, S) pairs of one call.
static __device__ __align__(256) unsigned char g_attn_static_scratch[ATTN_STATIC_SCRATCH_BYTES];

std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices];        // device address of the array, per device

} // namespace

extern "C" attn_status attn_decode_static(const float *q, const void *k_cache, const void *v_cache,
                                          const int32_t *positions, float *out, int n_seq,
                                          int n_head, int n_kv_head, int head_dim, float scale,
                                          int64_t cap, int n_splits, int split_len, int variant,
                                          attn_stream_t stream)
{
    // Nothing to launch, or arguments the regular path rejects anyway: let it
    // answer (it returns before any CUDA call for these).
    if (n_seq <= 0 || n_head <= 0 || n_kv_head <= 0 || head_dim <= 0 || n_splits < 0 ||
        n_head % n_kv_head != 0)
        return attn_decode_ex(q, k_cache, v_cache, positions, out, n_seq, n_head, n_kv_head,
                              head_dim, scale, cap, n_splits, split_len, variant, nullptr, 0, stream);

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mu);
        if (!g_static_ptr[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_attn_static_scratch);
            if (e != cudaSuccess || !p) return ATTN_ERR_CUDA;
            g_static_ptr[dev] = p;
        }
        scratch = g_static_ptr[dev];
    }
    // attn_decode_ex plans the call exactly as it would with its own workspace
    // (n_splits == 0: the split count for this variant, the early-start flag
    // and the cache type included) and answers ATTN_ERR_WORKSPACE, before
    // launching anything, when that plan needs more than the fixed array.
    return attn_decode_ex(q, k_cache, v_cache, positions, out, n_seq, n_head, n_kv_head, head_dim,
                          scale, cap, n_splits, split_len, variant, scratch,
                          ATTN_STATIC_SCRATCH_BYTES, stream);
}
