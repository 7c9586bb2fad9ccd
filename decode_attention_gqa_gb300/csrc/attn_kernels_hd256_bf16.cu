// Kernels for head_dim 256 over a bf16 KV cache (partial variants for group sizes 1..8, combine).
#include "attn_kernels_impl.cuh"

namespace attn {
cudaError_t launch_hd256_bf16(const LaunchRequest &r) { return launch_for_hd<256, __nv_bfloat16>(r); }
} // namespace attn
