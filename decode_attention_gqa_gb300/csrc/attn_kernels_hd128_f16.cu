// Kernels for head_dim 128 over a f16 KV cache (partial variants for group sizes 1..8, combine).
#include "attn_kernels_impl.cuh"

namespace attn {
cudaError_t launch_hd128_f16(const LaunchRequest &r) { return launch_for_hd<128, __half>(r); }
KernelInfo kernel_info_hd128(int group, int variant, bool multi) { return kernel_info_for_hd<128>(group, variant, multi); }
bool fused_fits_hd128() { return fused_cluster_fits<128>(); }
} // namespace attn
