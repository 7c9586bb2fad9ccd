// Kernels for head_dim 64 over a f16 KV cache (partial variants for group sizes 1..8, combine).
#include "attn_kernels_impl.cuh"

namespace attn {
cudaError_t launch_hd64_f16(const LaunchRequest &r) { return launch_for_hd<64, __half>(r); }
KernelInfo kernel_info_hd64(int group, int variant, bool multi) { return kernel_info_for_hd<64>(group, variant, multi); }
} // namespace attn
