// Kernels for head_dim 128 (partial variants for group sizes 1..8, combine).
#include "attn_kernels_impl.cuh"

namespace attn {
cudaError_t launch_hd128(const LaunchRequest &r) { return launch_for_hd<128>(r); }
KernelInfo kernel_info_hd128(int group, int variant) { return kernel_info_for_hd<128>(group, variant); }
} // namespace attn
