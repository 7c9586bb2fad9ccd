// Kernels for head_dim 256 (partial variants for group sizes 1..8, combine).
#include "attn_kernels_impl.cuh"

namespace attn {
cudaError_t launch_hd256(const LaunchRequest &r) { return launch_for_hd<256>(r); }
KernelInfo kernel_info_hd256(int group, int variant) { return kernel_info_for_hd<256>(group, variant); }
} // namespace attn
