// Instantiation of the fused forward kernel for head_dim 256 (one translation unit per
// head_dim so the variants compile in parallel).
#include "attn_fwd_kernel.cuh"

namespace gbattn {
cudaError_t launch_fwd_256(const FwdLaunch &a) { return launch_fwd_d<256>(a); }
}  // namespace gbattn
