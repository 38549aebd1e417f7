// Instantiation of the fused forward kernel for head_dim 64 (one translation unit per
// head_dim so the variants compile in parallel).
#include "attn_fwd_kernel.cuh"

namespace gbattn {
cudaError_t launch_fwd_64(const FwdLaunch &a) { return launch_fwd_d<64>(a); }
int splitkv_clusters_64() { return splitkv_max_clusters<64>(); }
}  // namespace gbattn
