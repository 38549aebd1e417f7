// Instantiation of the fused forward kernel for head_dim 512 (one translation unit per
// head_dim so the variants compile in parallel).
#include "attn_fwd_kernel.cuh"

namespace gbattn {
cudaError_t launch_fwd_512(const FwdLaunch &a) { return launch_fwd_d<512>(a); }
int splitkv_clusters_512() { return splitkv_max_clusters<512>(); }
}  // namespace gbattn
