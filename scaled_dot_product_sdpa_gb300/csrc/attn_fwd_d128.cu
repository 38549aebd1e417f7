// Instantiation of the fused forward kernel for head_dim 128 (one translation unit per
// head_dim so the variants compile in parallel).
#include "attn_fwd_kernel.cuh"

namespace gbattn {
cudaError_t launch_fwd_128(const FwdLaunch &a) { return launch_fwd_d<128>(a); }
int splitkv_clusters_128() { return splitkv_max_clusters<128>(); }
}  // namespace gbattn
