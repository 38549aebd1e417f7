// Instantiation of the two-tile (ping-pong) forward kernel for head_dim 64.
#include "attn_fwd_pp.cuh"

namespace gbattn {
cudaError_t launch_fwd_pp_64(const FwdLaunch &a) { return launch_fwd_pp_d<64>(a); }
}  // namespace gbattn
