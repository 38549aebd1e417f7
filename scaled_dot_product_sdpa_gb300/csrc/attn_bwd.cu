// Instantiations and launches of the backward kernels (attn_bwd.cuh): the dQ kernel, then
// the dK/dV kernel, on the caller's stream, each a persistent grid of one CTA per SM
// (programmatic dependent launch: a dK/dV CTA starts on an SM the dQ kernel has left and
// loads its Q, K, V and dO tiles and runs its first products while the dQ kernel finishes;
// only its loads of the row statistics wait until the dQ kernel has completed).
#include "attn_bwd.cuh"

namespace gbattn {

template <int D, bool CAUSAL>
cudaError_t launch_bwd_variant(const BwdLaunch &a) {
  using C = BwdCfg<D>;
  auto *kdkdv = attn_bwd_dkdv_kernel<D, CAUSAL>;
  auto *kdq = attn_bwd_dq_kernel<D, CAUSAL>;
  static int configured_mask = 0;  // one bit per device ordinal < 31
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 31 || !(configured_mask & (1 << dev))) {
    if ((e = cudaFuncSetAttribute(kdkdv, cudaFuncAttributeMaxDynamicSharedMemorySize, C::KV_SMEM)) != cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize, C::Q_SMEM)) != cudaSuccess)
      return e;
    if (dev < 31) configured_mask |= (1 << dev);
  }
  // The dQ kernel first: it writes the row statistics the dK/dV kernel reads.
  e = launch_pdl(kdq, a.grid, C::THREADS, C::Q_SMEM, a.stream, a.tm_q128, a.tm_k128, a.tm_v128, a.tm_do128,
                 a.tm_dq128, a.p);
  if (e != cudaSuccess) return e;
  return launch_pdl(kdkdv, a.grid, C::THREADS, C::KV_SMEM, a.stream, a.tm_q128, a.tm_k128, a.tm_v128, a.tm_do128,
                    a.tm_dk128, a.tm_dv128, a.p);
}

cudaError_t launch_bwd_64(const BwdLaunch &a) {
  return a.causal ? launch_bwd_variant<64, true>(a) : launch_bwd_variant<64, false>(a);
}
cudaError_t launch_bwd_128(const BwdLaunch &a) {
  return a.causal ? launch_bwd_variant<128, true>(a) : launch_bwd_variant<128, false>(a);
}

}  // namespace gbattn
