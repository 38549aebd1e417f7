// Instantiations and launches of the backward kernels (attn_bwd.cuh): the dK/dV kernel
// and the dQ kernel, one after the other on the caller's stream (the dQ kernel does not
// depend on the first; programmatic dependent launch lets its prologue overlap).
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
  const int items = a.p.BH * a.p.nQ;
  e = launch_pdl(kdkdv, items, 256, C::KV_SMEM, a.stream, a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.tm_do, a.tm_dk, a.tm_dv,
                 a.p);
  if (e != cudaSuccess) return e;
  return launch_pdl(kdq, items, 256, C::Q_SMEM, a.stream, a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.tm_do, a.tm_dq, a.p);
}

cudaError_t launch_bwd_64(const BwdLaunch &a) {
  return a.causal ? launch_bwd_variant<64, true>(a) : launch_bwd_variant<64, false>(a);
}
cudaError_t launch_bwd_128(const BwdLaunch &a) {
  return a.causal ? launch_bwd_variant<128, true>(a) : launch_bwd_variant<128, false>(a);
}

}  // namespace gbattn
