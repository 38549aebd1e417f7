// debug_kernels.cu -- test hooks of the C ABI.
//
// attn_debug_scores_kernel: the QK stage alone ("no-softmax mode", STAGE_D.md of
//   nvfp4-megamoe-kernel, option 2 of its closing list): S = scale * Q K^T for one
//   128 x 128 tile per CTA, written out as fp32.  The head_dim reduction runs exactly as
//   in the fused kernel: TMA brings 64-column slices of Q and K (128-byte swizzle),
//   tcgen05.mma accumulates every slice into one tensor-memory accumulator, and only then
//   is S read (logits are additive over head_dim sub-tiles, same notes, section 2).
// attn_wait_probe_kernel: waits on a barrier that nothing completes, to show that a
//   bounded wait turns into a readable status instead of a hang.
#include <cuda_runtime.h>

#include "attn_fwd_kernel.cuh"

namespace gbattn {

template <int D>
__global__ void __launch_bounds__(128, 1)
    attn_debug_scores_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                             float *__restrict__ s, int L, int nQ, float scale, unsigned *status,
                             long long limit) {
  constexpr int NCH = D / 64, CHUNK = 128 * 128;
  constexpr uint32_t IDESC = idesc_f16_f32(128, 128, 0, 0);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t qbuf = base, kbuf = base + CHUNK;
  const uint32_t bar_full = base + 2 * CHUNK, bar_mma = bar_full + 8, bar_done = bar_full + 16;
  uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + 2 * CHUNK + 24);
  volatile uint32_t *const abort_flag = tmem_slot + 1;

  const int qt = blockIdx.x / nQ, kt = blockIdx.x - (blockIdx.x / nQ) * nQ, bh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_done, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    int loads = 0, commits = 0;
    bool ok = true;
    for (int c = 0; c < NCH && ok; ++c) {
      if (c > 0 && !(ok = wait_bounded(bar_mma, (c - 1) & 1, abort_flag, status, kDevTimeoutMma, limit))) break;
      mbar_arrive_expect_tx(bar_full, 2 * CHUNK);
      tma_load_3d(qbuf, &tm_q, c * 64, qt * 128, bh, bar_full);
      tma_load_3d(kbuf, &tm_k, c * 64, kt * 128, bh, bar_full);
      ++loads;
      if (!(ok = wait_bounded(bar_full, c & 1, abort_flag, status, kDevTimeoutLoad, limit))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_ss(tmem, sdesc_sw128(qbuf + kk * 32, 16, 1024), sdesc_sw128(kbuf + kk * 32, 16, 1024), IDESC,
                (c | kk) != 0 ? 1u : 0u);
      umma_commit(bar_mma);
      ++commits;
    }
    if (ok) {
      umma_commit(bar_done);
    } else {
      // Drain whatever is still in flight before the CTA may exit.
      if (loads > 0) wait_drain(bar_full, (loads - 1) & 1, limit);
      umma_commit(bar_done);
      wait_drain(bar_done, 0, limit);
    }
  }
  __syncwarp();
  bool ok = wait_bounded(bar_done, 0, abort_flag, status, kDevTimeoutSoftmax, limit);
  ok = __all_sync(0xffffffffu, ok);
  if (ok && !*abort_flag) {
    tc_fence_after();
    uint32_t r[128];
    tmem_ld32x128(tmem + (static_cast<uint32_t>(warp * 32) << 16), r);
    const int grow = qt * 128 + warp * 32 + lane;
    if (grow < L) {
      float *dst = s + (static_cast<long long>(bh) * L + grow) * L + kt * 128;
      const int ncol = min(128, L - kt * 128);
      for (int c = 0; c < ncol; ++c) dst[c] = __uint_as_float(r[c]) * scale;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

__global__ void attn_wait_probe_kernel(unsigned *status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    wait_bounded(smem_u32(&bar), 0, reinterpret_cast<volatile uint32_t *>(&abort_flag), status, kDevTimeoutProbe,
                 limit);
}

constexpr int kDebugSmem = 1024 + 2 * 128 * 128 + 64;

template <int D>
static cudaError_t launch_scores_d(const CUtensorMap &tq, const CUtensorMap &tk, float *s, int BH, int L,
                                   float scale, unsigned *status, long long limit, cudaStream_t st) {
  auto *kern = attn_debug_scores_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDebugSmem);
  if (e != cudaSuccess) return e;
  const int nQ = (L + 127) / 128;
  dim3 grid(nQ * nQ, BH);
  kern<<<grid, 128, kDebugSmem, st>>>(tq, tk, s, L, nQ, scale, status, limit);
  return cudaGetLastError();
}

cudaError_t launch_debug_scores(int d, const CUtensorMap &tq, const CUtensorMap &tk, float *s, int BH, int L,
                                float scale, unsigned *status, long long limit, cudaStream_t st) {
  switch (d) {
    case 64: return launch_scores_d<64>(tq, tk, s, BH, L, scale, status, limit, st);
    case 128: return launch_scores_d<128>(tq, tk, s, BH, L, scale, status, limit, st);
    case 256: return launch_scores_d<256>(tq, tk, s, BH, L, scale, status, limit, st);
    case 512: return launch_scores_d<512>(tq, tk, s, BH, L, scale, status, limit, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_wait_probe(unsigned *status, long long limit, cudaStream_t st) {
  attn_wait_probe_kernel<<<1, 32, 0, st>>>(status, limit);
  return cudaGetLastError();
}

}  // namespace gbattn
