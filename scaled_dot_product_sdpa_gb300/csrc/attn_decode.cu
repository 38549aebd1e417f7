// attn_decode.cu -- the decode kernel (see attn_decode.cuh) and its launches.
//
// `groups` thread-block clusters per head, `ranks` CTAs in each; rank r of group g owns the
// keys [(g ranks + r) keys_per_rank, min(L, (g ranks + r + 1) keys_per_rank)).  A CTA of 256
// threads:
//   - streams its K and V tiles (KT keys each) through a 3-stage ring with TMA, 128-byte
//     swizzled, so that the row reads below spread over all shared-memory banks (two CTAs
//     fit on an SM: one CTA's tile loop, about 1.2 k cycles per 32 KB tile, is bound by its
//     barriers and dependent phases, and the second CTA fills those gaps);
//   - per tile: s_j = c2 q.k_j (base-2 logits), split over TPK threads per key, each
//     holding 32 of q's elements in registers; the tile's maximum; p_j = 2^(s_j - m) with
//     the running maximum m, earlier partial sums scaled by 2^(m_old - m); o += sum_j p_j
//     v_j, each thread owning 8 output columns for 4 of the tile's keys;
//   - at the end reduces its partial (m, l, o) over its threads, writes it into rank 0's
//     shared memory (distributed shared memory) and arrives on rank 0's barrier.
// Rank 0 waits (bounded) for every rank, merges M = max_r m_r, w_r = 2^(m_r - M),
// o = sum_r w_r o_r / sum_r w_r l_r, lse = (M + log2 sum_r w_r l_r) ln 2, and stores them
// (one group per head), or stores o and the base-2 lse as the group's partial in the
// workspace, for attn_decode_merge_kernel (several groups).
// Arithmetic as in the forward kernels: fp16 inputs, fp32 products and sums, 2^x on the
// special-function unit, o rounded to fp16 to nearest even.
#include <cuda_fp16.h>

#include "attn_decode.cuh"
#include "attn_fwd_kernel.cuh"

namespace gbattn {

template <int D>
struct DecCfg {
  static constexpr int NT = 256;                // threads per CTA
  static constexpr int KT = dec_key_tile(D);    // keys per tile: 16 KB of K, 16 KB of V
  static constexpr int NBOX = D / 64;           // 64-column (128-byte) boxes per row
  static constexpr int BOX_BYTES = KT * 128;
  static constexpr int TILE_BYTES = NBOX * BOX_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile, then V tile
  static constexpr int NST = 3;                 // ring stages
  static constexpr int MAXR = dec_max_ranks_for(D);
  static constexpr int TPK = NT / KT;           // threads per key in the QK step
  static constexpr int RT = D / 8;              // threads per value row in the PV step
  static constexpr int KG = NT / RT;            // key groups in the PV step
  static_assert(D / TPK == 32, "QK step: 32 head_dim elements per thread");
  static_assert(KT / KG == 4, "PV step: 4 keys per thread per tile");
  static_assert(KG * D * 4 <= NST * STAGE_BYTES, "the final reduction reuses the ring");
  static constexpr int PART_FLOATS = D + 2;     // o[D], m, l
  static constexpr int OFF_P = NST * STAGE_BYTES;
  static constexpr int OFF_RED = OFF_P + KT * 4;
  static constexpr int OFF_PARTS = OFF_RED + 16 * 4;
  static constexpr int OFF_BAR = OFF_PARTS + MAXR * PART_FLOATS * 4;
  static constexpr int NBAR = NST + 1;          // FULL[NST], PARTS
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + 8 * NBAR + 16;
  static_assert(OFF_BAR % 8 == 0, "barrier alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// 8 fp16 values of a 16-byte vector, as fp32.
__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

template <int D>
__global__ void __launch_bounds__(256, 2)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const DecParams p) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t ring_s = base;
  const uint32_t parts_s = base + C::OFF_PARTS;
  const uint32_t bar_s = base + C::OFF_BAR;
  float *const pbuf = reinterpret_cast<float *>(base_ptr + C::OFF_P);
  float *const red = reinterpret_cast<float *>(base_ptr + C::OFF_RED);
  const float *const parts = reinterpret_cast<const float *>(base_ptr + C::OFF_PARTS);
  volatile uint32_t *const abort_flag = reinterpret_cast<uint32_t *>(base_ptr + C::OFF_BAR + 8 * C::NBAR);
  auto BAR = [&](int i) -> uint32_t { return bar_s + 8u * static_cast<uint32_t>(i); };
  constexpr int B_PARTS = C::NST;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int cl = static_cast<int>(blockIdx.x) / p.ranks;  // cluster
  const int bh = cl / p.groups, grp = cl - bh * p.groups;
  const int k0 = (grp * p.ranks + static_cast<int>(rank)) * p.keys_per_rank;
  const int k1 = min(p.L, k0 + p.keys_per_rank);
  const int ntiles = k1 > k0 ? (k1 - k0 + C::KT - 1) / C::KT : 0;

  if (tid == 0) {
    for (int i = 0; i < C::NST; ++i) mbar_init(BAR(i), 1);
    mbar_init(BAR(B_PARTS), static_cast<uint32_t>(p.ranks));  // arrived on by every rank (used on rank 0)
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  // Every rank's barriers are initialised before any rank arrives on rank 0's.
  cluster_sync_all();
  grid_launch_dependents();
  grid_wait_prior();  // inputs may be the previous kernel's outputs

  // ---------------------------------------------------------------- loads (thread 0)
  int issued = 0;
  auto issue = [&](int i) {
    const uint32_t s = static_cast<uint32_t>(i % C::NST);
    const uint32_t st = ring_s + s * C::STAGE_BYTES;
    mbar_arrive_expect_tx(BAR(s), C::STAGE_BYTES);  // rows past L are zero-filled and counted
    const int y = k0 + i * C::KT;
#pragma unroll
    for (int b = 0; b < C::NBOX; ++b) {
      tma_load_3d(st + b * C::BOX_BYTES, &tm_k, b * 64, y, bh, BAR(s));
      tma_load_3d(st + C::TILE_BYTES + b * C::BOX_BYTES, &tm_v, b * 64, y, bh, BAR(s));
    }
    ++issued;
  };
  if (tid == 0)
    for (int i = 0; i < ntiles && i < C::NST; ++i) issue(i);

  // This thread's share of the QK step: key slot kq of every tile, q elements
  // [part * 32, part * 32 + 32) held in registers.
  const int kq = tid / C::TPK, part = tid % C::TPK;
  float qr[32];
  {
    const uint4 *qg = reinterpret_cast<const uint4 *>(static_cast<const __half *>(p.q) +
                                                      static_cast<size_t>(bh) * D + part * 32);
#pragma unroll
    for (int c = 0; c < 4; ++c) unpack8(qg[c], qr + 8 * c);
  }
  // PV step: columns [cc * 8, cc * 8 + 8) over the keys 4g .. 4g + 3 of every tile.
  const int g = tid / C::RT, cc = tid % C::RT;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  float m = -INFINITY;  // running maximum of the base-2 logits (the same in every thread)
  float lpart = 0.f;    // sum of p over key slot kq (kept by the part-0 thread of each slot)
  bool ok = true;
  int i = 0;
  for (; i < ntiles; ++i) {
    const uint32_t s = static_cast<uint32_t>(i % C::NST);
    const uint32_t st = ring_s + s * C::STAGE_BYTES;
    const bool got = wait_bounded(BAR(s), (i / C::NST) & 1, abort_flag, p.status, kDevTimeoutLoad, p.wait_limit);
    // ---- s = c2 q.k for key slot kq, this thread's 32 elements, then across the TPK threads
    float dot0 = 0.f, dot1 = 0.f;
    if (got) {
      const uint32_t row = st + (part >> 1) * C::BOX_BYTES + kq * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float kf[8];
        unpack8(ld_shared_v4(row + (((((part & 1) << 2) + c) ^ (kq & 7)) << 4)), kf);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          dot0 = fmaf(qr[8 * c + e], kf[e], dot0);
          dot1 = fmaf(qr[8 * c + e + 1], kf[e + 1], dot1);
        }
      }
    }
    float dot = dot0 + dot1;
#pragma unroll
    for (int o = 1; o < C::TPK; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    const int key = k0 + i * C::KT + kq;
    const float sv = key < k1 ? dot * p.c2 : -INFINITY;
    float mx = sv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp] = mx;
    // The previous tile's stage is refilled by TMA (async proxy) after this barrier: order
    // this thread's generic-proxy reads of it before that.
    fence_proxy_async_smem();
    if (__syncthreads_or(!got)) {  // every thread leaves together when a load timed out
      ok = false;
      break;
    }
    float mt = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) mt = fmaxf(mt, red[w]);
    const float m_new = fmaxf(m, mt);     // finite: every tile holds at least one key
    const float alpha = ex2_approx(m - m_new);  // 2^-inf = 0 on the first tile
    m = m_new;
    const float pj = ex2_approx(sv - m_new);    // keys past the range: 2^-inf = 0
    if (part == 0) {
      pbuf[kq] = pj;
      lpart = lpart * alpha + pj;
    }
    // Every thread has finished the previous tile: its stage can be refilled.
    if (tid == 0 && i >= 1 && i - 1 + C::NST < ntiles) issue(i - 1 + C::NST);
    __syncthreads();  // p of this tile is visible
    // ---- o = o * alpha + sum over this thread's 4 keys of p_j v_j[columns]
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= alpha;
    const float4 p4 = *reinterpret_cast<const float4 *>(pbuf + 4 * g);
    const float pk[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int kk = 4 * g + t;
      float vf[8];
      unpack8(ld_shared_v4(st + C::TILE_BYTES + (cc >> 3) * C::BOX_BYTES + kk * 128 + (((cc & 7) ^ (kk & 7)) << 4)),
              vf);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(pk[t], vf[e], acc[e]);
    }
  }
  // Loads issued but never consumed (after a timeout) land before the ring is reused.
  if (tid == 0)
    for (int j = i; j < issued; ++j) wait_drain(BAR(j % C::NST), (j / C::NST) & 1, p.wait_limit);
  __syncthreads();

  // ---------------------------------------------------------------- this rank's partial
  float *const red_o = reinterpret_cast<float *>(base_ptr);  // [KG][D], in the ring
  {
    float4 *dst = reinterpret_cast<float4 *>(red_o + g * D + cc * 8);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  float ls = part == 0 ? lpart : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
  if (lane == 0) red[8 + warp] = ls;
  __syncthreads();
  const uint32_t dst = mapa_shared(parts_s + rank * (C::PART_FLOATS * 4), 0);
  for (int c = tid; c < D; c += C::NT) {
    float o = 0.f;
#pragma unroll 4
    for (int gg = 0; gg < C::KG; ++gg) o += red_o[gg * D + c];
    st_cluster_f32(dst + c * 4, o);
  }
  if (tid == 0) {
    float lt = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) lt += red[8 + w];
    st_cluster_f32(dst + D * 4, m);
    st_cluster_f32(dst + (D + 1) * 4, lt);
  }
  fence_acq_rel_cluster();
  __syncthreads();
  if (tid == 0) mbar_arrive_cluster(mapa_shared(BAR(B_PARTS), 0));

  // ---------------------------------------------------------------- merge (rank 0)
  if (rank != 0) return;
  // A rank that timed out still arrives after at most one more wait limit (and a drain):
  // wait longer than that, so that no rank writes into this CTA after it has exited.
  bool have = mbar_try_acquire_cluster(BAR(B_PARTS), 0);
  if (!have) {
    const long long t0 = clock64(), lim = 3 * p.wait_limit;
    while (!(have = mbar_try_acquire_cluster(BAR(B_PARTS), 0))) {
      if (clock64() - t0 > lim) {
        atomicCAS(p.status, 0u, kDevTimeoutMerge);
        break;
      }
    }
  }
  if (!have || !ok) return;
  float M = -INFINITY;
  for (int r = 0; r < p.ranks; ++r) M = fmaxf(M, parts[r * C::PART_FLOATS + D]);
  float Lsum = 0.f;
  for (int r = 0; r < p.ranks; ++r)
    Lsum += ex2_approx(parts[r * C::PART_FLOATS + D] - M) * parts[r * C::PART_FLOATS + D + 1];
  if (p.groups > 1) {
    // This group's partial: o normalised over the group's keys and its base-2 lse.  A group
    // without keys (M = -inf: every rank's range is empty) writes o = 0, lse = -inf, which
    // the merge weighs 0.
    float *const row = p.ws + static_cast<size_t>(cl) * (D + 2);
    const bool empty = !(M > -INFINITY);
    const float inv = empty ? 0.f : 1.0f / Lsum;
    for (int c = tid; c < D; c += C::NT) {
      float o = 0.f;
      if (!empty)
        for (int r = 0; r < p.ranks; ++r)
          o += ex2_approx(parts[r * C::PART_FLOATS + D] - M) * parts[r * C::PART_FLOATS + c];
      row[c] = o * inv;
    }
    if (tid == 0) row[D] = empty ? -INFINITY : M + __log2f(Lsum);
    return;
  }
  const float inv = 1.0f / Lsum;
  __half *const og = static_cast<__half *>(p.o) + static_cast<size_t>(bh) * D;
  for (int c = tid; c < D; c += C::NT) {
    float o = 0.f;
    for (int r = 0; r < p.ranks; ++r)
      o += ex2_approx(parts[r * C::PART_FLOATS + D] - M) * parts[r * C::PART_FLOATS + c];
    og[c] = __float2half_rn(o * inv);
  }
  if (tid == 0) p.lse[bh] = (M + __log2f(Lsum)) * 0.69314718055994531f;
}

// Merge of the groups' partials, one CTA of D threads per head (launched after the decode
// kernel, whose partials it waits for).
template <int D>
__global__ void __launch_bounds__(D, 1) attn_decode_merge_kernel(const DecParams p) {
  grid_launch_dependents();
  grid_wait_prior();
  const int bh = static_cast<int>(blockIdx.x), c = threadIdx.x;
  const float *const rows = p.ws + static_cast<size_t>(bh) * p.groups * (D + 2);
  float M = -INFINITY;
  for (int g = 0; g < p.groups; ++g) M = fmaxf(M, rows[g * (D + 2) + D]);
  float wsum = 0.f, o = 0.f;
  for (int g = 0; g < p.groups; ++g) {
    const float lg = rows[g * (D + 2) + D];
    if (!(lg > -INFINITY)) continue;  // a group without keys
    const float w = ex2_approx(lg - M);
    wsum += w;
    o += w * rows[g * (D + 2) + c];
  }
  static_cast<__half *>(p.o)[static_cast<size_t>(bh) * D + c] = __float2half_rn(o / wsum);
  if (c == 0) p.lse[bh] = (M + __log2f(wsum)) * 0.69314718055994531f;
}

template <int D>
cudaError_t launch_decode_d(const DecLaunch &a) {
  using C = DecCfg<D>;
  auto *kern = attn_decode_kernel<D>;
  static int configured_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 31 || !(configured_mask & (1 << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    if (dev < 31) configured_mask |= (1 << dev);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.p.BH) * static_cast<unsigned>(a.p.groups * a.p.ranks));
  cfg.blockDim = dim3(C::NT);
  cfg.dynamicSmemBytes = static_cast<size_t>(C::SMEM_BYTES);
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.p.ranks);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, a.tm_k, a.tm_v, a.p);
  if (e != cudaSuccess || a.p.groups == 1) return e;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(static_cast<unsigned>(a.p.BH));
  mcfg.blockDim = dim3(D);
  mcfg.stream = a.stream;
  mcfg.attrs = attr + 1;  // programmatic dependent launch only
  mcfg.numAttrs = 1;
  return cudaLaunchKernelEx(&mcfg, attn_decode_merge_kernel<D>, a.p);
}

// The widest cluster (at most dec_max_ranks_for(D)) the device can run.
template <int D>
int decode_max_ranks_d() {
  using C = DecCfg<D>;
  auto *kern = attn_decode_kernel<D>;
  constexpr int R = C::MAXR;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(R);
  cfg.blockDim = dim3(C::NT);
  cfg.dynamicSmemBytes = static_cast<size_t>(C::SMEM_BYTES);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = R;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return R < 8 ? R : 8;
  }
  return n > 0 ? R : (R < 8 ? R : 8);
}

cudaError_t launch_decode_64(const DecLaunch &a) { return launch_decode_d<64>(a); }
cudaError_t launch_decode_128(const DecLaunch &a) { return launch_decode_d<128>(a); }
cudaError_t launch_decode_256(const DecLaunch &a) { return launch_decode_d<256>(a); }
cudaError_t launch_decode_512(const DecLaunch &a) { return launch_decode_d<512>(a); }

int decode_max_ranks(int d) {
  switch (d) {
    case 64: return decode_max_ranks_d<64>();
    case 128: return decode_max_ranks_d<128>();
    case 256: return decode_max_ranks_d<256>();
    default: return decode_max_ranks_d<512>();
  }
}

}  // namespace gbattn
