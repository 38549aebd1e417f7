// softmax_tile.cuh -- one online-softmax step over a 128-column S tile held in tensor
// memory, one query row per thread (the softmax stage of "An Optimal Mapper Meets a Real
// GPU", "Experiment one", item (3): a real row max, exponent, sum and divide).
//
// In base 2: with c2 = scale * log2(e), the running maximum m (log2 units) and the
// running sum l satisfy, after every tile,
//     l = sum_j 2^(s_j * c2 - m)   over the keys seen so far,
// and O (in tensor memory) = sum_j 2^(s_j * c2 - m) v_j.  m is raised lazily: only when a
// tile's maximum exceeds it by more than 8 (a factor 256, harmless in fp16 P and fp32
// sums); then O and l are multiplied by 2^(m_old - m_new).  The final O / l and
// LSE = (m + log2 l) * ln 2 do not depend on when m was raised.
//
// Latency, not arithmetic, bounds this step (one warp per scheduler per Q tile), so:
// both halves of S are read with one wait; the max uses eight independent chains of
// three-input max; s * c2 - m uses packed f32x2 FMA; the row sum uses four packed f32x2
// partial sums; the first half of P is stored while the second half is computed.
#pragma once

#include "ptx.cuh"

namespace gbattn {

// s_tmem / o_tmem: this warp's lane base plus the S / O column.  Columns >= lim are
// masked to -inf (lim = row + 1 on a causal diagonal tile, L - first key on a ragged last
// tile, 128 otherwise).  P (fp16) is written over the first 64 columns of the S tile.
// Warp-collective (tcgen05.ld/st): all 32 lanes must call it together.
// `before_rescale()` runs only when this warp rescales O (a tile but the first whose
// maximum exceeds the running one by more than 8), before O is touched: a caller whose
// PV into O may still be in flight waits for it there.  If it returns false the step
// stops and returns false.  It returns whether it ran through `rescaled`.
struct NoWait {
  __device__ bool operator()() const { return true; }
};
// The step on a row of S already in registers (ra: columns 0-63, rb: 64-127, fp32 bits);
// P still goes to s_tmem.
template <int DV, class Hook = NoWait>
__device__ __forceinline__ bool softmax_regs(uint32_t (&ra)[64], uint32_t (&rb)[64], uint32_t s_tmem,
                                             uint32_t o_tmem, int lim, float c2, bool first, float &m_used,
                                             float &l, const Hook &before_rescale = Hook(),
                                             bool *rescaled = nullptr) {
  float *sa = reinterpret_cast<float *>(ra);
  if (lim < 64) {
#pragma unroll
    for (int c = 0; c < 64; ++c)
      if (c >= lim) sa[c] = -INFINITY;
  }
  float mk[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    mk[k] = fmax3(sa[8 * k], sa[8 * k + 1], sa[8 * k + 2]);
    mk[k] = fmax3(mk[k], sa[8 * k + 3], sa[8 * k + 4]);
    mk[k] = fmax3(mk[k], sa[8 * k + 5], sa[8 * k + 6]);
    mk[k] = fmaxf(mk[k], sa[8 * k + 7]);
  }
  float *sb = reinterpret_cast<float *>(rb);
  if (lim < 128) {
#pragma unroll
    for (int c = 0; c < 64; ++c)
      if (c + 64 >= lim) sb[c] = -INFINITY;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    mk[k] = fmax3(mk[k], sb[8 * k], sb[8 * k + 1]);
    mk[k] = fmax3(mk[k], sb[8 * k + 2], sb[8 * k + 3]);
    mk[k] = fmax3(mk[k], sb[8 * k + 4], sb[8 * k + 5]);
    mk[k] = fmax3(mk[k], sb[8 * k + 6], sb[8 * k + 7]);
  }
  const float mx = fmax3(fmax3(mk[0], mk[1], mk[2]), fmax3(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
  const float m_tile = mx * c2;
  if (rescaled) *rescaled = false;
  if (first) {
    m_used = (m_tile == -INFINITY) ? 0.f : m_tile;
    l = 0.f;
  } else if (__any_sync(0xffffffffu, m_tile > m_used + 8.0f)) {
    if (rescaled) *rescaled = true;
    if (!before_rescale()) return false;  // no PV into O may be in flight from here on
    const float m_new = fmaxf(m_used, m_tile);
    const float alpha = ex2_approx(m_used - m_new);
    m_used = m_new;
    l *= alpha;
#pragma unroll 1
    for (int c32 = 0; c32 < DV / 32; ++c32) {
      uint32_t orr[32];
      tmem_ld32x32(o_tmem + c32 * 32, orr);
#pragma unroll
      for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
      tmem_st32x32(o_tmem + c32 * 32, orr);
    }
  }
  const uint64_t c2x2 = f32x2(c2, c2), negm = f32x2(-m_used, -m_used);
  uint64_t acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = f32x2(0.f, 0.f);
  // P in two halves: the first half's store is in flight while the second is computed.
  uint32_t pa[32], pb[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    float x0, x1;
    f32x2_split(ffma2(f32x2(sa[2 * c], sa[2 * c + 1]), c2x2, negm), x0, x1);
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    acc[c & 3] = fadd2(acc[c & 3], f32x2(p0, p1));
    pa[c] = pack_f16x2(p0, p1);
  }
  tmem_st32x32_async(s_tmem, pa);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    float x0, x1;
    f32x2_split(ffma2(f32x2(sb[2 * c], sb[2 * c + 1]), c2x2, negm), x0, x1);
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    acc[c & 3] = fadd2(acc[c & 3], f32x2(p0, p1));
    pb[c] = pack_f16x2(p0, p1);
  }
  tmem_st32x32_async(s_tmem + 32, pb);
  const uint64_t s01 = fadd2(acc[0], acc[1]), s23 = fadd2(acc[2], acc[3]);
  float lo, hi;
  f32x2_split(fadd2(s01, s23), lo, hi);
  l += lo + hi;
  tmem_wait_st_fence32(pa);
  tmem_wait_st_fence32(pb);
  return true;
}

// Epilogue of one query row: O / l as fp16 into the swizzled staging tile of the TMA store
// (64-column chunks of 128-byte rows, CHUNK bytes apart; the 16-byte pieces of a row are
// XOR-swizzled by row & 7).  128 columns of O are loaded from tensor memory with both
// loads in flight and one wait, so the loads' latencies overlap.
template <int DV>
__device__ __forceinline__ void stage_o_row(uint32_t o_tmem, uint32_t stage, int row, float inv_l) {
  constexpr int CHUNK = 128 * 128;
  auto put64 = [&](const uint32_t (&r)[64], int chunk64) {
    const uint32_t rowaddr = stage + chunk64 * CHUNK + row * 128;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint32_t h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        h[i] = pack_f16x2(__uint_as_float(r[8 * q + 2 * i]) * inv_l, __uint_as_float(r[8 * q + 2 * i + 1]) * inv_l);
      st_shared_v4(rowaddr + ((q ^ (row & 7)) << 4), h[0], h[1], h[2], h[3]);
    }
  };
#pragma unroll 1
  for (int c = 0; c < DV; c += 128) {
    uint32_t a[64], b[64];
    tmem_ld32x64_async(o_tmem + c, a);
    if constexpr (DV > 64) tmem_ld32x64_async(o_tmem + c + 64, b);
    tmem_wait_ld_fence64(a);
    if constexpr (DV > 64) tmem_wait_ld_fence64(b);
    put64(a, c / 64);
    if constexpr (DV > 64) put64(b, c / 64 + 1);
  }
}

// fp16x2 -> two fp32 (low half first), exact.
__device__ __forceinline__ void unpack_f16x2(uint32_t v, float &lo, float &hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(v));
}

// Epilogue of one query row of a query tile whose keys two CTAs shared: out = w_own * O
// (this CTA's unnormalised accumulator in tensor memory) + w_peer * O_peer (the other
// CTA's partial, normalised, fp16, in the staging layout at `recv`), as fp16 into the
// staging tile.  The weights carry the merge over the two disjoint key ranges.
template <int DV>
__device__ __forceinline__ void merge_o_row(uint32_t o_tmem, uint32_t recv, uint32_t stage, int row, float w_own,
                                            float w_peer) {
  constexpr int CHUNK = 128 * 128;
  auto put64 = [&](const uint32_t (&r)[64], int chunk64) {
    const uint32_t off = chunk64 * CHUNK + row * 128;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t sw = (q ^ (row & 7)) << 4;
      const uint4 x = ld_shared_v4(recv + off + sw);
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
      uint32_t h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a, b;
        unpack_f16x2(xs[i], a, b);
        h[i] = pack_f16x2(fmaf(w_own, __uint_as_float(r[8 * q + 2 * i]), w_peer * a),
                          fmaf(w_own, __uint_as_float(r[8 * q + 2 * i + 1]), w_peer * b));
      }
      st_shared_v4(stage + off + sw, h[0], h[1], h[2], h[3]);
    }
  };
#pragma unroll 1
  for (int c = 0; c < DV; c += 128) {
    uint32_t a[64], b[64];
    tmem_ld32x64_async(o_tmem + c, a);
    if constexpr (DV > 64) tmem_ld32x64_async(o_tmem + c + 64, b);
    tmem_wait_ld_fence64(a);
    if constexpr (DV > 64) tmem_wait_ld_fence64(b);
    put64(a, c / 64);
    if constexpr (DV > 64) put64(b, c / 64 + 1);
  }
}

template <int DV, class Hook = NoWait>
__device__ __forceinline__ bool softmax_tile(uint32_t s_tmem, uint32_t o_tmem, int lim, float c2, bool first,
                                             float &m_used, float &l, const Hook &before_rescale = Hook(),
                                             bool *rescaled = nullptr) {
  uint32_t ra[64], rb[64];
  // Both halves of S in flight at once, then one wait.
  tmem_ld32x64_async(s_tmem, ra);
  tmem_ld32x64_async(s_tmem + 64, rb);
  tmem_wait_ld_fence64(ra);
  tmem_wait_ld_fence64(rb);
  return softmax_regs<DV>(ra, rb, s_tmem, o_tmem, lim, c2, first, m_used, l, before_rescale, rescaled);
}

}  // namespace gbattn
