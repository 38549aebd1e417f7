// attn_bwd.cuh -- SDPA backward pass on sm_103a: dQ, dK, dV for an upstream gradient dO.
//
// What it computes ("Validating Memory-Optimal Transformer Kernels on Real Hardware",
// section 4, "Paper II: Backward Pass and Fused Forward+Backward": the gradients GQ, GK,
// GV of the attention output through the score gradient GS), per head, with the forward
// pass's row LSE (natural log) and output O:
//     P_ij  = exp(scale q_i.k_j - LSE_i)          (0 where the causal mask hides j > i)
//     D_i   = dO_i . O_i                          (= sum_j P_ij dP_ij)
//     dV_j  = sum_i P_ij dO_i
//     dP_ij = dO_i . v_j
//     dS_ij = P_ij (dP_ij - D_i)
//     dK_j  = scale sum_i dS_ij q_i,     dQ_i = scale sum_j dS_ij k_j
// The page's GPU finding is that the atomic accumulations of GK / GV cost more than they
// save; here no atomics are used at all: two kernels, one per output side, run in this
// order:
//
//   attn_bwd_dq_kernel: work item = (head, 128-query tile i), Q_i, dO_i and O_i resident,
//     the key rows streamed in 64-row tiles j:  S = Q_i K_j^T and dP = dO_i V_j^T on the
//     tensor core; dS is formed; then dQ_i += dS K_j.  It also forms the row statistics
//     LSE_i log2(e) and D_i = dO_i . O_i of its tile and writes them to a workspace of
//     8 bytes per query row (the only memory beyond the inputs and outputs).
//   attn_bwd_dkdv_kernel: work item = (head, 128-key tile j), K_j and V_j resident, the
//     query rows streamed in 64-row tiles i together with their row statistics:
//     S^T = K_j Q_i^T and dP^T = V_j dO_i^T; P^T and dS^T are formed in fp16 over the
//     same tensor-memory columns; then dV_j += P^T dO_i and dK_j += dS^T Q_i.
// Both recompute P from the forward LSE (no L x L matrix is stored).  The tensor-core
// operand forms are the forward kernels': K-major A and B from shared memory for the
// logit-like products (N = 64), A from tensor memory with an MN-major B for the
// accumulations (N = head_dim).
//
// Pipelining: S and dP are double-buffered in tensor memory, so the tensor core computes
// step s+1's S and dP while the elementwise warps work on step s; the streamed tiles sit
// in a ring deep enough (4 stages at head_dim 128, 8 at 64) for the loads to run two steps
// ahead.  Both kernels are persistent: one CTA per SM walks the items longest first, in
// "snake" order (CTA b takes items b, 2G-1-b, 2G+b, ... of the sorted list, G = grid size),
// so that the per-CTA totals even out.  The epilogue writes the accumulators from tensor
// memory straight to global memory (each thread one row), so the next item's loads are
// not held up by a staging buffer.
//
// Warp roles (384 threads): warp 0 TMA producer; warp 1 tensor-memory owner and MMA
// issuer; warps 2-3 the row statistics (dQ kernel only; idle in the other); warps 4-7 and
// 8-11 two elementwise warpgroups, each taking one half of the 64 columns of every S / dP
// tile, and the epilogue.
// Every wait is bounded (about two seconds of SM clock), as in the forward kernels.
#pragma once

#include <cuda_fp16.h>

#include "attn_fwd_kernel.cuh"

namespace gbattn {

struct BwdParams {
  const float *lse;        // [BH, L] forward LSE (natural log)
  __half *dq, *dk, *dv;    // [BH, L, D] outputs
  float *ws_lse2, *ws_d;   // workspace [BH, Lp] each: LSE log2(e) (+inf past L) and D
  unsigned *status;
  long long wait_limit;
  int BH, L;
  int Lp;                  // L rounded up to a multiple of 128 (workspace row stride)
  int n128, n64;           // ceil(L / 128), ceil(L / 64)
  int items;               // BH * n128 work items per kernel
  float c2;                // scale * log2(e)
  float scale;
};

struct BwdLaunch {
  // Resident operands use 128-row boxes, streamed operands 64-row boxes.
  CUtensorMap tm_q128, tm_do128, tm_o128, tm_k128, tm_v128, tm_q64, tm_do64, tm_k64, tm_v64;
  BwdParams p;
  int grid;  // persistent CTAs (<= items)
  bool causal;
  cudaStream_t stream;
};

template <int D>
struct BwdCfg {
  static constexpr int THREADS = 384;
  static constexpr int NCH = D / 64;                  // 64-column chunks of a tile
  static constexpr int RCHUNK = 128 * 128;            // resident tile: 128 rows x 64 fp16 columns
  static constexpr int RTILE = NCH * RCHUNK;
  static constexpr int SCHUNK = 64 * 128;             // streamed tile: 64 rows x 64 fp16 columns
  static constexpr int STILE = NCH * SCHUNK;
  static constexpr int NS = D == 64 ? 8 : 4;          // ring stages
  static constexpr uint32_t IDESC_S = idesc_f16_f32(128, 64, 0, 0);    // 128 x 64 logit-like
  static constexpr uint32_t IDESC_ACC = idesc_f16_f32(128, D, 0, 1);   // B MN-major, N = D
  static constexpr int TMEM_COLS = 512;
  // dK/dV kernel: [K][V][ring: NS x stage][barriers]; a stage is [Q][dO][LSE log2 e: 64 fp32]
  // [D: 64 fp32][pad to 1 KB] (the next stage's tiles stay 1 KB aligned for the swizzle).
  static constexpr int ST_OFF = 2 * STILE;
  static constexpr int STAGE = 2 * STILE + 1024;
  static constexpr int KV_OFF_RING = 2 * RTILE;
  static constexpr int KV_OFF_BAR = KV_OFF_RING + NS * STAGE;
  static constexpr int KB_KVFULL = 0, KB_IDONE = 1, KB_FULL = 2, KB_EMPTY = 2 + NS, KB_SFULL = 2 + 2 * NS,
                       KB_DPFULL = KB_SFULL + 2, KB_PFULL = KB_DPFULL + 2, KB_DSFULL = KB_PFULL + 2,
                       KB_KVFREE = KB_DSFULL + 2, KB_DRAIN = KB_KVFREE + 1, KB_N = KB_DRAIN + 1;
  static constexpr int KV_SMEM = 1024 + KV_OFF_BAR + 8 * KB_N + 16;
  // dQ kernel: [Q][dO][O][ring: NS x (K, V)][row stats: lse 128 | D 128 fp32][barriers]
  static constexpr int Q_OFF_RING = 3 * RTILE;
  static constexpr int Q_OFF_ST = Q_OFF_RING + NS * 2 * STILE;
  static constexpr int Q_OFF_BAR = Q_OFF_ST + 256 * 4;
  static constexpr int QB_QFULL = 0, QB_IDONE = 1, QB_RFULL = 2, QB_FULL = 3, QB_EMPTY = 3 + NS,
                       QB_SFULL = 3 + 2 * NS, QB_DPFULL = QB_SFULL + 2, QB_DSFULL = QB_DPFULL + 2,
                       QB_QFREE = QB_DSFULL + 2, QB_DRAIN = QB_QFREE + 1, QB_N = QB_DRAIN + 1;
  // QFREE: the item's Q, dO and O buffers may be refilled: the MMA warp's commit after its
  // last S and dP products, every statistics thread (done reading dO and O) and every
  // elementwise thread (done reading the statistics).
  static constexpr int QFREE_COUNT = 1 + 64 + 256;
  static constexpr int Q_SMEM = 1024 + Q_OFF_BAR + 8 * QB_N + 16;
  static_assert(KV_SMEM <= 232448 && Q_SMEM <= 232448, "shared memory budget");
  static_assert(256 + 2 * D <= TMEM_COLS, "tensor memory budget");
};

// Shared-memory address of 16-byte chunk c (8 fp16 values) of row r of a tile loaded by
// TMA with the 128-byte swizzle in 64-column boxes of `chunk` bytes each.
__device__ __forceinline__ uint32_t bwd_chunk_addr(uint32_t tile, int chunk, int r, int c) {
  return tile + (c >> 3) * chunk + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Item index of round r for CTA b of G (snake order over the longest-first list).
__device__ __forceinline__ int bwd_item(int r, int b, int G) { return r * G + ((r & 1) ? G - 1 - b : b); }

// Tensor-memory column offset of k-step kk (16 of the 64 reduction rows) of a P^T / dS^T /
// dS operand: the warpgroup of column half h packs its 32 columns into [32 h, 32 h + 16).
__device__ __forceinline__ uint32_t bwd_a_col(int kk) {
  return static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8);
}

// Sum of the 8 fp16 products of two 16-byte chunks (fp32).
__device__ __forceinline__ float bwd_dot8(uint4 a, uint4 b) {
  const uint32_t as[4] = {a.x, a.y, a.z, a.w}, bs[4] = {b.x, b.y, b.z, b.w};
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&as[h]));
    const float2 y = __half22float2(*reinterpret_cast<const __half2 *>(&bs[h]));
    acc0 = fmaf(x.x, y.x, acc0);
    acc1 = fmaf(x.y, y.y, acc1);
  }
  return acc0 + acc1;
}

// LSE of rows row0 + lane and row0 + 32 + lane of the 128-row query tile at query q0
// (+inf past L), for bwd_row_stats; loaded ahead of the tile's shared-memory work.
__device__ __forceinline__ void bwd_row_lse(const BwdParams &p, int bh, int q0, int row0, int lane, float (&l)[2]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int qrow = q0 + row0 + 32 * i + lane;
    l[i] = qrow < p.L ? __ldg(p.lse + static_cast<long long>(bh) * p.L + qrow) : INFINITY;
  }
}

// Row statistics of rows [row0, row0 + 64) of the 128-row query tile at query q0 (one
// warp; lane l takes rows row0 + l and row0 + 32 + l), from their LSE (bwd_row_lse) and
// the swizzled dO and O tiles in shared memory: stat[r] = LSE_r log2(e) (+inf past L, so
// that P = 0 there) and stat[128 + r] = D_r = dO_r . O_r, also written to the workspace
// (row r of the padded [BH, Lp] layout).
template <int D>
__device__ __forceinline__ void bwd_row_stats(const BwdParams &p, int bh, int q0, uint32_t do_tile, uint32_t o_tile,
                                              float *stat, int row0, int lane, const float (&lse)[2]) {
  constexpr int CH = BwdCfg<D>::RCHUNK;
  constexpr float kLog2e = 1.4426950408889634f;
  const long long wrow0 = static_cast<long long>(bh) * p.Lp + q0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int row = row0 + 32 * i + lane;
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; c += 2) {
      acc0 += bwd_dot8(ld_shared_v4(bwd_chunk_addr(do_tile, CH, row, c)),
                       ld_shared_v4(bwd_chunk_addr(o_tile, CH, row, c)));
      acc1 += bwd_dot8(ld_shared_v4(bwd_chunk_addr(do_tile, CH, row, c + 1)),
                       ld_shared_v4(bwd_chunk_addr(o_tile, CH, row, c + 1)));
    }
    const float dd = acc0 + acc1, ls = lse[i] * kLog2e;
    stat[row] = ls;
    stat[128 + row] = dd;
    p.ws_lse2[wrow0 + row] = ls;
    p.ws_d[wrow0 + row] = dd;
  }
}

// Epilogue: NC columns of an fp32 accumulator row in tensor memory, times `mult`, to fp16
// at `dst` (row-contiguous, 16-byte aligned).  The loads are warp-collective; the stores
// happen only where `store`.
template <int NC>
__device__ __forceinline__ void bwd_store_row(uint32_t acc_tmem, __half *dst, float mult, bool store) {
#pragma unroll 1
  for (int c32 = 0; c32 < NC / 32; ++c32) {
    uint32_t r[32];
    tmem_ld32x32(acc_tmem + c32 * 32, r);
    uint32_t h[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) h[i] = pack_f16x2(__uint_as_float(r[2 * i]) * mult, __uint_as_float(r[2 * i + 1]) * mult);
    if (store) {
      uint4 *out = reinterpret_cast<uint4 *>(dst + c32 * 32);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) out[q4] = make_uint4(h[4 * q4], h[4 * q4 + 1], h[4 * q4 + 2], h[4 * q4 + 3]);
    }
  }
}

// ======================================================================== dK / dV
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t k_s = base, v_s = base + C::RTILE, ring_s = base + C::KV_OFF_RING;
  const uint32_t bar_s = base + C::KV_OFF_BAR;
  uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + C::KV_OFF_BAR + 8 * C::KB_N);
  volatile uint32_t *const abort_flag = tmem_slot + 1;
  auto BAR = [&](int i) -> uint32_t { return bar_s + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long LIM = p.wait_limit;
  const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  // Item idx: key tile kt of head bh (kt ascending = longest first when causal); its steps
  // are the 64-row query tiles from q_first on.
  auto decode = [&](int idx, int &bh, int &kt, int &q_first, int &nsteps) {
    kt = idx / p.BH;
    bh = idx - kt * p.BH;
    q_first = CAUSAL ? 2 * kt : 0;
    nsteps = p.n64 - q_first;
  };
  auto stage_addr = [&](int gg) -> uint32_t { return ring_s + (gg % C::NS) * C::STAGE; };

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::KB_KVFULL), 1);
    mbar_init(BAR(C::KB_IDONE), 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(BAR(C::KB_FULL + i), 1);
      mbar_init(BAR(C::KB_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(C::KB_SFULL + i), 1);
      mbar_init(BAR(C::KB_DPFULL + i), 1);
      mbar_init(BAR(C::KB_PFULL + i), 256);
      mbar_init(BAR(C::KB_DSFULL + i), 256);
    }
    mbar_init(BAR(C::KB_KVFREE), 1);
    mbar_init(BAR(C::KB_DRAIN), 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_launch_dependents();
  grid_wait_prior();
  // Tensor memory: step buffer b (= global step & 1) holds S^T at [128 b, 128 b + 64) (P^T
  // packed over its first 16 columns of each 32-column half) and dP^T at [128 b + 64,
  // 128 b + 128) (dS^T likewise); dV [256, 256+D), dK [256+D, 256+2D).
  constexpr uint32_t C_DV = 256, C_DK = 256 + D;
  auto c_s = [](int gg) -> uint32_t { return static_cast<uint32_t>(gg & 1) * 128u; };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int g = 0, issued = 0, kv_loads = 0;
      for (int r = 0; ok && r * G < p.items; ++r) {
        const int idx = bwd_item(r, cta, G);
        if (idx >= p.items) continue;
        int bh, kt, q_first, nsteps;
        decode(idx, bh, kt, q_first, nsteps);
        for (int s = 0; s < nsteps; ++s, ++g) {
          const int st = g % C::NS;
          if (!(ok = wait_bounded(BAR(C::KB_EMPTY + st), ((g / C::NS) & 1) ^ 1u, abort_flag, p.status, kDevTimeoutLoad,
                                  LIM)))
            break;
          const uint32_t stage = stage_addr(g);
          const long long wrow = static_cast<long long>(bh) * p.Lp + (q_first + s) * 64;
          mbar_arrive_expect_tx(BAR(C::KB_FULL + st), 2 * C::STILE + 512);
          for (int c = 0; c < C::NCH; ++c) {
            tma_load_3d(stage + c * C::SCHUNK, &tm_q, c * 64, (q_first + s) * 64, bh, BAR(C::KB_FULL + st));
            tma_load_3d(stage + C::STILE + c * C::SCHUNK, &tm_do, c * 64, (q_first + s) * 64, bh, BAR(C::KB_FULL + st));
          }
          // The 64 rows' statistics, written by the dQ kernel (byte offsets multiples of 256).
          bulk_load(stage + C::ST_OFF, p.ws_lse2 + wrow, 256, BAR(C::KB_FULL + st));
          bulk_load(stage + C::ST_OFF + 256, p.ws_d + wrow, 256, BAR(C::KB_FULL + st));
          ++issued;
          if (s == 0) {
            // K and V of this item, once the previous item's last S^T and dP^T products (the
            // only readers of K and V) are complete: up to two steps before that item ends.
            if (kv_loads > 0 && !(ok = wait_bounded(BAR(C::KB_KVFREE), (kv_loads - 1) & 1, abort_flag, p.status,
                                                    kDevTimeoutLoad, LIM)))
              break;
            mbar_arrive_expect_tx(BAR(C::KB_KVFULL), 2 * C::RTILE);
            for (int c = 0; c < C::NCH; ++c) {
              tma_load_3d(k_s + c * C::RCHUNK, &tm_k, c * 64, kt * 128, bh, BAR(C::KB_KVFULL));
              tma_load_3d(v_s + c * C::RCHUNK, &tm_v, c * 64, kt * 128, bh, BAR(C::KB_KVFULL));
            }
            ++kv_loads;
          }
        }
      }
      // Drain: every load issued lands before the CTA may exit.
      if (kv_loads > 0) wait_drain(BAR(C::KB_KVFULL), (kv_loads - 1) & 1, LIM);
      for (int s = issued > C::NS ? issued - C::NS : 0; s < issued; ++s)
        wait_drain(BAR(C::KB_FULL + s % C::NS), (s / C::NS) & 1, LIM);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      int g = 0, it = 0;
      auto wait = [&](int b, uint32_t ph) -> bool {
        return wait_bounded(BAR(b), ph, abort_flag, p.status, kDevTimeoutMma, LIM);
      };
      const SDesc ka = sdesc_split(sdesc_sw128(k_s, 16, 1024)), va = sdesc_split(sdesc_sw128(v_s, 16, 1024));
      // S^T = K Q^T and dP^T = V dO^T of global step gg into its buffer (head_dim summed
      // over its 64-column chunks).
      auto issue_sdp = [&](int gg) {
        const uint32_t stage = stage_addr(gg);
        const SDesc qb = sdesc_split(sdesc_sw128(stage, 16, 1024));
        const SDesc dob = sdesc_split(sdesc_sw128(stage + C::STILE, 16, 1024));
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + c_s(gg), ka, c * C::RCHUNK + kk * 32, qb, c * C::SCHUNK + kk * 32, C::IDESC_S,
                        (c | kk) != 0 ? 1u : 0u);
        umma_commit(BAR(C::KB_SFULL + (gg & 1)));
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + c_s(gg) + 64, va, c * C::RCHUNK + kk * 32, dob, c * C::SCHUNK + kk * 32, C::IDESC_S,
                        (c | kk) != 0 ? 1u : 0u);
        umma_commit(BAR(C::KB_DPFULL + (gg & 1)));
      };
      auto stage_ready = [&](int gg) { return wait(C::KB_FULL + gg % C::NS, (gg / C::NS) & 1); };
      for (int r = 0; ok && r * G < p.items; ++r) {
        const int idx = bwd_item(r, cta, G);
        if (idx >= p.items) continue;
        int bh, kt, q_first, nsteps;
        decode(idx, bh, kt, q_first, nsteps);
        if (!(ok = wait(C::KB_KVFULL, it & 1) && stage_ready(g))) break;
        tc_fence_after();
        issue_sdp(g);
        if (nsteps > 1) {
          if (!(ok = stage_ready(g + 1))) break;
          tc_fence_after();
          issue_sdp(g + 1);
        }
        if (nsteps <= 2) umma_commit(BAR(C::KB_KVFREE));  // the item's last S^T, dP^T are issued
        for (int s = 0; s < nsteps; ++s, ++g) {
          const uint32_t stage = stage_addr(g);
          const uint32_t pb = (static_cast<uint32_t>(g) >> 1) & 1u;
          // dV += P^T dO
          if (!(ok = wait(C::KB_PFULL + (g & 1), pb))) break;
          tc_fence_after();
          const SDesc dom = sdesc_split(sdesc_sw128(stage + C::STILE, C::SCHUNK, 1024));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ts_off(tmem + C_DV, tmem + c_s(g) + bwd_a_col(kk), dom, kk * 2048, C::IDESC_ACC,
                        (s > 0 || kk > 0) ? 1u : 0u);
          // dK += dS^T Q
          if (!(ok = wait(C::KB_DSFULL + (g & 1), pb))) break;
          tc_fence_after();
          const SDesc qm = sdesc_split(sdesc_sw128(stage, C::SCHUNK, 1024));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ts_off(tmem + C_DK, tmem + c_s(g) + 64 + bwd_a_col(kk), qm, kk * 2048, C::IDESC_ACC,
                        (s > 0 || kk > 0) ? 1u : 0u);
          umma_commit(BAR(C::KB_EMPTY + g % C::NS));
          if (s + 2 < nsteps) {
            if (!(ok = stage_ready(g + 2))) break;
            tc_fence_after();
            issue_sdp(g + 2);  // into this step's buffers, read in order after dV, dK above
            if (s + 3 == nsteps) umma_commit(BAR(C::KB_KVFREE));
          }
        }
        if (!ok) break;
        umma_commit(BAR(C::KB_IDONE));  // K, V free; dV, dK final
        ++it;
      }
      umma_commit(BAR(C::KB_DRAIN));  // every MMA issued so far is complete
      wait_drain(BAR(C::KB_DRAIN), 0, LIM);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ elementwise warpgroups
    const int h = (warp - 4) >> 2;        // query columns [32 h, 32 h + 32) of every tile
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row of the tile == tensor-memory lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.c2;
    auto wait_warp = [&](int b, uint32_t ph) -> bool {
      return __all_sync(0xffffffffu, wait_bounded(BAR(b), ph, abort_flag, p.status, kDevTimeoutSoftmax, LIM));
    };
    bool ok = true;
    int g = 0, it = 0;
    for (int r = 0; ok && r * G < p.items; ++r) {
      const int idx = bwd_item(r, cta, G);
      if (idx >= p.items) continue;
      int bh, kt, q_first, nsteps;
      decode(idx, bh, kt, q_first, nsteps);
      for (int s = 0; s < nsteps; ++s, ++g) {
        const int st = g % C::NS;
        const uint32_t pb = (static_cast<uint32_t>(g) >> 1) & 1u;
        const uint32_t s_col = tmem + lane_base + c_s(g) + 32 * h, dp_col = s_col + 64;
        const float *const lse_h = reinterpret_cast<const float *>(base_ptr + (stage_addr(g) - base) + C::ST_OFF) + 32 * h;
        const float *const dd_h = lse_h + 64;
        // The stage (its statistics included) has landed: the S^T of this step is computed from it.
        if (!(ok = wait_warp(C::KB_SFULL + (g & 1), pb) && wait_warp(C::KB_FULL + st, (g / C::NS) & 1))) break;
        tc_fence_after();
        // P phase: P^T = exp2(S^T c2 - LSE log2 e), masked on the two diagonal query tiles
        // (query before key), packed to fp16 into the first 16 of its 32 columns.
        const bool diag = CAUSAL && s < 2;
        float pv[32];
        {
          uint32_t sr[32];
          tmem_ld32x32(s_col, sr);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            float pp = ex2_approx(fmaf(__uint_as_float(sr[c]), c2, -lse_h[c]));
            if (diag && s * 64 + 32 * h + c < row) pp = 0.f;
            pv[c] = pp;
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack_f16x2(pv[2 * i], pv[2 * i + 1]);
          tmem_st32x16(s_col, pk);
        }
        tc_fence_before();
        mbar_arrive(BAR(C::KB_PFULL + (g & 1)));
        // dS phase: dS^T = P^T (dP^T - D), packed likewise.
        if (!(ok = wait_warp(C::KB_DPFULL + (g & 1), pb))) break;
        tc_fence_after();
        {
          uint32_t dr[32];
          tmem_ld32x32(dp_col, dr);
          uint32_t dk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            dk[i] = pack_f16x2(pv[2 * i] * (__uint_as_float(dr[2 * i]) - dd_h[2 * i]),
                               pv[2 * i + 1] * (__uint_as_float(dr[2 * i + 1]) - dd_h[2 * i + 1]));
          tmem_st32x16(dp_col, dk);
        }
        tc_fence_before();
        // The statistics read above sit in a stage that TMA refills once it is released.
        fence_proxy_async_smem();
        mbar_arrive(BAR(C::KB_DSFULL + (g & 1)));
      }
      if (!ok) break;
      // ---------------------------------------------------------------- epilogue
      // Warpgroup 0 writes dV, warpgroup 1 writes scale * dK, one key row per thread.
      if (!(ok = wait_warp(C::KB_IDONE, it & 1))) break;
      tc_fence_after();
      const int krow = kt * 128 + row;
      __half *const dst = (h == 0 ? p.dv : p.dk) + (static_cast<long long>(bh) * p.L + krow) * D;
      bwd_store_row<D>(tmem + lane_base + (h == 0 ? C_DV : C_DK), dst, h == 0 ? 1.0f : p.scale,
                       krow < p.L && *abort_flag == 0u);
      tc_fence_before();
      ++it;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ======================================================================== dQ
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_o, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t q_s = base, do_s = base + C::RTILE, o_s = base + 2 * C::RTILE, ring_s = base + C::Q_OFF_RING;
  float *const stat_s = reinterpret_cast<float *>(base_ptr + C::Q_OFF_ST);  // [lse 128 | D 128]
  const uint32_t bar_s = base + C::Q_OFF_BAR;
  uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + C::Q_OFF_BAR + 8 * C::QB_N);
  volatile uint32_t *const abort_flag = tmem_slot + 1;
  auto BAR = [&](int i) -> uint32_t { return bar_s + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long LIM = p.wait_limit;
  const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  // Item idx: query tile qt of head bh, longest first (causal: the last query tiles see the
  // most key tiles); its steps are the 64-row key tiles 0 .. nsteps-1.
  auto decode = [&](int idx, int &bh, int &qt, int &nsteps) {
    const int grp = idx / p.BH;
    bh = idx - grp * p.BH;
    qt = CAUSAL ? p.n128 - 1 - grp : grp;
    nsteps = CAUSAL ? min(p.n64, 2 * qt + 2) : p.n64;
  };
  auto stage_addr = [&](int gg) -> uint32_t { return ring_s + (gg % C::NS) * 2 * C::STILE; };

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::QB_QFULL), 1);
    mbar_init(BAR(C::QB_IDONE), 1);
    mbar_init(BAR(C::QB_RFULL), 64);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(BAR(C::QB_FULL + i), 1);
      mbar_init(BAR(C::QB_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(C::QB_SFULL + i), 1);
      mbar_init(BAR(C::QB_DPFULL + i), 1);
      mbar_init(BAR(C::QB_DSFULL + i), 256);
    }
    mbar_init(BAR(C::QB_QFREE), C::QFREE_COUNT);
    mbar_init(BAR(C::QB_DRAIN), 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_o);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_launch_dependents();
  grid_wait_prior();
  // Tensor memory: step buffer b holds S at [128 b, 128 b + 64) and dP at [128 b + 64,
  // 128 b + 128) (dS packed over the first 16 columns of each 32-column half); dQ [256, 256+D).
  constexpr uint32_t C_DQ = 256;
  auto c_s = [](int gg) -> uint32_t { return static_cast<uint32_t>(gg & 1) * 128u; };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int g = 0, issued = 0, q_loads = 0;
      for (int r = 0; ok && r * G < p.items; ++r) {
        const int idx = bwd_item(r, cta, G);
        if (idx >= p.items) continue;
        int bh, qt, nsteps;
        decode(idx, bh, qt, nsteps);
        for (int s = 0; s < nsteps; ++s, ++g) {
          const int st = g % C::NS;
          if (!(ok = wait_bounded(BAR(C::QB_EMPTY + st), ((g / C::NS) & 1) ^ 1u, abort_flag, p.status, kDevTimeoutLoad,
                                  LIM)))
            break;
          const uint32_t stage = stage_addr(g);
          mbar_arrive_expect_tx(BAR(C::QB_FULL + st), 2 * C::STILE);
          for (int c = 0; c < C::NCH; ++c) {
            tma_load_3d(stage + c * C::SCHUNK, &tm_k, c * 64, s * 64, bh, BAR(C::QB_FULL + st));
            tma_load_3d(stage + C::STILE + c * C::SCHUNK, &tm_v, c * 64, s * 64, bh, BAR(C::QB_FULL + st));
          }
          ++issued;
          if (s == 0) {
            // Q, dO and O of this item, once the previous item's last S and dP products are
            // complete and its statistics are formed and read (up to two steps before it ends).
            if (q_loads > 0 && !(ok = wait_bounded(BAR(C::QB_QFREE), (q_loads - 1) & 1, abort_flag, p.status,
                                                   kDevTimeoutLoad, LIM)))
              break;
            mbar_arrive_expect_tx(BAR(C::QB_QFULL), 3 * C::RTILE);
            for (int c = 0; c < C::NCH; ++c) {
              tma_load_3d(q_s + c * C::RCHUNK, &tm_q, c * 64, qt * 128, bh, BAR(C::QB_QFULL));
              tma_load_3d(do_s + c * C::RCHUNK, &tm_do, c * 64, qt * 128, bh, BAR(C::QB_QFULL));
              tma_load_3d(o_s + c * C::RCHUNK, &tm_o, c * 64, qt * 128, bh, BAR(C::QB_QFULL));
            }
            ++q_loads;
          }
        }
      }
      if (q_loads > 0) wait_drain(BAR(C::QB_QFULL), (q_loads - 1) & 1, LIM);
      for (int s = issued > C::NS ? issued - C::NS : 0; s < issued; ++s)
        wait_drain(BAR(C::QB_FULL + s % C::NS), (s / C::NS) & 1, LIM);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      int g = 0, it = 0;
      auto wait = [&](int b, uint32_t ph) -> bool {
        return wait_bounded(BAR(b), ph, abort_flag, p.status, kDevTimeoutMma, LIM);
      };
      const SDesc qa = sdesc_split(sdesc_sw128(q_s, 16, 1024)), doa = sdesc_split(sdesc_sw128(do_s, 16, 1024));
      // S = Q K^T and dP = dO V^T of global step gg into its buffer.
      auto issue_sdp = [&](int gg) {
        const uint32_t stage = stage_addr(gg);
        const SDesc kb = sdesc_split(sdesc_sw128(stage, 16, 1024));
        const SDesc vb = sdesc_split(sdesc_sw128(stage + C::STILE, 16, 1024));
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + c_s(gg), qa, c * C::RCHUNK + kk * 32, kb, c * C::SCHUNK + kk * 32, C::IDESC_S,
                        (c | kk) != 0 ? 1u : 0u);
        umma_commit(BAR(C::QB_SFULL + (gg & 1)));
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + c_s(gg) + 64, doa, c * C::RCHUNK + kk * 32, vb, c * C::SCHUNK + kk * 32, C::IDESC_S,
                        (c | kk) != 0 ? 1u : 0u);
        umma_commit(BAR(C::QB_DPFULL + (gg & 1)));
      };
      auto stage_ready = [&](int gg) { return wait(C::QB_FULL + gg % C::NS, (gg / C::NS) & 1); };
      for (int r = 0; ok && r * G < p.items; ++r) {
        const int idx = bwd_item(r, cta, G);
        if (idx >= p.items) continue;
        int bh, qt, nsteps;
        decode(idx, bh, qt, nsteps);
        if (!(ok = wait(C::QB_QFULL, it & 1) && stage_ready(g))) break;
        tc_fence_after();
        issue_sdp(g);
        if (nsteps > 1) {
          if (!(ok = stage_ready(g + 1))) break;
          tc_fence_after();
          issue_sdp(g + 1);
        }
        if (nsteps <= 2) umma_commit(BAR(C::QB_QFREE));  // the item's last S, dP are issued
        for (int s = 0; s < nsteps; ++s, ++g) {
          // dQ += dS K
          if (!(ok = wait(C::QB_DSFULL + (g & 1), (static_cast<uint32_t>(g) >> 1) & 1u))) break;
          tc_fence_after();
          const SDesc km = sdesc_split(sdesc_sw128(stage_addr(g), C::SCHUNK, 1024));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ts_off(tmem + C_DQ, tmem + c_s(g) + 64 + bwd_a_col(kk), km, kk * 2048, C::IDESC_ACC,
                        (s > 0 || kk > 0) ? 1u : 0u);
          umma_commit(BAR(C::QB_EMPTY + g % C::NS));
          if (s + 2 < nsteps) {
            if (!(ok = stage_ready(g + 2))) break;
            tc_fence_after();
            issue_sdp(g + 2);  // into this step's buffers, read in order after dQ above
            if (s + 3 == nsteps) umma_commit(BAR(C::QB_QFREE));
          }
        }
        if (!ok) break;
        umma_commit(BAR(C::QB_IDONE));  // Q, dO free; dQ final
        ++it;
      }
      umma_commit(BAR(C::QB_DRAIN));
      wait_drain(BAR(C::QB_DRAIN), 0, LIM);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------------ row statistics
    const int w = warp - 2;  // rows [64 w, 64 w + 64) of the item's query tile
    int it = 0;
    float lse_next[2];
    bool have_next = false;
    for (int r = 0; r * G < p.items; ++r) {
      const int idx = bwd_item(r, cta, G);
      if (idx >= p.items) continue;
      int bh, qt, nsteps;
      decode(idx, bh, qt, nsteps);
      float lse_cur[2];
      if (have_next) {
        lse_cur[0] = lse_next[0];
        lse_cur[1] = lse_next[1];
      } else {
        bwd_row_lse(p, bh, qt * 128, 64 * w, lane, lse_cur);
      }
      // The next item's LSE is loaded while this item runs.
      const int nidx = bwd_item(r + 1, cta, G);
      have_next = nidx < p.items;
      if (have_next) {
        int nbh, nqt, nn;
        decode(nidx, nbh, nqt, nn);
        bwd_row_lse(p, nbh, nqt * 128, 64 * w, lane, lse_next);
      }
      const bool ok = __all_sync(0xffffffffu, wait_bounded(BAR(C::QB_QFULL), it & 1, abort_flag, p.status,
                                                           kDevTimeoutSoftmax, LIM));
      if (!ok) break;
      bwd_row_stats<D>(p, bh, qt * 128, do_s, o_s, stat_s, 64 * w, lane, lse_cur);
      fence_proxy_async_smem();  // dO and O are refilled by TMA for the next item
      mbar_arrive(BAR(C::QB_RFULL));
      mbar_arrive(BAR(C::QB_QFREE));
      ++it;
    }
  } else {
    // ------------------------------------------------------------------ elementwise warpgroups
    const int h = (warp - 4) >> 2;        // key columns [32 h, 32 h + 32) of every tile
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // query row of the tile == tensor-memory lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.c2;
    auto wait_warp = [&](int b, uint32_t ph) -> bool {
      return __all_sync(0xffffffffu, wait_bounded(BAR(b), ph, abort_flag, p.status, kDevTimeoutSoftmax, LIM));
    };
    bool ok = true;
    int g = 0, it = 0;
    for (int r = 0; ok && r * G < p.items; ++r) {
      const int idx = bwd_item(r, cta, G);
      if (idx >= p.items) continue;
      int bh, qt, nsteps;
      decode(idx, bh, qt, nsteps);
      if (!(ok = wait_warp(C::QB_RFULL, it & 1))) break;
      const float lrow = stat_s[row], drow = stat_s[128 + row];
      mbar_arrive(BAR(C::QB_QFREE));  // the statistics buffer may take the next item's
      const int qrow = qt * 128 + row;
      for (int s = 0; s < nsteps; ++s, ++g) {
        const uint32_t pb = (static_cast<uint32_t>(g) >> 1) & 1u;
        const uint32_t s_col = tmem + lane_base + c_s(g) + 32 * h, dp_col = s_col + 64;
        // P (registers only): P = exp2(S c2 - LSE log2 e), masked where the key comes after
        // the query or lies past L.
        if (!(ok = wait_warp(C::QB_SFULL + (g & 1), pb))) break;
        tc_fence_after();
        const int key0 = s * 64 + 32 * h;
        const bool edge = (CAUSAL && key0 + 31 > qt * 128) || key0 + 32 > p.L;
        float pv[32];
        {
          uint32_t sr[32];
          tmem_ld32x32(s_col, sr);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            float pp = ex2_approx(fmaf(__uint_as_float(sr[c]), c2, -lrow));
            if (edge && ((CAUSAL && key0 + c > qrow) || key0 + c >= p.L)) pp = 0.f;
            pv[c] = pp;
          }
        }
        // dS = P (dP - D), packed to fp16 into the first 16 of its 32 columns.
        if (!(ok = wait_warp(C::QB_DPFULL + (g & 1), pb))) break;
        tc_fence_after();
        {
          uint32_t dr[32];
          tmem_ld32x32(dp_col, dr);
          uint32_t dk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            dk[i] = pack_f16x2(pv[2 * i] * (__uint_as_float(dr[2 * i]) - drow),
                               pv[2 * i + 1] * (__uint_as_float(dr[2 * i + 1]) - drow));
          tmem_st32x16(dp_col, dk);
        }
        tc_fence_before();
        mbar_arrive(BAR(C::QB_DSFULL + (g & 1)));
      }
      if (!ok) break;
      // ---------------------------------------------------------------- epilogue
      // scale * dQ: warpgroup h writes columns [h D/2, (h+1) D/2) of its query row.
      if (!(ok = wait_warp(C::QB_IDONE, it & 1))) break;
      tc_fence_after();
      __half *const dst = p.dq + (static_cast<long long>(bh) * p.L + qrow) * D + h * (D / 2);
      bwd_store_row<D / 2>(tmem + lane_base + C_DQ + h * (D / 2), dst, p.scale, qrow < p.L && *abort_flag == 0u);
      tc_fence_before();
      ++it;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

cudaError_t launch_bwd_64(const BwdLaunch &a);
cudaError_t launch_bwd_128(const BwdLaunch &a);

}  // namespace gbattn
