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
// save; here no atomics are used at all: two kernels, one per output side.
//
//   attn_bwd_dkdv_kernel: one CTA per (head, 128-key tile j), K_j and V_j resident, the
//     query tiles i streamed:  S^T = K_j Q_i^T and dP^T = V_j dO_i^T on the tensor core;
//     a warpgroup (one key row per thread) forms P^T and dS^T in fp16 over the same
//     tensor-memory columns; then dV_j += P^T dO_i and dK_j += dS^T Q_i.
//   attn_bwd_dq_kernel: one CTA per (head, 128-query tile i), Q_i, dO_i, O_i resident, the
//     key tiles j streamed:  S = Q_i K_j^T and dP = dO_i V_j^T; the warpgroup (one query
//     row per thread) forms dS; then dQ_i += dS K_j.
// Both recompute P from the forward LSE (no L x L matrix is stored) and form D_i from the
// O and dO tiles they load (no separate pass or scratch buffer).  The tensor-core operand
// forms are the forward kernels': K-major A and B from shared memory for the logit-like
// products, A from tensor memory with an MN-major B for the accumulations.  Items run
// longest first (a grid of one CTA per item; the hardware hands the next item to the
// first free SM).
//
// Warp roles (256 threads): warp 0 TMA producer; warp 1 tensor-memory owner and MMA
// issuer; warps 4-7 the elementwise warpgroup and the epilogue; warps 2, 3 idle.
// Every wait is bounded (about two seconds of SM clock), as in the forward kernels.
#pragma once

#include <cuda_fp16.h>

#include "attn_fwd_kernel.cuh"

namespace gbattn {

struct BwdParams {
  const float *lse;        // [BH, L] forward LSE (natural log)
  unsigned *status;
  long long wait_limit;
  int BH, L, nQ;
  float c2;                // scale * log2(e)
  float scale;
};

struct BwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_o, tm_do, tm_dq, tm_dk, tm_dv;
  BwdParams p;
  bool causal;
  cudaStream_t stream;
};

template <int D>
struct BwdCfg {
  static constexpr int NCH = D / 64;                  // 64-column chunks of a tile
  static constexpr int CHUNK = 128 * 128;             // a 128-row x 64-column fp16 box
  static constexpr int TILE = NCH * CHUNK;            // one 128 x D tile
  static constexpr int NS = 2;                        // ring stages (pairs of tiles)
  static constexpr uint32_t IDESC_SS = idesc_f16_f32(128, 128, 0, 0);  // 128 x 128 logit-like
  static constexpr uint32_t IDESC_ACC = idesc_f16_f32(128, D, 0, 1);   // B MN-major, N = D
  static constexpr int TMEM_COLS = 512;
  // dK/dV kernel: [K][V][ring: NS x (Q, dO)][O][lse, D: 2 x 128 fp32][barriers]
  static constexpr int KV_OFF_RING = 2 * TILE;
  static constexpr int KV_OFF_O = KV_OFF_RING + NS * 2 * TILE;
  static constexpr int KV_OFF_LD = KV_OFF_O + TILE;
  static constexpr int KV_OFF_BAR = KV_OFF_LD + 2 * 128 * 4;
  // barriers: KVFULL, FULL[NS], EMPTY[NS], OFULL, OEMPTY, SFULL, PFULL, DONE, DRAIN
  static constexpr int KB_KVFULL = 0, KB_FULL = 1, KB_EMPTY = 1 + NS, KB_OFULL = 1 + 2 * NS,
                       KB_OEMPTY = KB_OFULL + 1, KB_SFULL = KB_OEMPTY + 1, KB_PFULL = KB_SFULL + 1,
                       KB_DONE = KB_PFULL + 1, KB_DRAIN = KB_DONE + 1, KB_N = KB_DRAIN + 1;
  static constexpr int KV_SMEM = 1024 + KV_OFF_BAR + 8 * KB_N + 16;
  // dQ kernel: [Q][dO][O][ring: NS x (K, V)][barriers]
  static constexpr int Q_OFF_RING = 3 * TILE;
  static constexpr int Q_OFF_BAR = Q_OFF_RING + NS * 2 * TILE;
  // barriers: QFULL, FULL[NS], EMPTY[NS], SFULL, PFULL, DONE, DRAIN
  static constexpr int QB_QFULL = 0, QB_FULL = 1, QB_EMPTY = 1 + NS, QB_SFULL = 1 + 2 * NS,
                       QB_PFULL = QB_SFULL + 1, QB_DONE = QB_PFULL + 1, QB_DRAIN = QB_DONE + 1, QB_N = QB_DRAIN + 1;
  static constexpr int Q_SMEM = 1024 + Q_OFF_BAR + 8 * QB_N + 16;
  static_assert(KV_SMEM <= 232448 && Q_SMEM <= 232448, "shared memory budget");
  static_assert(256 + 2 * D <= TMEM_COLS, "tensor memory budget");
};

// Shared-memory address of 16-byte chunk c (8 fp16 values) of row r of a 128-row tile
// loaded by TMA with the 128-byte swizzle in 64-column boxes.
template <int D>
__device__ __forceinline__ uint32_t bwd_chunk_addr(uint32_t tile, int r, int c) {
  return tile + (c >> 3) * BwdCfg<D>::CHUNK + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// dO_r . O_r for row r of two swizzled tiles (fp32 products and sum).
template <int D>
__device__ __forceinline__ float bwd_row_dot(uint32_t a_tile, uint32_t b_tile, int r) {
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const uint4 x = ld_shared_v4(bwd_chunk_addr<D>(a_tile, r, c));
    const uint4 y = ld_shared_v4(bwd_chunk_addr<D>(b_tile, r, c));
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&xs[h]));
      const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&ys[h]));
      acc0 = fmaf(a.x, b.x, acc0);
      acc1 = fmaf(a.y, b.y, acc1);
    }
  }
  return acc0 + acc1;
}

// 32 fp16 pairs from 64 fp32 values.
__device__ __forceinline__ void bwd_pack64(const float (&x)[64], uint32_t (&out)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) out[i] = pack_f16x2(x[2 * i], x[2 * i + 1]);
}

// Epilogue helper: tensor-memory accumulator row (D fp32 columns) * mult -> fp16 into a
// swizzled staging tile (the layout a TMA store reads), 32 columns at a time.
template <int D>
__device__ __forceinline__ void bwd_stage_row(uint32_t acc_tmem, uint32_t stage, int row, float mult) {
#pragma unroll 1
  for (int c32 = 0; c32 < D / 32; ++c32) {
    uint32_t r[32];
    tmem_ld32x32(acc_tmem + c32 * 32, r);
    uint32_t h[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) h[i] = pack_f16x2(__uint_as_float(r[2 * i]) * mult, __uint_as_float(r[2 * i + 1]) * mult);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4)
      st_shared_v4(bwd_chunk_addr<D>(stage, row, c32 * 4 + q4), h[4 * q4], h[4 * q4 + 1], h[4 * q4 + 2], h[4 * q4 + 3]);
  }
}

// ======================================================================== dK / dV
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(256, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                         const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dk,
                         const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t k_s = base, v_s = base + C::TILE, ring_s = base + C::KV_OFF_RING, o_s = base + C::KV_OFF_O;
  float *const lse_s = reinterpret_cast<float *>(base_ptr + C::KV_OFF_LD);  // per query column, x log2(e)
  float *const dd_s = lse_s + 128;                                           // D per query column
  const uint32_t bar_s = base + C::KV_OFF_BAR;
  uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + C::KV_OFF_BAR + 8 * C::KB_N);
  volatile uint32_t *const abort_flag = tmem_slot + 1;
  auto BAR = [&](int i) -> uint32_t { return bar_s + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long LIM = p.wait_limit;

  // Item: key tile kt of head bh, longest first (causal: the first key tiles see the most
  // query tiles).
  const int grp = static_cast<int>(blockIdx.x) / p.BH;
  const int bh = static_cast<int>(blockIdx.x) - grp * p.BH;
  const int kt = grp;
  const int q_first = CAUSAL ? kt : 0;
  const int nsteps = p.nQ - q_first;

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::KB_KVFULL), 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(BAR(C::KB_FULL + i), 1);
      mbar_init(BAR(C::KB_EMPTY + i), 1);
    }
    mbar_init(BAR(C::KB_OFULL), 1);
    mbar_init(BAR(C::KB_OEMPTY), 128);
    mbar_init(BAR(C::KB_SFULL), 1);
    mbar_init(BAR(C::KB_PFULL), 128);
    mbar_init(BAR(C::KB_DONE), 1);
    mbar_init(BAR(C::KB_DRAIN), 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
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
  // Tensor memory: S^T [0,128) (P^T over its first 64 columns), dP^T [128,256) (dS^T over
  // its first 64 columns), dV [256, 256+D), dK [256+D, 256+2D).
  constexpr uint32_t C_S = 0, C_DP = 128, C_DV = 256, C_DK = 256 + D;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(BAR(C::KB_KVFULL), 2 * C::TILE);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_3d(k_s + c * C::CHUNK, &tm_k, c * 64, kt * 128, bh, BAR(C::KB_KVFULL));
        tma_load_3d(v_s + c * C::CHUNK, &tm_v, c * 64, kt * 128, bh, BAR(C::KB_KVFULL));
      }
      for (int s = 0; s < nsteps && ok; ++s) {
        const int qi = q_first + s;
        const int st = s % C::NS;
        if (!(ok = wait_bounded(BAR(C::KB_EMPTY + st), ((s / C::NS) & 1) ^ 1u, abort_flag, p.status, kDevTimeoutLoad,
                                LIM)))
          break;
        const uint32_t stage = ring_s + st * 2 * C::TILE;
        mbar_arrive_expect_tx(BAR(C::KB_FULL + st), 2 * C::TILE);
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(stage + c * C::CHUNK, &tm_q, c * 64, qi * 128, bh, BAR(C::KB_FULL + st));
          tma_load_3d(stage + C::TILE + c * C::CHUNK, &tm_do, c * 64, qi * 128, bh, BAR(C::KB_FULL + st));
        }
        if (!(ok = wait_bounded(BAR(C::KB_OEMPTY), (s & 1) ^ 1u, abort_flag, p.status, kDevTimeoutLoad, LIM))) break;
        mbar_arrive_expect_tx(BAR(C::KB_OFULL), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(o_s + c * C::CHUNK, &tm_o, c * 64, qi * 128, bh, BAR(C::KB_OFULL));
      }
      // Drain: loads in flight land before the CTA may exit.
      wait_drain(BAR(C::KB_KVFULL), 0, LIM);
      for (int s = nsteps > C::NS ? nsteps - C::NS : 0; s < nsteps; ++s)
        wait_drain(BAR(C::KB_FULL + s % C::NS), (s / C::NS) & 1, LIM);
      if (nsteps > 0) wait_drain(BAR(C::KB_OFULL), (nsteps - 1) & 1, LIM);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = wait_bounded(BAR(C::KB_KVFULL), 0, abort_flag, p.status, kDevTimeoutMma, LIM);
      const SDesc ka = sdesc_split(sdesc_sw128(k_s, 16, 1024)), va = sdesc_split(sdesc_sw128(v_s, 16, 1024));
      for (int s = 0; s < nsteps && ok; ++s) {
        const int st = s % C::NS;
        if (!(ok = wait_bounded(BAR(C::KB_FULL + st), (s / C::NS) & 1, abort_flag, p.status, kDevTimeoutMma, LIM)))
          break;
        tc_fence_after();
        const uint32_t stage = ring_s + st * 2 * C::TILE;
        const SDesc qb = sdesc_split(sdesc_sw128(stage, 16, 1024));
        const SDesc dob = sdesc_split(sdesc_sw128(stage + C::TILE, 16, 1024));
        // S^T = K Q^T, dP^T = V dO^T (head_dim summed over every 64-wide chunk).
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + C_S, ka, c * C::CHUNK + kk * 32, qb, c * C::CHUNK + kk * 32, C::IDESC_SS,
                        (c | kk) != 0 ? 1u : 0u);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + C_DP, va, c * C::CHUNK + kk * 32, dob, c * C::CHUNK + kk * 32, C::IDESC_SS,
                        (c | kk) != 0 ? 1u : 0u);
        umma_commit(BAR(C::KB_SFULL));
        // P^T and dS^T (fp16) in tensor memory, then dV += P^T dO, dK += dS^T Q.
        if (!(ok = wait_bounded(BAR(C::KB_PFULL), s & 1, abort_flag, p.status, kDevTimeoutMma, LIM))) break;
        tc_fence_after();
        const SDesc dom = sdesc_split(sdesc_sw128(stage + C::TILE, C::CHUNK, 1024));
        const SDesc qm = sdesc_split(sdesc_sw128(stage, C::CHUNK, 1024));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_off(tmem + C_DV, tmem + C_S + kk * 8u, dom, kk * 2048, C::IDESC_ACC, (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_off(tmem + C_DK, tmem + C_DP + kk * 8u, qm, kk * 2048, C::IDESC_ACC, (s > 0 || kk > 0) ? 1u : 0u);
        umma_commit(BAR(C::KB_EMPTY + st));
      }
      umma_commit(BAR(C::KB_DONE));  // every MMA issued so far is complete
      wait_drain(BAR(C::KB_DONE), 0, LIM);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ elementwise warpgroup
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row of the tile == tensor-memory lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.c2;
    constexpr float kLog2e = 1.4426950408889634f;
    bool ok = true;
    auto wait_warp = [&](uint32_t b, uint32_t ph) -> bool {
      const bool r = wait_bounded(b, ph, abort_flag, p.status, kDevTimeoutSoftmax, LIM);
      return __all_sync(0xffffffffu, r);
    };
    auto wg_sync = [] { asm volatile("bar.sync 1, 128;" ::: "memory"); };
    // Every warp of the group runs every step and reaches every named barrier, also after
    // a wait of its own timed out (`ok` false: the work is skipped, the barriers are not),
    // so that a timeout can never leave the other warps stuck at a barrier.
    for (int s = 0; s < nsteps; ++s) {
      const int qi = q_first + s;
      const int st = s % C::NS;
      const uint32_t stage = ring_s + st * 2 * C::TILE;
      // D and LSE of this query tile: thread `row` does query `row`.
      if (ok) ok = wait_warp(BAR(C::KB_FULL + st), (s / C::NS) & 1);
      if (ok) ok = wait_warp(BAR(C::KB_OFULL), s & 1);
      const int qrow = qi * 128 + row;
      float dval = 0.f, lval = INFINITY;  // query rows past L: P = 0
      if (ok) {
        dval = bwd_row_dot<D>(stage + C::TILE, o_s, row);
        // The O buffer (and this dO tile) is refilled by TMA, in the async proxy: order these
        // generic-proxy reads before the release that lets the producer overwrite it.
        fence_proxy_async_smem();
        mbar_arrive(BAR(C::KB_OEMPTY));
        if (qrow < p.L) lval = p.lse[static_cast<long long>(bh) * p.L + qrow] * kLog2e;
      }
      wg_sync();  // every thread is done reading the previous step's values
      lse_s[row] = lval;
      dd_s[row] = dval;
      wg_sync();
      if (ok) ok = wait_warp(BAR(C::KB_SFULL), s & 1);
      if (!ok) continue;
      tc_fence_after();
      // Row `row` of S^T and dP^T: columns = the tile's 128 queries, in two halves.
      const bool diag = CAUSAL && qi == kt;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t sr[64], dr[64];
        tmem_ld32x64(tmem + lane_base + C_S + h * 64, sr);
        tmem_ld32x64(tmem + lane_base + C_DP + h * 64, dr);
        float pv[64], dsv[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int col = h * 64 + c;
          float pp = ex2_approx(__uint_as_float(sr[c]) * c2 - lse_s[col]);
          if (diag && col < row) pp = 0.f;  // query before key: masked
          pv[c] = pp;
          dsv[c] = pp * (__uint_as_float(dr[c]) - dd_s[col]);
        }
        uint32_t pk[32], dk[32];
        bwd_pack64(pv, pk);
        bwd_pack64(dsv, dk);
        tmem_st32x32(tmem + lane_base + C_S + h * 32, pk);
        tmem_st32x32(tmem + lane_base + C_DP + h * 32, dk);
      }
      tc_fence_before();
      mbar_arrive(BAR(C::KB_PFULL));
    }
    // ---------------------------------------------------------------- epilogue
    // dV and scale * dK into the (no longer read) K and V tiles, then TMA stores.
    if (ok) ok = wait_warp(BAR(C::KB_DONE), 0);
    if (ok) {
      tc_fence_after();
      bwd_stage_row<D>(tmem + lane_base + C_DV, v_s, row, 1.0f);
      bwd_stage_row<D>(tmem + lane_base + C_DK, k_s, row, p.scale);
      fence_proxy_async_smem();
    }
    wg_sync();
    if (warp == 4 && lane == 0 && ok && *abort_flag == 0u) {
      for (int c = 0; c < C::NCH; ++c) {
        tma_store_3d(&tm_dv, v_s + c * C::CHUNK, c * 64, kt * 128, bh);
        tma_store_3d(&tm_dk, k_s + c * C::CHUNK, c * 64, kt * 128, bh);
      }
      bulk_commit();
      bulk_wait0();
    }
    __syncwarp();
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
__global__ void __launch_bounds__(256, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dq,
                       const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t q_s = base, do_s = base + C::TILE, o_s = base + 2 * C::TILE, ring_s = base + C::Q_OFF_RING;
  const uint32_t bar_s = base + C::Q_OFF_BAR;
  uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + C::Q_OFF_BAR + 8 * C::QB_N);
  volatile uint32_t *const abort_flag = tmem_slot + 1;
  auto BAR = [&](int i) -> uint32_t { return bar_s + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long LIM = p.wait_limit;

  // Item: query tile qt of head bh, longest first (causal: the last query tiles see the
  // most key tiles).
  const int grp = static_cast<int>(blockIdx.x) / p.BH;
  const int bh = static_cast<int>(blockIdx.x) - grp * p.BH;
  const int qt = CAUSAL ? p.nQ - 1 - grp : grp;
  const int nsteps = CAUSAL ? qt + 1 : p.nQ;

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::QB_QFULL), 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(BAR(C::QB_FULL + i), 1);
      mbar_init(BAR(C::QB_EMPTY + i), 1);
    }
    mbar_init(BAR(C::QB_SFULL), 1);
    mbar_init(BAR(C::QB_PFULL), 128);
    mbar_init(BAR(C::QB_DONE), 1);
    mbar_init(BAR(C::QB_DRAIN), 1);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
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
  // Tensor memory: S [0,128), dP [128,256) (dS over its first 64 columns), dQ [256, 256+D).
  constexpr uint32_t C_S = 0, C_DP = 128, C_DQ = 256;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(BAR(C::QB_QFULL), 3 * C::TILE);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_3d(q_s + c * C::CHUNK, &tm_q, c * 64, qt * 128, bh, BAR(C::QB_QFULL));
        tma_load_3d(do_s + c * C::CHUNK, &tm_do, c * 64, qt * 128, bh, BAR(C::QB_QFULL));
        tma_load_3d(o_s + c * C::CHUNK, &tm_o, c * 64, qt * 128, bh, BAR(C::QB_QFULL));
      }
      for (int s = 0; s < nsteps && ok; ++s) {
        const int st = s % C::NS;
        if (!(ok = wait_bounded(BAR(C::QB_EMPTY + st), ((s / C::NS) & 1) ^ 1u, abort_flag, p.status, kDevTimeoutLoad,
                                LIM)))
          break;
        const uint32_t stage = ring_s + st * 2 * C::TILE;
        mbar_arrive_expect_tx(BAR(C::QB_FULL + st), 2 * C::TILE);
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(stage + c * C::CHUNK, &tm_k, c * 64, s * 128, bh, BAR(C::QB_FULL + st));
          tma_load_3d(stage + C::TILE + c * C::CHUNK, &tm_v, c * 64, s * 128, bh, BAR(C::QB_FULL + st));
        }
      }
      wait_drain(BAR(C::QB_QFULL), 0, LIM);
      for (int s = nsteps > C::NS ? nsteps - C::NS : 0; s < nsteps; ++s)
        wait_drain(BAR(C::QB_FULL + s % C::NS), (s / C::NS) & 1, LIM);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = wait_bounded(BAR(C::QB_QFULL), 0, abort_flag, p.status, kDevTimeoutMma, LIM);
      const SDesc qa = sdesc_split(sdesc_sw128(q_s, 16, 1024)), doa = sdesc_split(sdesc_sw128(do_s, 16, 1024));
      for (int s = 0; s < nsteps && ok; ++s) {
        const int st = s % C::NS;
        if (!(ok = wait_bounded(BAR(C::QB_FULL + st), (s / C::NS) & 1, abort_flag, p.status, kDevTimeoutMma, LIM)))
          break;
        tc_fence_after();
        const uint32_t stage = ring_s + st * 2 * C::TILE;
        const SDesc kb = sdesc_split(sdesc_sw128(stage, 16, 1024));
        const SDesc vb = sdesc_split(sdesc_sw128(stage + C::TILE, 16, 1024));
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + C_S, qa, c * C::CHUNK + kk * 32, kb, c * C::CHUNK + kk * 32, C::IDESC_SS,
                        (c | kk) != 0 ? 1u : 0u);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + C_DP, doa, c * C::CHUNK + kk * 32, vb, c * C::CHUNK + kk * 32, C::IDESC_SS,
                        (c | kk) != 0 ? 1u : 0u);
        umma_commit(BAR(C::QB_SFULL));
        if (!(ok = wait_bounded(BAR(C::QB_PFULL), s & 1, abort_flag, p.status, kDevTimeoutMma, LIM))) break;
        tc_fence_after();
        const SDesc km = sdesc_split(sdesc_sw128(stage, C::CHUNK, 1024));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_off(tmem + C_DQ, tmem + C_DP + kk * 8u, km, kk * 2048, C::IDESC_ACC, (s > 0 || kk > 0) ? 1u : 0u);
        umma_commit(BAR(C::QB_EMPTY + st));
      }
      umma_commit(BAR(C::QB_DONE));
      wait_drain(BAR(C::QB_DONE), 0, LIM);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // query row of the tile == tensor-memory lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int qrow = qt * 128 + row;
    const float c2 = p.c2;
    constexpr float kLog2e = 1.4426950408889634f;
    bool ok = true;
    auto wait_warp = [&](uint32_t b, uint32_t ph) -> bool {
      const bool r = wait_bounded(b, ph, abort_flag, p.status, kDevTimeoutSoftmax, LIM);
      return __all_sync(0xffffffffu, r);
    };
    float lval = INFINITY, dval = 0.f;
    if ((ok = wait_warp(BAR(C::QB_QFULL), 0))) {
      dval = bwd_row_dot<D>(do_s, o_s, row);
      if (qrow < p.L) lval = p.lse[static_cast<long long>(bh) * p.L + qrow] * kLog2e;
    }
    for (int s = 0; s < nsteps && ok; ++s) {
      if (!(ok = wait_warp(BAR(C::QB_SFULL), s & 1))) break;
      tc_fence_after();
      const bool diag = CAUSAL && s == qt;
      const int kbase = s * 128;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t sr[64], dr[64];
        tmem_ld32x64(tmem + lane_base + C_S + h * 64, sr);
        tmem_ld32x64(tmem + lane_base + C_DP + h * 64, dr);
        float dsv[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int col = h * 64 + c;
          float pp = ex2_approx(__uint_as_float(sr[c]) * c2 - lval);
          if ((diag && col > row) || kbase + col >= p.L) pp = 0.f;  // key after query, or past L
          dsv[c] = pp * (__uint_as_float(dr[c]) - dval);
        }
        uint32_t dk[32];
        bwd_pack64(dsv, dk);
        tmem_st32x32(tmem + lane_base + C_DP + h * 32, dk);
      }
      tc_fence_before();
      mbar_arrive(BAR(C::QB_PFULL));
    }
    // ---------------------------------------------------------------- epilogue
    // The named barrier is reached by every warp of the group, whatever its `ok`.
    if (ok) ok = wait_warp(BAR(C::QB_DONE), 0);
    if (ok) {
      tc_fence_after();
      bwd_stage_row<D>(tmem + lane_base + C_DQ, o_s, row, p.scale);  // O no longer read
      fence_proxy_async_smem();
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (warp == 4 && lane == 0 && ok && *abort_flag == 0u) {
      for (int c = 0; c < C::NCH; ++c) tma_store_3d(&tm_dq, o_s + c * C::CHUNK, c * 64, qt * 128, bh);
      bulk_commit();
      bulk_wait0();
    }
    __syncwarp();
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
