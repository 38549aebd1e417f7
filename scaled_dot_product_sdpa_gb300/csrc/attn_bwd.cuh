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
//   attn_bwd_dq_kernel: work item = (head, 128-query tile i), Q_i and dO_i resident, the
//     key rows streamed in 128-row tiles j (K and V in rings of their own):  S = Q_i K_j^T
//     and dP = dO_i V_j^T on the tensor core; dS is formed; then dQ_i += dS K_j.  Its
//     elementwise warps also form the row statistics LSE_i log2(e) and D_i = dO_i . O_i
//     (O and LSE read from global memory one item ahead) and write them to a workspace
//     of 8 bytes per query row (the only memory beyond the inputs and outputs).
//   attn_bwd_dkdv_kernel: work item = (head, 128-key tile j), K_j and V_j resident, the
//     query rows streamed in 128-row tiles i (Q, dO and the row statistics in rings of
//     their own):  S^T = K_j Q_i^T and dP^T = V_j dO_i^T; P^T and dS^T are formed in fp16
//     over the same tensor-memory columns; then dV_j += P^T dO_i and dK_j += dS^T Q_i.
// Both recompute P from the forward LSE (no L x L matrix is stored).  The tensor-core
// operand forms are the forward kernels': K-major A and B from shared memory for the
// logit-like products (N = 128), A from tensor memory with an MN-major B for the
// accumulations (N = head_dim).
//
// Pipelining: every step is 128 streamed rows.  In the dQ kernel S is double-buffered in
// tensor memory, so step s+1's S runs while the elementwise warps work on step s; in the
// dK/dV kernel (whose tensor memory holds S^T, dP^T, dV and dK) the products are ordered
// dV(s), S^T(s+1), dK(s), dP^T(s+1), so that each runs while the warps form the next
// P or dS.  The streamed operands sit in rings deep enough for their loads to run about
// two steps ahead.  Both kernels are persistent: one CTA per SM walks the items longest
// first, in "snake" order (CTA b takes items b, 2G-1-b, 2G+b, ... of the sorted list,
// G = grid size), so that the per-CTA totals even out.  The epilogue stages the
// accumulators (fp16) in the ring slots of the item's last step, which its last products
// have just released, and writes them out by TMA store; the producer refills such a slot
// once the store has read it.  (Each thread storing its own row to global memory made 32
// partial-line writes per instruction and cost 1.5 to 3 us per item.)
//
// Warp roles (384 threads): warp 0 TMA producer; warp 1 tensor-memory owner and MMA
// issuer; warps 2-3 idle; warps 4-7 and 8-11 two elementwise warpgroups, each taking one
// half of the 128 columns of every S / dP tile (and, in the dQ kernel, one half of every
// row of the row statistics), and the epilogue.
// Every wait is bounded (about two seconds of SM clock), as in the forward kernels.
#pragma once

#include <cuda_fp16.h>

#include "attn_fwd_kernel.cuh"

namespace gbattn {

constexpr unsigned kDevSmemAlign = 7;  // dynamic shared memory not 1 KB aligned

struct BwdParams {
  const float *lse;        // [BH, L] forward LSE (natural log)
  const __half *o;         // [BH, L, D] forward output
  float *ws_lse2, *ws_d;   // workspace [BH, Lp] each: LSE log2(e) (+inf past L) and D
  unsigned *status;
  long long wait_limit;
  int BH, L;
  int Lp;                  // L rounded up to a multiple of 128 (workspace row stride)
  int n128;               // ceil(L / 128)
  int items;               // BH * n128 work items per kernel
  float c2;                // scale * log2(e)
  float scale;
};

struct BwdLaunch {
  CUtensorMap tm_q128, tm_do128, tm_k128, tm_v128;  // 128-row x 64-column boxes
  CUtensorMap tm_dq128, tm_dk128, tm_dv128;         // the outputs, same boxes (TMA stores)
  BwdParams p;
  int grid;  // persistent CTAs (<= items)
  bool causal;
  cudaStream_t stream;
};

template <int D>
struct BwdCfg {
  static constexpr int THREADS = 384;
  static constexpr int NCH = D / 64;                  // 64-column chunks of a tile
  static constexpr int RCHUNK = 128 * 128;            // a tile: 128 rows x 64 fp16 columns per box
  static constexpr int RTILE = NCH * RCHUNK;
  static constexpr uint32_t IDESC_S128 = idesc_f16_f32(128, 128, 0, 0);  // 128 x 128 logit-like
  static constexpr uint32_t IDESC_ACC = idesc_f16_f32(128, D, 0, 1);   // B MN-major, N = D
  static constexpr int TMEM_COLS = 512;
  // dK/dV kernel (128-query steps): [K][V][Q ring: NQS tiles][dO ring: NDS tiles][row
  // statistics: 2 x (LSE log2 e: 128 fp32, D: 128 fp32)][barriers].  No alignment slack:
  // the dynamic shared memory starts 1 KB aligned (checked in the kernel).
  static constexpr int NQS = D == 64 ? 6 : 3, NDS = D == 64 ? 4 : 2;
  static constexpr int KV_OFF_Q = 2 * RTILE;
  static constexpr int KV_OFF_DO = KV_OFF_Q + NQS * RTILE;
  static constexpr int KV_OFF_ST = KV_OFF_DO + NDS * RTILE;
  static constexpr int KV_OFF_BAR = KV_OFF_ST + 2 * 1024;
  static constexpr int KB_KVFULL = 0, KB_KVFREE = 1, KB_IDONE = 2, KB_QFULL = 3, KB_QEMPTY = 3 + NQS,
                       KB_DOFULL = 3 + 2 * NQS, KB_DOEMPTY = KB_DOFULL + NDS, KB_STFULL = KB_DOEMPTY + NDS,
                       KB_STEMPTY = KB_STFULL + 2, KB_SFULL = KB_STEMPTY + 2, KB_DPFULL = KB_SFULL + 1,
                       KB_PFULL = KB_DPFULL + 1, KB_DSFULL = KB_PFULL + 1, KB_DRAIN = KB_DSFULL + 1,
                       KB_STGQ = KB_DRAIN + 1, KB_STGDO = KB_STGQ + NQS, KB_STAGED = KB_STGDO + NDS,
                       KB_N = KB_STAGED + 1;
  // STGQ / STGDO: the epilogue's TMA stores have read the Q / dO slot it staged dK / dV in
  // (one per slot); STAGED: every elementwise thread has written its row of the staged tiles.
  static constexpr int KV_SMEM = KV_OFF_BAR + 8 * KB_N + 16;
  // dQ kernel (128-key steps): [Q][dO][K ring: NKS x 128-row tiles][V ring: NVS x 128-row
  // tiles][D halves: 2 x 128 fp32][barriers]
  static constexpr int NKS = D == 64 ? 6 : 3, NVS = D == 64 ? 4 : 2;
  static constexpr int Q_OFF_K = 2 * RTILE;
  static constexpr int Q_OFF_V = Q_OFF_K + NKS * RTILE;
  static constexpr int Q_OFF_ST = Q_OFF_V + NVS * RTILE;
  static constexpr int Q_OFF_BAR = Q_OFF_ST + 256 * 4;
  static constexpr int QB_QFULL = 0, QB_QFREE = 1, QB_DOFULL = 2, QB_DOFREE = 3, QB_DPART = 4, QB_IDONE = 5,
                       QB_KFULL = 6, QB_KEMPTY = 6 + NKS, QB_VFULL = 6 + 2 * NKS, QB_VEMPTY = QB_VFULL + NVS,
                       QB_SFULL = QB_VEMPTY + NVS, QB_DPFULL = QB_SFULL + 2, QB_DSFULL = QB_DPFULL + 1,
                       QB_DRAIN = QB_DSFULL + 1, QB_STGK = QB_DRAIN + 1, QB_STAGED = QB_STGK + NKS,
                       QB_N = QB_STAGED + 1;
  // STGK: the epilogue's TMA store has read the K slot it staged dQ in (one per slot);
  // STAGED: every elementwise thread has written its row of the staged tile.
  // DOFREE: the dO buffer may be refilled: the MMA warp's commit after the item's last dP
  // product and every elementwise thread (done reading dO for D).
  static constexpr int DOFREE_COUNT = 1 + 256;
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

// Epilogue staging: NC columns of an fp32 accumulator row in tensor memory, times `mult`,
// to fp16 in row r of a shared-memory tile laid out as the TMA boxes (`chunk` bytes per
// 64-column box, 128-byte swizzle) from 16-byte unit u0 on; a TMA store then writes the
// tile out with whole-line transactions (a thread per row storing to global memory
// directly would touch 32 rows per instruction).
template <int NC>
__device__ __forceinline__ void bwd_stage_row(uint32_t acc_tmem, uint32_t tile, int chunk, int r, int u0,
                                              float mult) {
  constexpr int W = NC % 64 == 0 ? 64 : 32;  // columns per tensor-memory load
#pragma unroll 1
  for (int cw = 0; cw < NC / W; ++cw) {
    uint32_t v[W];
    if constexpr (W == 64)
      tmem_ld32x64(acc_tmem + cw * W, v);
    else
      tmem_ld32x32(acc_tmem + cw * W, v);
#pragma unroll
    for (int q4 = 0; q4 < W / 8; ++q4)
      st_shared_v4(bwd_chunk_addr(tile, chunk, r, u0 + (W / 8) * cw + q4),
                   pack_f16x2(__uint_as_float(v[8 * q4]) * mult, __uint_as_float(v[8 * q4 + 1]) * mult),
                   pack_f16x2(__uint_as_float(v[8 * q4 + 2]) * mult, __uint_as_float(v[8 * q4 + 3]) * mult),
                   pack_f16x2(__uint_as_float(v[8 * q4 + 4]) * mult, __uint_as_float(v[8 * q4 + 5]) * mult),
                   pack_f16x2(__uint_as_float(v[8 * q4 + 6]) * mult, __uint_as_float(v[8 * q4 + 7]) * mult));
  }
}

// ======================================================================== dK / dV
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                         const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  if (base & 1023u) {  // the layout has no alignment slack (every thread leaves here)
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, kDevSmemAlign);
    return;
  }
  uint8_t *const base_ptr = smem_raw;
  const uint32_t k_s = base, v_s = base + C::RTILE, q_ring = base + C::KV_OFF_Q, do_ring = base + C::KV_OFF_DO;
  float *const stat_s = reinterpret_cast<float *>(base_ptr + C::KV_OFF_ST);  // [2][lse 128 | D 128]
  const uint32_t stat_a = base + C::KV_OFF_ST;
  const uint32_t bar_s = base + C::KV_OFF_BAR;
  uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + C::KV_OFF_BAR + 8 * C::KB_N);
  volatile uint32_t *const abort_flag = tmem_slot + 1;
  auto BAR = [&](int i) -> uint32_t { return bar_s + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long LIM = p.wait_limit;
  const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  // Item idx: key tile kt of head bh (kt ascending = longest first when causal); its steps
  // are the 128-row query tiles from q_first on.
  auto decode = [&](int idx, int &bh, int &kt, int &q_first, int &nsteps) {
    kt = idx / p.BH;
    bh = idx - kt * p.BH;
    q_first = CAUSAL ? kt : 0;
    nsteps = p.n128 - q_first;
  };
  auto q_tile = [&](int gg) -> uint32_t { return q_ring + (gg % C::NQS) * C::RTILE; };
  auto do_tile = [&](int gg) -> uint32_t { return do_ring + (gg % C::NDS) * C::RTILE; };

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::KB_KVFULL), 1);
    mbar_init(BAR(C::KB_KVFREE), 1);
    mbar_init(BAR(C::KB_IDONE), 1);
    for (int i = 0; i < C::NQS; ++i) {
      mbar_init(BAR(C::KB_QFULL + i), 1);
      mbar_init(BAR(C::KB_QEMPTY + i), 1);
    }
    for (int i = 0; i < C::NDS; ++i) {
      mbar_init(BAR(C::KB_DOFULL + i), 1);
      mbar_init(BAR(C::KB_DOEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(C::KB_STFULL + i), 1);
      mbar_init(BAR(C::KB_STEMPTY + i), 256);
    }
    mbar_init(BAR(C::KB_SFULL), 1);
    mbar_init(BAR(C::KB_DPFULL), 1);
    mbar_init(BAR(C::KB_PFULL), 256);
    mbar_init(BAR(C::KB_DSFULL), 256);
    mbar_init(BAR(C::KB_DRAIN), 1);
    for (int i = 0; i < C::NQS; ++i) mbar_init(BAR(C::KB_STGQ + i), 1);
    for (int i = 0; i < C::NDS; ++i) mbar_init(BAR(C::KB_STGDO + i), 1);
    mbar_init(BAR(C::KB_STAGED), 256);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dk);
    tma_prefetch_desc(&tm_dv);
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
  // The producer and the MMA thread start on Q, K, V and dO (which the dQ kernel does not
  // write) before the dQ kernel has completed; the producer waits for it before its first
  // load of the row statistics (which the dQ kernel writes), every other thread here.  The
  // dQ kernel lets this one launch only after its own wait, so the kernels before both
  // have completed by then.
  if (warp >= 2) grid_wait_prior();
  // Tensor memory: S^T [0,128) (P^T packed into [0,32) and [64,96)), dP^T [128,256) (dS^T
  // likewise), dV [256, 256+D), dK [256+D, 256+2D).
  constexpr uint32_t C_S = 0, C_DP = 128, C_DV = 256, C_DK = 256 + D;
  auto a_col = [](int kk) -> uint32_t { return static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8); };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int g = 0, nq = 0, ndo = 0, nst = 0, kv_loads = 0;
      // The epilogue stages dK and dV in the Q and dO slots of its item's last step: such a
      // slot is refilled only once the TMA stores have read it.  Bit b of stg_pend: slot b
      // (Q slots from bit 0, dO slots from bit 8) awaits that; of stg_par: the phase.
      uint32_t stg_pend = 0u, stg_par = 0u;
      auto stage_read = [&](int b, int bar) -> bool {
        if (!((stg_pend >> b) & 1u)) return true;
        const uint32_t ph = (stg_par >> b) & 1u;
        stg_pend &= ~(1u << b);
        stg_par ^= 1u << b;
        return wait_bounded(BAR(bar), ph, abort_flag, p.status, kDevTimeoutLoad, LIM);
      };
      for (int r = 0; ok && r * G < p.items; ++r) {
        const int idx = bwd_item(r, cta, G);
        if (idx >= p.items) continue;
        int bh, kt, q_first, nsteps;
        decode(idx, bh, kt, q_first, nsteps);
        for (int s = 0; s < nsteps; ++s, ++g) {
          const int qi = q_first + s;
          if (!(ok = wait_bounded(BAR(C::KB_QEMPTY + g % C::NQS), ((g / C::NQS) & 1) ^ 1u, abort_flag, p.status,
                                  kDevTimeoutLoad, LIM) &&
                     stage_read(g % C::NQS, C::KB_STGQ + g % C::NQS)))
            break;
          mbar_arrive_expect_tx(BAR(C::KB_QFULL + g % C::NQS), C::RTILE);
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(q_tile(g) + c * C::RCHUNK, &tm_q, c * 64, qi * 128, bh, BAR(C::KB_QFULL + g % C::NQS));
          ++nq;
          if (s == 0) {
            // K and V of this item, once the previous item's last S^T and dP^T products (the
            // only readers of K and V) are complete.
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
          if (!(ok = wait_bounded(BAR(C::KB_DOEMPTY + g % C::NDS), ((g / C::NDS) & 1) ^ 1u, abort_flag, p.status,
                                  kDevTimeoutLoad, LIM) &&
                     stage_read(8 + g % C::NDS, C::KB_STGDO + g % C::NDS)))
            break;
          mbar_arrive_expect_tx(BAR(C::KB_DOFULL + g % C::NDS), C::RTILE);
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(do_tile(g) + c * C::RCHUNK, &tm_do, c * 64, qi * 128, bh, BAR(C::KB_DOFULL + g % C::NDS));
          ++ndo;
          // The 128 rows' statistics, written by the dQ kernel (byte offsets multiples of 512).
          if (nst == 0) grid_wait_prior();
          if (!(ok = wait_bounded(BAR(C::KB_STEMPTY + (g & 1)), ((g >> 1) & 1) ^ 1u, abort_flag, p.status,
                                  kDevTimeoutLoad, LIM)))
            break;
          const long long wrow = static_cast<long long>(bh) * p.Lp + qi * 128;
          mbar_arrive_expect_tx(BAR(C::KB_STFULL + (g & 1)), 1024);
          bulk_load(stat_a + (g & 1) * 1024, p.ws_lse2 + wrow, 512, BAR(C::KB_STFULL + (g & 1)));
          bulk_load(stat_a + (g & 1) * 1024 + 512, p.ws_d + wrow, 512, BAR(C::KB_STFULL + (g & 1)));
          ++nst;
        }
        stg_pend |= (1u << ((g - 1) % C::NQS)) | (1u << (8 + (g - 1) % C::NDS));
      }
      // Drain: every load issued lands before the CTA may exit.
      if (kv_loads > 0) wait_drain(BAR(C::KB_KVFULL), (kv_loads - 1) & 1, LIM);
      for (int i = nq > C::NQS ? nq - C::NQS : 0; i < nq; ++i)
        wait_drain(BAR(C::KB_QFULL + i % C::NQS), (i / C::NQS) & 1, LIM);
      for (int i = ndo > C::NDS ? ndo - C::NDS : 0; i < ndo; ++i)
        wait_drain(BAR(C::KB_DOFULL + i % C::NDS), (i / C::NDS) & 1, LIM);
      for (int i = nst > 2 ? nst - 2 : 0; i < nst; ++i) wait_drain(BAR(C::KB_STFULL + (i & 1)), (i >> 1) & 1, LIM);
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
      auto q_ready = [&](int gg) { return wait(C::KB_QFULL + gg % C::NQS, (gg / C::NQS) & 1); };
      auto do_ready = [&](int gg) { return wait(C::KB_DOFULL + gg % C::NDS, (gg / C::NDS) & 1); };
      // S^T = K Q^T and dP^T = V dO^T of global step gg (head_dim summed over its chunks).
      auto issue_s = [&](int gg) {
        const SDesc qb = sdesc_split(sdesc_sw128(q_tile(gg), 16, 1024));
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + C_S, ka, c * C::RCHUNK + kk * 32, qb, c * C::RCHUNK + kk * 32, C::IDESC_S128,
                        (c | kk) != 0 ? 1u : 0u);
        umma_commit(BAR(C::KB_SFULL));
      };
      auto issue_dp = [&](int gg) {
        const SDesc dob = sdesc_split(sdesc_sw128(do_tile(gg), 16, 1024));
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + C_DP, va, c * C::RCHUNK + kk * 32, dob, c * C::RCHUNK + kk * 32, C::IDESC_S128,
                        (c | kk) != 0 ? 1u : 0u);
        umma_commit(BAR(C::KB_DPFULL));
      };
      for (int r = 0; ok && r * G < p.items; ++r) {
        const int idx = bwd_item(r, cta, G);
        if (idx >= p.items) continue;
        int bh, kt, q_first, nsteps;
        decode(idx, bh, kt, q_first, nsteps);
        if (!(ok = wait(C::KB_KVFULL, it & 1) && q_ready(g))) break;
        tc_fence_after();
        issue_s(g);
        if (!(ok = do_ready(g))) break;
        tc_fence_after();
        issue_dp(g);
        if (nsteps == 1) umma_commit(BAR(C::KB_KVFREE));  // the item's last S^T, dP^T are issued
        for (int s = 0; s < nsteps; ++s, ++g) {
          const bool more = s + 1 < nsteps;
          // dV += P^T dO; then this step's dO tile is free.
          if (!(ok = wait(C::KB_PFULL, g & 1))) break;
          tc_fence_after();
          const SDesc dom = sdesc_split(sdesc_sw128(do_tile(g), C::RCHUNK, 1024));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts_off(tmem + C_DV, tmem + C_S + a_col(kk), dom, kk * 2048, C::IDESC_ACC, (s > 0 || kk > 0) ? 1u : 0u);
          umma_commit(BAR(C::KB_DOEMPTY + g % C::NDS));
          if (more) {
            if (!(ok = q_ready(g + 1))) break;
            tc_fence_after();
            issue_s(g + 1);  // into S^T, read in order after dV above
          }
          // dK += dS^T Q; then this step's Q tile is free.
          if (!(ok = wait(C::KB_DSFULL, g & 1))) break;
          tc_fence_after();
          const SDesc qm = sdesc_split(sdesc_sw128(q_tile(g), C::RCHUNK, 1024));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts_off(tmem + C_DK, tmem + C_DP + a_col(kk), qm, kk * 2048, C::IDESC_ACC, (s > 0 || kk > 0) ? 1u : 0u);
          umma_commit(BAR(C::KB_QEMPTY + g % C::NQS));
          if (more) {
            if (!(ok = do_ready(g + 1))) break;
            tc_fence_after();
            issue_dp(g + 1);  // into dP^T, read in order after dK above
            if (s + 2 == nsteps) umma_commit(BAR(C::KB_KVFREE));
          }
        }
        if (!ok) break;
        umma_commit(BAR(C::KB_IDONE));  // dV, dK final
        ++it;
      }
      umma_commit(BAR(C::KB_DRAIN));  // every MMA issued so far is complete
      wait_drain(BAR(C::KB_DRAIN), 0, LIM);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ elementwise warpgroups
    const int h = (warp - 4) >> 2;        // query columns [64 h, 64 h + 64) of every tile
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // key row of the tile == tensor-memory lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.c2;
    auto wait_warp = [&](int b, uint32_t ph) -> bool {
      return __all_sync(0xffffffffu, wait_bounded(BAR(b), ph, abort_flag, p.status, kDevTimeoutSoftmax, LIM));
    };
    bool ok = true;
    int g = 0, it = 0;
    // Thread (warp 4, lane 0) issues the epilogue's TMA stores; it hands their slots back
    // to the producer (once the stores have read them) during the next item's first step,
    // so that the read does not hold up that step.  stg_gl: last step of the item whose
    // slots are still held, or -1.
    int stg_gl = -1;
    for (int r = 0; ok && r * G < p.items; ++r) {
      const int idx = bwd_item(r, cta, G);
      if (idx >= p.items) continue;
      int bh, kt, q_first, nsteps;
      decode(idx, bh, kt, q_first, nsteps);
      for (int s = 0; s < nsteps; ++s, ++g) {
        const float *const lse_h = stat_s + (g & 1) * 256 + 64 * h;
        const float *const dd_h = lse_h + 128;
        const uint32_t s_col = tmem + lane_base + C_S + 64 * h, dp_col = tmem + lane_base + C_DP + 64 * h;
        if (!(ok = wait_warp(C::KB_SFULL, g & 1) && wait_warp(C::KB_STFULL + (g & 1), (g >> 1) & 1))) break;
        tc_fence_after();
        // P phase: P^T = exp2(S^T c2 - LSE log2 e), masked on the diagonal tile (query
        // before key), packed to fp16 into the first 32 of its 64 columns.
        const bool diag = CAUSAL && s == 0;
        float pv[64];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sr[32];
          tmem_ld32x32(s_col + 32 * half, sr);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int col = 32 * half + c;
            float pp = ex2_approx(fmaf(__uint_as_float(sr[c]), c2, -lse_h[col]));
            if (diag && 64 * h + col < row) pp = 0.f;
            pv[col] = pp;
          }
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack_f16x2(pv[2 * i], pv[2 * i + 1]);
          tmem_st32x32(s_col, pk);
        }
        tc_fence_before();
        mbar_arrive(BAR(C::KB_PFULL));
        if (stg_gl >= 0) {  // only the storing thread holds slots
          bulk_wait_read0();
          mbar_arrive(BAR(C::KB_STGQ + stg_gl % C::NQS));
          mbar_arrive(BAR(C::KB_STGDO + stg_gl % C::NDS));
          stg_gl = -1;
        }
        // dS phase: dS^T = P^T (dP^T - D), packed likewise.
        if (!(ok = wait_warp(C::KB_DPFULL, g & 1))) break;
        tc_fence_after();
        {
          uint32_t dk[32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t dr[32];
            tmem_ld32x32(dp_col + 32 * half, dr);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int col = 32 * half + 2 * i;
              dk[16 * half + i] = pack_f16x2(pv[col] * (__uint_as_float(dr[2 * i]) - dd_h[col]),
                                             pv[col + 1] * (__uint_as_float(dr[2 * i + 1]) - dd_h[col + 1]));
            }
          }
          tmem_st32x32(dp_col, dk);
        }
        tc_fence_before();
        // The statistics read above are refilled by a bulk copy (async proxy).
        fence_proxy_async_smem();
        mbar_arrive(BAR(C::KB_STEMPTY + (g & 1)));
        mbar_arrive(BAR(C::KB_DSFULL));
      }
      if (!ok) break;
      // ---------------------------------------------------------------- epilogue
      // Warpgroup 0 stages dV in the dO slot of the item's last step, warpgroup 1 stages
      // scale * dK in its Q slot (both free once the item's last products are complete), one
      // key row per thread; one thread then stores both tiles by TMA (rows past L clipped).
      if (!(ok = wait_warp(C::KB_IDONE, it & 1))) break;
      tc_fence_after();
      const int gl = g - 1;
      bwd_stage_row<D>(tmem + lane_base + (h == 0 ? C_DV : C_DK), h == 0 ? do_tile(gl) : q_tile(gl), C::RCHUNK,
                       row, 0, h == 0 ? 1.0f : p.scale);
      tc_fence_before();
      fence_proxy_async_smem();  // the staged rows are read by TMA (async proxy)
      mbar_arrive(BAR(C::KB_STAGED));
      if (warp == 4 && lane == 0) {
        ok = wait_bounded(BAR(C::KB_STAGED), it & 1, abort_flag, p.status, kDevTimeoutSoftmax, LIM);
        if (ok && *abort_flag == 0u) {
          for (int c = 0; c < C::NCH; ++c) {
            tma_store_3d(&tm_dv, do_tile(gl) + c * C::RCHUNK, c * 64, kt * 128, bh);
            tma_store_3d(&tm_dk, q_tile(gl) + c * C::RCHUNK, c * 64, kt * 128, bh);
          }
          bulk_commit();
        }
        stg_gl = gl;
      }
      if (warp == 4) ok = __shfl_sync(0xffffffffu, ok, 0);
      ++it;
    }
    if (warp == 4 && lane == 0) bulk_wait0();  // the stores are complete before the CTA exits
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ======================================================================== dQ
// Steps of 128 key rows: K and V stream through rings of their own (K is read by S and by
// the dQ product of its step, V only by dP), S is double-buffered in tensor memory.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t q_s = base, do_s = base + C::RTILE, k_ring = base + C::Q_OFF_K, v_ring = base + C::Q_OFF_V;
  float *const dpart = reinterpret_cast<float *>(base_ptr + C::Q_OFF_ST);  // [half][128 rows]
  const uint32_t bar_s = base + C::Q_OFF_BAR;
  uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + C::Q_OFF_BAR + 8 * C::QB_N);
  volatile uint32_t *const abort_flag = tmem_slot + 1;
  auto BAR = [&](int i) -> uint32_t { return bar_s + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long LIM = p.wait_limit;
  const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  // Item idx: query tile qt of head bh, longest first (causal: the last query tiles see the
  // most key tiles); its steps are the 128-row key tiles 0 .. nsteps-1.
  auto decode = [&](int idx, int &bh, int &qt, int &nsteps) {
    const int grp = idx / p.BH;
    bh = idx - grp * p.BH;
    qt = CAUSAL ? p.n128 - 1 - grp : grp;
    nsteps = CAUSAL ? qt + 1 : p.n128;
  };
  auto k_tile = [&](int gg) -> uint32_t { return k_ring + (gg % C::NKS) * C::RTILE; };
  auto v_tile = [&](int gg) -> uint32_t { return v_ring + (gg % C::NVS) * C::RTILE; };

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::QB_QFULL), 1);
    mbar_init(BAR(C::QB_QFREE), 1);
    mbar_init(BAR(C::QB_DOFULL), 1);
    mbar_init(BAR(C::QB_DOFREE), C::DOFREE_COUNT);
    mbar_init(BAR(C::QB_DPART), 256);
    mbar_init(BAR(C::QB_IDONE), 1);
    for (int i = 0; i < C::NKS; ++i) {
      mbar_init(BAR(C::QB_KFULL + i), 1);
      mbar_init(BAR(C::QB_KEMPTY + i), 1);
    }
    for (int i = 0; i < C::NVS; ++i) {
      mbar_init(BAR(C::QB_VFULL + i), 1);
      mbar_init(BAR(C::QB_VEMPTY + i), 1);
    }
    mbar_init(BAR(C::QB_SFULL), 1);
    mbar_init(BAR(C::QB_SFULL + 1), 1);
    mbar_init(BAR(C::QB_DPFULL), 1);
    mbar_init(BAR(C::QB_DSFULL), 256);
    mbar_init(BAR(C::QB_DRAIN), 1);
    for (int i = 0; i < C::NKS; ++i) mbar_init(BAR(C::QB_STGK + i), 1);
    mbar_init(BAR(C::QB_STAGED), 256);
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Dependents launch only once the kernels before this one have completed (the dK/dV
  // kernel reads its inputs before its own wait).
  grid_wait_prior();
  grid_launch_dependents();
  // Tensor memory: S of step gg at [128 (gg & 1), +128), dP at [256, 384) (dS packed over
  // [256, 288) and [320, 352)), dQ at [384, 384 + D).
  constexpr uint32_t C_DP = 256, C_DQ = 384;
  static_assert(C_DQ + D <= BwdCfg<D>::TMEM_COLS, "tensor memory budget");
  auto c_s = [](int gg) -> uint32_t { return static_cast<uint32_t>(gg & 1) * 128u; };

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int g = 0, nk = 0, nv = 0, it = 0;  // K and V tiles issued, items whose Q and dO are issued
      bool q_pending = false;              // this item's Q is issued, its dO not yet
      // The epilogue stages dQ in the K slot of its item's last step: such a slot is refilled
      // only once the TMA store has read it.  Bit b of stg_pend: slot b awaits that; of
      // stg_par: the phase.
      uint32_t stg_pend = 0u, stg_par = 0u;
      auto stage_read = [&](int b) -> bool {
        if (!((stg_pend >> b) & 1u)) return true;
        const uint32_t ph = (stg_par >> b) & 1u;
        stg_pend &= ~(1u << b);
        stg_par ^= 1u << b;
        return wait_bounded(BAR(C::QB_STGK + b), ph, abort_flag, p.status, kDevTimeoutLoad, LIM);
      };
      for (int r = 0; ok && r * G < p.items; ++r) {
        const int idx = bwd_item(r, cta, G);
        if (idx >= p.items) continue;
        int bh, qt, nsteps;
        decode(idx, bh, qt, nsteps);
        for (int s = 0; s < nsteps; ++s, ++g) {
          if (!(ok = wait_bounded(BAR(C::QB_KEMPTY + g % C::NKS), ((g / C::NKS) & 1) ^ 1u, abort_flag, p.status,
                                  kDevTimeoutLoad, LIM) &&
                     stage_read(g % C::NKS)))
            break;
          mbar_arrive_expect_tx(BAR(C::QB_KFULL + g % C::NKS), C::RTILE);
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(k_tile(g) + c * C::RCHUNK, &tm_k, c * 64, s * 128, bh, BAR(C::QB_KFULL + g % C::NKS));
          ++nk;
          if (s == 0) {
            // Q and dO of this item, once the previous item's last S (Q) and last dP and D
            // (dO) are complete.
            if (it >= 1 && !(ok = wait_bounded(BAR(C::QB_QFREE), (it - 1) & 1, abort_flag, p.status, kDevTimeoutLoad,
                                               LIM)))
              break;
            mbar_arrive_expect_tx(BAR(C::QB_QFULL), C::RTILE);
            for (int c = 0; c < C::NCH; ++c)
              tma_load_3d(q_s + c * C::RCHUNK, &tm_q, c * 64, qt * 128, bh, BAR(C::QB_QFULL));
            q_pending = true;
            if (it >= 1 && !(ok = wait_bounded(BAR(C::QB_DOFREE), (it - 1) & 1, abort_flag, p.status, kDevTimeoutLoad,
                                               LIM)))
              break;
            mbar_arrive_expect_tx(BAR(C::QB_DOFULL), C::RTILE);
            for (int c = 0; c < C::NCH; ++c)
              tma_load_3d(do_s + c * C::RCHUNK, &tm_do, c * 64, qt * 128, bh, BAR(C::QB_DOFULL));
            q_pending = false;
            ++it;
          }
          if (!(ok = wait_bounded(BAR(C::QB_VEMPTY + g % C::NVS), ((g / C::NVS) & 1) ^ 1u, abort_flag, p.status,
                                  kDevTimeoutLoad, LIM)))
            break;
          mbar_arrive_expect_tx(BAR(C::QB_VFULL + g % C::NVS), C::RTILE);
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(v_tile(g) + c * C::RCHUNK, &tm_v, c * 64, s * 128, bh, BAR(C::QB_VFULL + g % C::NVS));
          ++nv;
        }
        stg_pend |= 1u << ((g - 1) % C::NKS);
      }
      // Drain: every load issued lands before the CTA may exit.
      if (it + (q_pending ? 1 : 0) > 0) wait_drain(BAR(C::QB_QFULL), (it + (q_pending ? 1 : 0) - 1) & 1, LIM);
      if (it > 0) wait_drain(BAR(C::QB_DOFULL), (it - 1) & 1, LIM);
      for (int i = nk > C::NKS ? nk - C::NKS : 0; i < nk; ++i)
        wait_drain(BAR(C::QB_KFULL + i % C::NKS), (i / C::NKS) & 1, LIM);
      for (int i = nv > C::NVS ? nv - C::NVS : 0; i < nv; ++i)
        wait_drain(BAR(C::QB_VFULL + i % C::NVS), (i / C::NVS) & 1, LIM);
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
      auto k_ready = [&](int gg) { return wait(C::QB_KFULL + gg % C::NKS, (gg / C::NKS) & 1); };
      auto v_ready = [&](int gg) { return wait(C::QB_VFULL + gg % C::NVS, (gg / C::NVS) & 1); };
      // S = Q K^T of global step gg into its buffer.
      auto issue_s = [&](int gg) {
        const SDesc kb = sdesc_split(sdesc_sw128(k_tile(gg), 16, 1024));
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + c_s(gg), qa, c * C::RCHUNK + kk * 32, kb, c * C::RCHUNK + kk * 32, C::IDESC_S128,
                        (c | kk) != 0 ? 1u : 0u);
        umma_commit(BAR(C::QB_SFULL + (gg & 1)));
      };
      // dP = dO V^T of global step gg; its V tile is free once this completes.
      auto issue_dp = [&](int gg) {
        const SDesc vb = sdesc_split(sdesc_sw128(v_tile(gg), 16, 1024));
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_off(tmem + C_DP, doa, c * C::RCHUNK + kk * 32, vb, c * C::RCHUNK + kk * 32, C::IDESC_S128,
                        (c | kk) != 0 ? 1u : 0u);
        umma_commit(BAR(C::QB_DPFULL));
        umma_commit(BAR(C::QB_VEMPTY + gg % C::NVS));
      };
      for (int r = 0; ok && r * G < p.items; ++r) {
        const int idx = bwd_item(r, cta, G);
        if (idx >= p.items) continue;
        int bh, qt, nsteps;
        decode(idx, bh, qt, nsteps);
        if (!(ok = wait(C::QB_QFULL, it & 1) && k_ready(g))) break;
        tc_fence_after();
        issue_s(g);
        if (!(ok = wait(C::QB_DOFULL, it & 1) && v_ready(g))) break;
        tc_fence_after();
        issue_dp(g);
        if (nsteps > 1) {
          if (!(ok = k_ready(g + 1))) break;
          tc_fence_after();
          issue_s(g + 1);
        }
        if (nsteps <= 2) umma_commit(BAR(C::QB_QFREE));  // the item's last S is issued
        if (nsteps <= 1) umma_commit(BAR(C::QB_DOFREE));  // and its last dP
        for (int s = 0; s < nsteps; ++s, ++g) {
          // dQ += dS K
          if (!(ok = wait(C::QB_DSFULL, g & 1))) break;
          tc_fence_after();
          const SDesc km = sdesc_split(sdesc_sw128(k_tile(g), C::RCHUNK, 1024));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts_off(tmem + C_DQ, tmem + C_DP + static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8), km,
                        kk * 2048, C::IDESC_ACC, (s > 0 || kk > 0) ? 1u : 0u);
          umma_commit(BAR(C::QB_KEMPTY + g % C::NKS));
          if (s + 1 < nsteps) {
            if (!(ok = v_ready(g + 1))) break;
            tc_fence_after();
            issue_dp(g + 1);  // into the dP columns, read in order after dQ above
            if (s + 2 == nsteps) umma_commit(BAR(C::QB_DOFREE));
          }
          if (s + 2 < nsteps) {
            if (!(ok = k_ready(g + 2))) break;
            tc_fence_after();
            issue_s(g + 2);  // into this step's S buffer (its P was consumed before dS)
            if (s + 3 == nsteps) umma_commit(BAR(C::QB_QFREE));
          }
        }
        if (!ok) break;
        umma_commit(BAR(C::QB_IDONE));  // dQ final
        ++it;
      }
      umma_commit(BAR(C::QB_DRAIN));
      wait_drain(BAR(C::QB_DRAIN), 0, LIM);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ elementwise warpgroups
    const int h = (warp - 4) >> 2;        // key columns [64 h, 64 h + 64) of every tile;
                                          // head_dim columns [h D/2, (h+1) D/2) of D and dQ
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // query row of the tile == tensor-memory lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.c2;
    constexpr float kLog2e = 1.4426950408889634f;
    constexpr int CPH = D / 16;           // 16-byte chunks of half a row
    auto wait_warp = [&](int b, uint32_t ph) -> bool {
      return __all_sync(0xffffffffu, wait_bounded(BAR(b), ph, abort_flag, p.status, kDevTimeoutSoftmax, LIM));
    };
    // O and LSE for the item at list round r, loaded one item ahead of their use.  O is read
    // coalesced: of the 32 x CPH 16-byte chunks of this warp's 32 rows (half h of each),
    // this thread holds chunks q = i 32 + lane (row q / CPH, chunk q % CPH of the half), so
    // that one load instruction covers whole line segments; LSE is this thread's own row.
    // The loads are unconditional (item and row clamped into range; o_valid marks a row
    // below L), so that nothing waits for them before their use.
    uint4 o_reg[CPH];
    float lse_reg;
    bool o_valid;
    auto fetch = [&](int r) {
      int fbh, fqt, fn;
      decode(min(bwd_item(r, cta, G), p.items - 1), fbh, fqt, fn);
      const long long hrow = static_cast<long long>(fbh) * p.L;
      o_valid = fqt * 128 + row < p.L;
      lse_reg = __ldg(p.lse + hrow + min(fqt * 128 + row, p.L - 1));
#pragma unroll
      for (int i = 0; i < CPH; ++i) {
        const int q = i * 32 + lane;
        const long long orow = hrow + min(fqt * 128 + quarter * 32 + q / CPH, p.L - 1);
        o_reg[i] = __ldg(reinterpret_cast<const uint4 *>(p.o + orow * D) + CPH * h + q % CPH);
      }
    };
    bool ok = true;
    int g = 0, it = 0;
    // Thread (warp 4, lane 0) issues the epilogue's TMA store; it hands the K slot back to
    // the producer (once the store has read it) at the next item's first step, so that the
    // read does not hold up the next item.  stg_gl: last step of the item whose slot is
    // still held, or -1.
    int stg_gl = -1;
    fetch(0);  // this CTA's first item: bwd_item(0, cta, G) = cta < G <= items
    for (int r = 0; ok && r * G < p.items; ++r) {
      const int idx = bwd_item(r, cta, G);
      if (idx >= p.items) continue;
      int bh, qt, nsteps;
      decode(idx, bh, qt, nsteps);
      const int qrow = qt * 128 + row;
      // Row statistics: D = dO . O, each warpgroup over its half of the row, the halves
      // added through shared memory; LSE log2(e).  Both go to the workspace.
      if (!(ok = wait_warp(C::QB_DOFULL, it & 1))) break;
      // Every dO chunk is read before any product is formed: the shared-memory reads are
      // ordered with the stores below, so reading them one row at a time would serialise
      // the loop.
      uint4 do_reg[CPH];
#pragma unroll
      for (int i = 0; i < CPH; ++i) {
        const int q = i * 32 + lane, rw = quarter * 32 + q / CPH;
        do_reg[i] = ld_shared_v4(bwd_chunk_addr(do_s, C::RCHUNK, rw, CPH * h + q % CPH));
      }
      float part[CPH];
#pragma unroll
      for (int i = 0; i < CPH; ++i) part[i] = bwd_dot8(do_reg[i], o_reg[i]);
#pragma unroll
      for (int m = 1; m < CPH; m <<= 1)
#pragma unroll
        for (int i = 0; i < CPH; ++i) part[i] += __shfl_xor_sync(0xffffffffu, part[i], m);
#pragma unroll
      for (int i = 0; i < CPH; ++i) {
        const int q = i * 32 + lane, rw = quarter * 32 + q / CPH;
        if (q % CPH == 0) dpart[h * 128 + rw] = qt * 128 + rw < p.L ? part[i] : 0.f;
      }
      const float lrow = o_valid ? lse_reg * kLog2e : INFINITY;
      mbar_arrive(BAR(C::QB_DPART));
      if (!(ok = wait_warp(C::QB_DPART, it & 1))) break;
      const float drow = dpart[row] + dpart[128 + row];
      if (h == 0) {
        const long long w = static_cast<long long>(bh) * p.Lp + qt * 128 + row;
        p.ws_lse2[w] = lrow;
        p.ws_d[w] = drow;
      }
      // dO (read above, in the generic proxy) is refilled by TMA once this arrives.
      fence_proxy_async_smem();
      mbar_arrive(BAR(C::QB_DOFREE));
      // The next item's O and LSE, while this item runs.
      {
        int rn = r + 1;
        while (rn * G < p.items && bwd_item(rn, cta, G) >= p.items) ++rn;
        fetch(rn);
      }
      for (int s = 0; s < nsteps; ++s, ++g) {
        const uint32_t s_col = tmem + lane_base + c_s(g) + 64 * h, dp_col = tmem + lane_base + C_DP + 64 * h;
        // P (registers only): P = exp2(S c2 - LSE log2 e), masked where the key comes after
        // the query (diagonal tile) or lies past L.
        if (!(ok = wait_warp(C::QB_SFULL + (g & 1), (static_cast<uint32_t>(g) >> 1) & 1u))) break;
        tc_fence_after();
        if (stg_gl >= 0) {  // only the storing thread holds a slot
          bulk_wait_read0();
          mbar_arrive(BAR(C::QB_STGK + stg_gl % C::NKS));
          stg_gl = -1;
        }
        const int key0 = s * 128 + 64 * h;
        const bool edge = (CAUSAL && s == qt) || key0 + 64 > p.L;
        float pv[64];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sr[32];
          tmem_ld32x32(s_col + 32 * half, sr);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int col = 32 * half + c;
            float pp = ex2_approx(fmaf(__uint_as_float(sr[c]), c2, -lrow));
            if (edge && ((CAUSAL && key0 + col > qrow) || key0 + col >= p.L)) pp = 0.f;
            pv[col] = pp;
          }
        }
        // dS = P (dP - D), packed to fp16 into the first 32 of its 64 columns.
        if (!(ok = wait_warp(C::QB_DPFULL, g & 1))) break;
        tc_fence_after();
        {
          uint32_t dk[32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t dr[32];
            tmem_ld32x32(dp_col + 32 * half, dr);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int col = 32 * half + 2 * i;
              dk[16 * half + i] = pack_f16x2(pv[col] * (__uint_as_float(dr[2 * i]) - drow),
                                             pv[col + 1] * (__uint_as_float(dr[2 * i + 1]) - drow));
            }
          }
          tmem_st32x32(dp_col, dk);
        }
        tc_fence_before();
        mbar_arrive(BAR(C::QB_DSFULL));
      }
      if (!ok) break;
      // ---------------------------------------------------------------- epilogue
      // scale * dQ, staged in the K slot of the item's last step (free once the item's last
      // product is complete): warpgroup h writes columns [h D/2, (h+1) D/2) of its query row;
      // one thread then stores the tile by TMA (rows past L clipped).
      if (!(ok = wait_warp(C::QB_IDONE, it & 1))) break;
      tc_fence_after();
      const int gl = g - 1;
      bwd_stage_row<D / 2>(tmem + lane_base + C_DQ + h * (D / 2), k_tile(gl), C::RCHUNK, row, h * (D / 16),
                           p.scale);
      tc_fence_before();
      fence_proxy_async_smem();  // the staged rows are read by TMA (async proxy)
      mbar_arrive(BAR(C::QB_STAGED));
      if (warp == 4 && lane == 0) {
        ok = wait_bounded(BAR(C::QB_STAGED), it & 1, abort_flag, p.status, kDevTimeoutSoftmax, LIM);
        if (ok && *abort_flag == 0u) {
          for (int c = 0; c < C::NCH; ++c) tma_store_3d(&tm_dq, k_tile(gl) + c * C::RCHUNK, c * 64, qt * 128, bh);
          bulk_commit();
        }
        stg_gl = gl;
      }
      if (warp == 4) ok = __shfl_sync(0xffffffffu, ok, 0);
      ++it;
    }
    if (warp == 4 && lane == 0) bulk_wait0();  // the store is complete before the CTA exits
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
