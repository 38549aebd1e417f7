// attn_fwd_pp.cuh -- two-tile SDPA forward for head_dim 64 and 128 on sm_103a.
//
// Same mathematics as attn_fwd_kernel.cuh ("An Optimal Mapper Meets a Real GPU",
// "Ground rules" / "Experiment one"): O = softmax(scale * Q K^T + causal mask) V and the
// row LSE, fused into one persistent kernel.  The work item is a 256-row query block
// split into two 128-row tiles Q0 and Q1 ("slots") that share every K/V tile the
// producer loads (half the K/V traffic per query row of the single-tile kernel).  Each
// slot has its own S buffer and O accumulator in tensor memory and its own softmax
// warpgroup:
//   TMEM columns  S0 [0,128)  S1 [128,256)  O0 [256, 256+D)  O1 [256+D, 256+2D).
//
// One thread issues every MMA, both slots' in one stream (see PPIssuer): PV_a of tile j
// comes right before QK_a of tile j+1 from that thread, so when softmax warpgroup a sees
// S of tile j+1 complete, PV of tile j is complete too (tcgen05 operations of one thread
// complete in order) and the lazy O rescale never waits for a PV; and the two slots
// alternate on the tensor core, so each softmax warpgroup works while the tensor core
// runs the other slot's PV and QK.  Under the causal mask Q0 needs key tiles 0..2qb and
// Q1 needs 0..2qb+1; the last one belongs to Q1 alone.
//
// Warp roles (384 threads):
//   warp 0      K/V producer: per item, K_0, V_0, K_1, V_1, ... into an mbarrier ring; a
//               stage is free again once slot 1's QK or PV of it is done (slot 1 reads every
//               K/V tile of an item, always after slot 0; one commit covers both).
//   warp 1      TMEM owner + MMA issuer;  warp 2 idle.
//   warp 3      Q loader and O store issuer.  Each slot has one Q buffer, released by the
//               commit of the slot's last QK of an item, so the next item's Q tile lands
//               while the last softmax and PV of the current one run.  Finished O tiles
//               go through one staging buffer that the slots take in turn (slot 0, then
//               slot 1, item by item): the store issuer grants it to a slot, the slot's
//               epilogue fills it, the issuer TMA-stores it and grants it to the other.
//   warps 4-7   softmax + epilogue of Q0;  warps 8-11  softmax + epilogue of Q1.
//
// Shared memory: [K/V ring: NST tiles][Q0][Q1][O staging][barriers].  One Q buffer per
// slot and a single staging buffer leave room for a deeper ring (4 stages at D = 128):
// the ring's depth is what hides the latency of the K/V loads.
#pragma once

#include "attn_fwd_kernel.cuh"
#include "softmax_tile.cuh"

namespace gbattn {
template <int D>
struct PPCfg {
  static constexpr int NCH = D / 64;
  static constexpr int CHUNK = 128 * 128;            // bytes of a 128-row x 64-col fp16 box
  static constexpr int TILE = NCH * CHUNK;           // one 128 x D tile
  static constexpr int TILE_BUDGET = 224 * 1024;
  static constexpr int NQBUF = 2;                    // Q buffers: one per slot
  static constexpr int NOBUF = 1;                    // O staging buffer, shared by the slots
  static constexpr int NST_FIT = (TILE_BUDGET - (NQBUF + NOBUF) * TILE) / TILE;
  static constexpr int NST = NST_FIT > 12 ? 12 : NST_FIT;
  // barrier indices (per slot a: index + a).  GRANT[a] hands the staging buffer to slot
  // a's epilogue, EPI[a] hands the filled buffer back; each completes once per item of the
  // slot, in order, so a parity wait on either can never be two phases behind.
  static constexpr int B_QFULL = 0, B_QEMPTY = 2, B_FULL = 4, B_EMPTY = 4 + NST;
  static constexpr int B_SFULL = 4 + 2 * NST, B_PFULL = B_SFULL + 2, B_OFINAL = B_PFULL + 2;
  static constexpr int B_OFREE = B_OFINAL + 2, B_GRANT = B_OFREE + 2, B_EPI = B_GRANT + 2;
  static constexpr int B_DRAIN = B_EPI + 2;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int TILE_BYTES = NST * TILE + (NQBUF + NOBUF) * TILE;
  static constexpr int SMEM_BYTES = 1024 + TILE_BYTES + 8 * NBAR + 16;
  static constexpr int O_COL = 256;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_QK = idesc_f16_f32(128, 128, 0, 0);
  static constexpr uint32_t IDESC_PV = idesc_f16_f32(128, D, 0, 1);
  static constexpr int kLaunchRegs = 168;  // 65536 / 384 rounded down to a multiple of 8
  static constexpr int kRegsLow = 104, kRegsHigh = 192;
  static_assert(NST >= 2, "ring too shallow");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(O_COL + 2 * D <= TMEM_COLS, "tensor memory budget");
};

struct PPItem {
  int bh, qb, n0, n1;  // key tiles needed by Q0 and Q1 (n1 >= n0 >= 1)
};

template <bool CAUSAL>
__device__ __forceinline__ PPItem pp_decode(int r, const FwdParams &p) {
  PPItem it;
  const int grp = r / p.BH;
  it.bh = r - grp * p.BH;
  it.qb = CAUSAL ? (p.nQB - 1 - grp) : grp;
  if (CAUSAL) {
    it.n0 = 2 * it.qb + 1;
    it.n1 = min(2 * it.qb + 2, p.nQ);
  } else {
    it.n0 = it.n1 = p.nQ;
  }
  return it;
}

template <int D>
__device__ __forceinline__ uint32_t pp_q_tile(uint32_t q_s, int slot) {
  return q_s + static_cast<uint32_t>(slot) * PPCfg<D>::TILE;
}

// The MMA issuer: one thread issues the tensor-core work of both slots, so the operations
// reach the tensor core in program order (MMAs issued by two threads are interleaved by
// the hardware, which makes both slots' S tiles complete together and both softmax
// warpgroups run at once while the tensor core idles).  Within an item the order is
//     QK0_0, QK1_0, then for each key tile j:  PV0_j, QK0_{j+1}, PV1_j, QK1_{j+1}
// so softmax warpgroup 0 works on S0 while the tensor core runs PV1 and QK1, and the
// other way round.  The next item's QK0_0 cannot be issued right after the slot's last PV
// (its Q tile is loaded only once the slot's last QK released the buffer): it is issued
// from inside the issuer's later waits as soon as its Q and K tiles have landed, and at
// the latest before the next item's QK1_0, so it never holds back slot 1's work.
// Ring positions follow the producer's load order: item by item, K_0, V_0, K_1, V_1, ...
// for the n1 key tiles of the item.
template <int D, bool CAUSAL>
struct PPIssuer {
  using C = PPCfg<D>;
  const FwdParams *p;
  uint32_t ring_s, q_s, bar_s, tmem;
  volatile uint32_t *abort_flag;
  uint32_t base = 0;                // ring position of K_0 of the current item
  uint32_t n_pv0 = 0, n_pv1 = 0;    // PVs per slot so far (phases of the P barriers)
  // The last ring position whose FULL phase this thread has seen complete: slot 1's QK and
  // PV of a key tile follow slot 0's, and do not probe the same stage again.
  uint32_t seen_full = ~0u, seen_v = ~0u;
  // The next item's slot-0 QK, while it waits for its Q and K tiles.
  bool side_pending = false, side_last = false;
  int side_il = 0;
  uint32_t side_base = 0;

  __device__ uint32_t bar(int i) const { return bar_s + 8u * static_cast<uint32_t>(i); }
  // A parity test is unambiguous only while the barrier is at most one phase behind: the
  // K_0 stage's previous use (ring position side_base - NST) must have completed.  The
  // issue order guarantees that for the kernel's own items (n1 - n0 <= 1: that position
  // is K_{n1-2} of the current item, already consumed by QK1_{n1-2}); items whose slot 1
  // needs three or more key tiles beyond slot 0's would break it (a host-side model of the
  // issue order checks both).
  __device__ bool side_ready() const {
    return mbar_test(bar(C::B_QFULL + 0), side_il & 1) &&
           mbar_test(bar(C::B_FULL + side_base % C::NST), (side_base / C::NST) & 1u);
  }
  // S_slot = Q_slot K_j^T for the K tile at ring position pos, then release the stage and
  // signal the softmax; after the slot's last key tile of the item (`last`) the Q buffer
  // is released too.  Its inputs must have landed.
  __device__ void qk_issue(int slot, uint32_t pos, bool last) {
    const SDesc a = sdesc_split(sdesc_sw128(pp_q_tile<D>(q_s, slot), 16, 1024));
    const SDesc b = sdesc_split(sdesc_sw128(ring_s + (pos % C::NST) * C::TILE, 16, 1024));
    const uint32_t d_tmem = tmem + static_cast<uint32_t>(slot) * 128u;
#pragma unroll
    for (int c = 0; c < C::NCH; ++c)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_ss_off(d_tmem, a, c * C::CHUNK + kk * 32, b, c * C::CHUNK + kk * 32, C::IDESC_QK,
                    (c | kk) != 0 ? 1u : 0u);
    umma_commit(bar(C::B_SFULL + slot));
    // Slot 1's QK of a K tile comes after slot 0's (or slot 0 does not use it): its commit
    // covers both and frees the stage.
    if (slot == 1) umma_commit(bar(C::B_EMPTY + pos % C::NST));
    if (last) umma_commit(bar(C::B_QEMPTY + slot));
  }
  // Wait for every phase of ws.  While the next item's slot-0 QK is pending, the wait
  // polls (suspending ~0.1 us at a time) and issues that QK as soon as its inputs are in.
  __device__ bool wait_all(const WaitSet &ws) {
    if (side_pending) {
      const long long t0 = clock64();
      uint32_t b, ph;
      while (ws.first_pending(b, ph)) {
        if (side_ready()) {
          tc_fence_after();
          qk_issue(0, side_base, side_last);
          seen_full = side_base;
          side_pending = false;
          if (!ws.wait(abort_flag, p->status, kDevTimeoutMma, p->wait_limit)) return false;
          break;
        }
        if (mbar_try_for(b, ph, 100u)) continue;
        if (*abort_flag) return false;
        if (clock64() - t0 > p->wait_limit) {
          atomicCAS(p->status, 0u, kDevTimeoutMma);
          *abort_flag = 1u;
          return false;
        }
      }
    } else if (!ws.wait(abort_flag, p->status, kDevTimeoutMma, p->wait_limit)) {
      return false;
    }
    tc_fence_after();
    return true;
  }
  // QK of key tile j of item il (ring position of its K_0: item_base) for `slot`.
  __device__ bool qk(int slot, int j, int il, uint32_t item_base, bool last) {
    const uint32_t pos = item_base + 2u * static_cast<uint32_t>(j);
    WaitSet ws;
    if (j == 0) ws.add(bar(C::B_QFULL + slot), il & 1);
    if (pos != seen_full) ws.add(bar(C::B_FULL + pos % C::NST), (pos / C::NST) & 1u);
    if (ws.n > 0 && !wait_all(ws)) return false;
    seen_full = pos;
    qk_issue(slot, pos, last);
    return true;
  }
  // O_slot (+)= P_slot V_j, then release V_j's stage (and signal the epilogue after the
  // slot's last tile of the item).
  __device__ bool pv(int slot, int j, int il, int n_slot) {
    const uint32_t pos = base + 2u * static_cast<uint32_t>(j) + 1u;
    const uint32_t np = slot == 0 ? n_pv0 : n_pv1;
    WaitSet ws;
    ws.add(bar(C::B_PFULL + slot), np & 1u);
    if (j == 0 && il > 0) ws.add(bar(C::B_OFREE + slot), (il - 1) & 1);
    const bool v_seen = slot == 1 && pos == seen_v;
    if (!v_seen) ws.add(bar(C::B_FULL + pos % C::NST), (pos / C::NST) & 1u);
    if (!wait_all(ws)) return false;
    seen_v = pos;
    const SDesc b = sdesc_split(sdesc_sw128(ring_s + (pos % C::NST) * C::TILE, C::CHUNK, 1024));
    const uint32_t o_tmem = tmem + C::O_COL + static_cast<uint32_t>(slot) * D;
    const uint32_t p_tmem = tmem + static_cast<uint32_t>(slot) * 128u;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      umma_ts_off(o_tmem, p_tmem + kk * 8u, b, kk * 2048, C::IDESC_PV, (j == 0 && kk == 0) ? 0u : 1u);
    if (slot == 1) umma_commit(bar(C::B_EMPTY + pos % C::NST));  // the V tile's last reader
    if (j == n_slot - 1) umma_commit(bar(C::B_OFINAL + slot));
    if (slot == 0)
      ++n_pv0;
    else
      ++n_pv1;
    return true;
  }
  __device__ void run(const SchedTable *tbl) {
    Sched sc(blockIdx.x, gridDim.x, p->n_items, tbl);
    int r;
    if (!sc.next(r)) return;
    PPItem cur = pp_decode<CAUSAL>(r, *p);
    if (!qk(0, 0, 0, 0, cur.n0 == 1) || !qk(1, 0, 0, 0, cur.n1 == 1)) return;
    for (int il = 0;; ++il) {
      Sched peek = sc;
      int rn;
      const bool has_next = peek.next(rn);
      const PPItem nxt = has_next ? pp_decode<CAUSAL>(rn, *p) : cur;
      const uint32_t next_base = base + 2u * static_cast<uint32_t>(cur.n1);
      for (int j = 0; j < cur.n1; ++j) {
        if (j < cur.n0) {
          if (!pv(0, j, il, cur.n0)) return;
          if (j + 1 < cur.n0) {
            if (!qk(0, j + 1, il, base, j + 2 == cur.n0)) return;
          } else if (has_next) {
            side_pending = true;
            side_il = il + 1;
            side_base = next_base;
            side_last = nxt.n0 == 1;
          }
        }
        if (!pv(1, j, il, cur.n1)) return;
        if (j + 1 < cur.n1 && !qk(1, j + 1, il, base, j + 2 == cur.n1)) return;
      }
      if (!has_next) return;
      if (side_pending) {
        side_pending = false;
        if (!qk(0, 0, il + 1, next_base, nxt.n0 == 1)) return;
      }
      if (!qk(1, 0, il + 1, next_base, nxt.n1 == 1)) return;
      sc = peek;
      cur = nxt;
      base = next_base;
    }
  }
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_pp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       const FwdParams p, const __grid_constant__ SchedTable tbl) {
  using C = PPCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t ring_s = base;                     // NST x TILE (first: see attn_fwd_kernel.cuh)
  const uint32_t q_s = ring_s + C::NST * C::TILE;   // Q[slot]
  const uint32_t o_s = q_s + C::NQBUF * C::TILE;    // O staging
  const uint32_t bar_s = o_s + C::NOBUF * C::TILE;  // NBAR x 8
  uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + (bar_s - base) + 8 * C::NBAR);
  volatile uint32_t *const abort_flag = tmem_slot + 1;
  auto BAR = [&](int i) -> uint32_t { return bar_s + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long LIM = p.wait_limit;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(C::B_QFULL + i), 1);
      mbar_init(BAR(C::B_QEMPTY + i), 1);
      mbar_init(BAR(C::B_GRANT + i), 1);
      mbar_init(BAR(C::B_EPI + i), 128);
      mbar_init(BAR(C::B_SFULL + i), 1);
      mbar_init(BAR(C::B_PFULL + i), 128);
      mbar_init(BAR(C::B_OFINAL + i), 1);
      mbar_init(BAR(C::B_OFREE + i), 128);
    }
    mbar_init(BAR(C::B_DRAIN), 1);
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(BAR(C::B_FULL + i), 1);
      mbar_init(BAR(C::B_EMPTY + i), 1);  // released by slot 1's use, the last
    }
    *abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
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
  // This CTA's first schedule entry, read while the previous kernel may still be running
  // (the kernel parameters never depend on it), so that the loaders' first reads of the
  // table after the wait below hit the constant cache.
  if (warp == 2 && lane == 0 && tbl.n > 0) {
    const int s0 = tbl.start[blockIdx.x];
    if (s0 < tbl.start[blockIdx.x + 1]) {
      const int i0 = tbl.items[s0];
      asm volatile("" ::"r"(i0));
    }
  }
  // The prologue above touches no global memory: the next kernel may launch now, and this
  // one waits here for the previous kernel's writes (inputs may be its outputs).
  grid_launch_dependents();
  grid_wait_prior();

  // Register split: the launch gives every thread kLaunchRegs; the warpgroup of the four
  // single-thread roles (warps 0-3) gives up registers that the two softmax warpgroups
  // take: 128 * kRegsLow + 256 * kRegsHigh <= 384 * kLaunchRegs.
  static_assert(128 * PPCfg<D>::kRegsLow + 256 * PPCfg<D>::kRegsHigh <= 384 * PPCfg<D>::kLaunchRegs,
                "register split exceeds the launch allocation");
  if (warp < 4) {
    setmaxnreg_to<PPCfg<D>::kLaunchRegs, PPCfg<D>::kRegsLow>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- K/V producer
      const uint64_t pol_kv = policy_evict_last();
      Sched sc(blockIdx.x, gridDim.x, p.n_items, &tbl);
      uint32_t it = 0;
      int r;
      bool ok = true;
      while (ok && sc.next(r)) {
        const PPItem item = pp_decode<CAUSAL>(r, p);
        for (int j = 0; j < item.n1 && ok; ++j)
          for (int kv = 0; kv < 2 && ok; ++kv, ++it) {
            const uint32_t s = it % C::NST, ph = (it / C::NST) & 1u;
            if (!(ok = wait_bounded(BAR(C::B_EMPTY + s), ph ^ 1u, abort_flag, p.status, kDevTimeoutLoad, LIM)))
              break;
            mbar_arrive_expect_tx(BAR(C::B_FULL + s), C::TILE);
            const CUtensorMap *tm = kv == 0 ? &tm_k : &tm_v;
#pragma unroll
            for (int c = 0; c < C::NCH; ++c)
              tma_load_3d_hint(ring_s + s * C::TILE + c * C::CHUNK, tm, c * 64, j * 128, item.bh, BAR(C::B_FULL + s),
                               pol_kv);
          }
      }
      // Drain: every load issued must have landed before the CTA may exit.
      const uint32_t first = it > static_cast<uint32_t>(C::NST) ? it - C::NST : 0u;
      for (uint32_t i = first; i < it; ++i) wait_drain(BAR(C::B_FULL + (i % C::NST)), (i / C::NST) & 1u, LIM);
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      PPIssuer<D, CAUSAL> is;
      is.p = &p;
      is.ring_s = ring_s;
      is.q_s = q_s;
      is.bar_s = bar_s;
      is.tmem = tmem;
      is.abort_flag = abort_flag;
      is.run(&tbl);
      // Drain: all MMAs issued by this thread complete before tensor memory is freed.
      umma_commit(BAR(C::B_DRAIN));
      wait_drain(BAR(C::B_DRAIN), 0, LIM);
    } else if (warp == 3 && lane == 0) {
      // ---------------------------------------------------------- Q loads and O stores
      const uint64_t pol_q = policy_evict_first();
      Sched sc(blockIdx.x, gridDim.x, p.n_items, &tbl);
      int r, il = 0;
      int nq[2] = {0, 0};  // Q loads issued per buffer
      bool ok = true;
      // Slot a's Q tile of the ql-th item, once the slot's last QK of item ql-1 released
      // the buffer.
      auto load_q = [&](int a, int ql, const PPItem &item) -> bool {
        if (!wait_bounded(BAR(C::B_QEMPTY + a), (ql & 1) ^ 1u, abort_flag, p.status, kDevTimeoutLoad, LIM))
          return false;
        mbar_arrive_expect_tx(BAR(C::B_QFULL + a), C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d_hint(pp_q_tile<D>(q_s, a) + c * C::CHUNK, &tm_q, c * 64, item.qb * 256 + a * 128, item.bh,
                           BAR(C::B_QFULL + a), pol_q);
        ++nq[a];
        return true;
      };
      // Slot a's O tile of the ol-th item, once its epilogue staged it; then the staging
      // buffer goes to the other slot.
      auto store_o = [&](int a, int ol, const PPItem &item) -> bool {
        if (!wait_bounded(BAR(C::B_EPI + a), ol & 1, abort_flag, p.status, kDevTimeoutEpilogue, LIM)) return false;
        const int qrow0 = item.qb * 256 + a * 128;
        if (qrow0 < p.L) {
          for (int c = 0; c < C::NCH; ++c) tma_store_3d(&tm_o, o_s + c * C::CHUNK, c * 64, qrow0, item.bh);
          bulk_commit();
          bulk_wait_read0();
        }
        mbar_arrive(BAR(C::B_GRANT + (a ^ 1)));
        return true;
      };
      mbar_arrive(BAR(C::B_GRANT + 0));  // slot 0's first epilogue has the buffer
      if (sc.next(r)) {
        PPItem cur = pp_decode<CAUSAL>(r, p);
        ok = load_q(0, 0, cur) && load_q(1, 0, cur);
        while (ok) {
          Sched peek = sc;
          int rn;
          const bool has_next = peek.next(rn);
          const PPItem nxt = has_next ? pp_decode<CAUSAL>(rn, p) : cur;
          // The next item's Q tiles first (they gate its first QKs), then this item's O.
          if (has_next && !(ok = load_q(0, il + 1, nxt) && load_q(1, il + 1, nxt))) break;
          if (!(ok = store_o(0, il, cur) && store_o(1, il, cur))) break;
          if (!has_next) break;
          sc = peek;
          cur = nxt;
          ++il;
        }
      }
      bulk_wait0();
      // Drain: the last Q load into each buffer must have landed (earlier ones were read).
      for (int a = 0; a < 2; ++a)
        if (nq[a] > 0) wait_drain(BAR(C::B_QFULL + a), (nq[a] - 1) & 1, LIM);
    }
    __syncwarp();
  } else {
    setmaxnreg_to<PPCfg<D>::kLaunchRegs, PPCfg<D>::kRegsHigh>();
    // ================================================= softmax + epilogue of one Q tile
    const int slot = (warp - 4) >> 2;  // warps 4-7: Q0, warps 8-11: Q1
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + lane_base + slot * 128u;
    const uint32_t o_tmem = tmem + lane_base + C::O_COL + slot * D;
    const float c2 = p.c2;
    Sched sc(blockIdx.x, gridDim.x, p.n_items, &tbl);
    uint32_t g = 0;  // S tiles of this slot so far
    int il = 0, r;
    bool ok = true;
    auto wait_warp = [&](uint32_t b, uint32_t ph) -> bool {
      const bool w = wait_bounded(b, ph, abort_flag, p.status, kDevTimeoutSoftmax, LIM);
      return __all_sync(0xffffffffu, w);
    };
    while (ok && sc.next(r)) {
      const PPItem item = pp_decode<CAUSAL>(r, p);
      const int n = slot == 0 ? item.n0 : item.n1;
      const int qrow0 = item.qb * 256 + slot * 128;  // first query row of this tile
      const int diag = 2 * item.qb + slot;           // causal: the key tile holding the diagonal
      float m_used = 0.f, l = 0.f;
      for (int j = 0; j < n; ++j, ++g) {
        if (!(ok = wait_warp(BAR(C::B_SFULL + slot), g & 1u))) break;
        tc_fence_after();
        // Keys past the diagonal (causal) or past L (ragged last tile) are masked.  PV of
        // the previous tile is complete here: it precedes this QK in the issue order.
        const int lim = CAUSAL ? (j == diag ? row + 1 : 128) : min(128, p.L - j * 128);
        softmax_tile<D>(s_tmem, o_tmem, lim, c2, j == 0, m_used, l);
        tc_fence_before();
        mbar_arrive(BAR(C::B_PFULL + slot));
      }
      if (!ok) break;
      // --------------------------------------------------------------- epilogue
      // O / l as fp16 into the staging buffer once it is granted to this slot (swizzled like
      // a TMA box), then the store issuer writes it out; LSE goes straight to global memory.
      if (!(ok = wait_warp(BAR(C::B_OFINAL + slot), il & 1))) break;
      if (!(ok = wait_warp(BAR(C::B_GRANT + slot), il & 1))) break;  // the staging buffer is ours
      tc_fence_after();
      stage_o_row<D>(o_tmem, o_s, row, 1.0f / l);
      tc_fence_before();
      mbar_arrive(BAR(C::B_OFREE + slot));  // O fully read: the next item's first PV may overwrite it
      const int grow = qrow0 + row;
      if (grow < p.L)
        p.lse[static_cast<long long>(item.bh) * p.L + grow] = (m_used + __log2f(l)) * 0.69314718055994531f;
      fence_proxy_async_smem();
      mbar_arrive(BAR(C::B_EPI + slot));
      ++il;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_pp_variant(const FwdLaunch &a) {
  using C = PPCfg<D>;
  auto *kern = attn_fwd_pp_kernel<D, CAUSAL>;
  static int configured_mask = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 31 || !(configured_mask & (1 << dev))) {
    // The warpgroup register split assumes the kernel is launched with kLaunchRegs
    // registers per thread; with fewer, setmaxnreg.inc could never be satisfied.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs < C::kLaunchRegs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 31) configured_mask |= (1 << dev);
  }
  return launch_pdl(kern, a.grid, 384, C::SMEM_BYTES, a.stream, a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p, *a.tbl);
}

template <int D>
cudaError_t launch_fwd_pp_d(const FwdLaunch &a) {
  return a.causal ? launch_fwd_pp_variant<D, true>(a) : launch_fwd_pp_variant<D, false>(a);
}

cudaError_t launch_fwd_pp_64(const FwdLaunch &a);
cudaError_t launch_fwd_pp_128(const FwdLaunch &a);

}  // namespace gbattn
