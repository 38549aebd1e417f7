// attn_fwd_kernel.cuh -- fused, persistent, warp-specialised SDPA forward for sm_103a.
//
// What it computes ("An Optimal Mapper Meets a Real GPU", "Ground rules" / "Experiment
// one"; STAGE_D.md of nvfp4-megamoe-kernel, sections 2, 3, 4 and 6):
//   O = softmax(scale * Q K^T + causal mask) V  and  LSE = log-sum-exp of each row,
// in ONE kernel: scores and weights live in tensor memory only, never in DRAM (the
// single-kernel fusion the first page finds missing from the mapper's search space).
//
// Work item = (batch*head bh, 128-row query tile qt, value-column half): head_dim 512
// splits the 512 output columns into two 256-wide items (tensor memory holds S twice
// plus a 256-column O).  Items are ordered longest first (causal: most key tiles first)
// and dealt to a persistent grid in a snake order; every CTA walks its own list, so no
// scheduler state lives in global memory.
//
// Key-range split (SPLITKV, on clusters of two CTAs): a long query tile's key tiles are
// shared by the two CTAs of a cluster, rank 0 taking the first ceil(n / 2) and rank 1 the
// rest; each CTA runs its part like an item, then rank 1 hands its partial O (normalised,
// fp16) and each row's (m, l) to rank 0 through shared memory, and rank 0 merges the two
// with the log-sum-exp weights -- exact because the two key ranges are disjoint (STAGE_D.md,
// section 2, "Merge").  Such split tiles come first in both CTAs' lists, in the same order.
//
// Head_dim split (DSPLIT, on clusters of two CTAs; an option at head_dim 512): each CTA
// holds half of Q and of every K tile, the two exchange their partial S tiles, and each
// produces half of the output columns.
//
// Warp roles (256 threads):
//   warp 0      TMA producer: Q tile per item, then K / V tiles through an mbarrier ring in
//               exactly the order the MMA issuer consumes them.
//   warp 1      TMEM owner + MMA issuer (one thread): S = Q K^T into one of two S buffers
//               (head_dim summed over every 64-wide slice before the softmax sees S),
//               then O += P V.  QK of the next key tile is issued before PV of the current
//               one, so the tensor core works while the softmax runs.
//   warps 4..7  softmax + epilogue, one query row per thread: row max, exp2, row sum,
//               lazy O rescale (only when the running max grows by more than 2^8), P as
//               fp16 back into tensor memory (aliasing S) or into shared memory; then
//               O / l -> fp16 -> swizzled staging tile -> TMA store, and LSE.
//   warp 2      key-range split, rank 1: copies each split tile's partial to rank 0 and
//               gives the staging Q buffer back once rank 0 has it; idle otherwise.
//   warp 3      idle.
//
// Every wait is bounded (about two seconds of SM clock); a wait that runs out records a
// status code, raises a CTA-wide abort flag, and the CTA drains its in-flight copies and
// MMAs, frees tensor memory and exits.
#pragma once

#include <cuda_runtime.h>

#include "ptx.cuh"
#include "softmax_tile.cuh"

namespace gbattn {

constexpr unsigned kDevTimeoutLoad = 1;
constexpr unsigned kDevTimeoutMma = 2;
constexpr unsigned kDevTimeoutSoftmax = 3;
constexpr unsigned kDevTimeoutEpilogue = 4;
constexpr unsigned kDevTimeoutProbe = 5;

struct FwdParams {
  float *lse;              // [BH, L] fp32
  unsigned *status;        // device status word (first error code wins)
  long long wait_limit;    // SM clock cycles a single wait may take before it gives up
  int BH, L, nQ, n_items;  // nQ = ceil(L / 128)
  int nQB;                 // ceil(L / 256): query blocks of the two-tile kernel
  float c2;                // scale * log2(e)
};

template <int D, bool P_TMEM, bool DSPLIT = false, bool SPLITKV = false>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int DVS = D > 256 ? D / 256 : 1;  // value-column splits per (bh, qt)
  static constexpr int DV = D / DVS;                 // O columns owned by one item
  static constexpr int NCH = D / 64;                 // 64-column chunks of a Q / K tile
  // head_dim split over a CTA pair: each CTA holds half of Q and of every K tile
  static constexpr int QCH = DSPLIT ? NCH / 2 : NCH;  // chunks of Q (and of each K tile) held
  static constexpr int NCHV = DV / 64;               // 64-column chunks of an item's V tile
  static constexpr int SC = D == 64 ? 1 : 2;         // chunks per ring stage
  static constexpr int KST = QCH / SC;               // ring stages per K tile (this CTA's chunks)
  static constexpr int VST = NCHV / SC;              // ring stages per V tile
  static constexpr int NQB = D <= 128 ? 2 : 1;       // Q buffers (also the O staging tiles)
  static constexpr bool LOOKAHEAD = NQB >= 2;        // next item's QKs before its last PVs
  // S buffers in tensor memory; the issuer runs QK NSB - 1 key tiles ahead of PV.  Three
  // would fit for O tiles of at most 128 columns, but measured slower on GB300: the QK two
  // tiles ahead needs its K tile one ring stage earlier, and with five stages of 32 KB that
  // costs more load latency than the earlier S saves.  (The P-in-shared-memory variant
  // would also need a third P buffer.)
  static constexpr int NSB = 2;
  static constexpr int CHUNK = 128 * 128;            // bytes of a 128-row x 64-col fp16 box
  static constexpr int STAGE = SC * CHUNK;
  static constexpr int QBYTES = QCH * CHUNK;
  // head_dim split: the peer's partial S tile (128 x 128 fp32), 16-byte chunks of each
  // 512-byte row XOR-swizzled by row & 7
  static constexpr int RBYTES = DSPLIT ? 128 * 128 * 4 : 0;
  // Key-range split over a CTA pair (split items): rank 1 hands its partial O (fp16,
  // normalised by its own l) and each row's (m, l) to rank 0, which merges.  The receive
  // area: a buffer of its own for head_dim <= 128; at head_dim 512 the Q buffer's columns
  // 256-511 (free once the item's last QK is done; an item writes only 256 columns of O).
  static constexpr bool CLUSTER = DSPLIT || SPLITKV;
  static constexpr int XBYTES = SPLITKV && D <= 128 ? D * 128 * 2 : 0;  // receive buffer
  static constexpr int STBYTES = SPLITKV ? 128 * 8 : 0;                 // (m, l) per row
  static constexpr int NPB = P_TMEM ? 0 : 2;         // shared-memory P buffers
  static constexpr int PBYTES = 2 * CHUNK;           // 128 x 128 fp16
  static constexpr int TILE_BUDGET = 224 * 1024;
  static constexpr int NST_FIT = (TILE_BUDGET - NQB * QBYTES - NPB * PBYTES - RBYTES - XBYTES) / STAGE;
  static constexpr int NST = NST_FIT > 8 ? 8 : NST_FIT;
  // barrier indices
  static constexpr int B_QFULL = 0, B_QEMPTY = 2, B_FULL = 4, B_EMPTY = 4 + NST;
  // ODONE[g & 1] completes when the PV of key tile g (counted across items) is done.
  static constexpr int B_SFULL = 4 + 2 * NST, B_PFULL = B_SFULL + NSB, B_ODONE = B_PFULL + NSB;
  static constexpr int B_OFREE = B_ODONE + 2, B_EPI = B_OFREE + 1, B_DRAIN = B_EPI + 1;
  // head_dim split: RECV completes when the peer's partial S is in this CTA's buffer,
  // RFREE when the peer has read this CTA's partial out of its own buffer
  static constexpr int B_RECV = B_DRAIN + 1, B_RFREE = B_RECV + 1;
  // key-range split: READY (on rank 1) completes when rank 0's receive area is free for
  // the split item, XRECV (on rank 0) when rank 1's partial has landed in it, XACK (on
  // rank 1) when rank 0 has it (rank 1's staging is free again), XSTAGED (on rank 1) when
  // its 128 softmax threads have staged their rows
  static constexpr int B_READY = B_RFREE + 1, B_XRECV = B_READY + 1, B_XACK = B_XRECV + 1;
  static constexpr int B_XSTAGED = B_XACK + 1;
  static constexpr int NBAR = B_XSTAGED + 1;
  static constexpr int TILE_BYTES = NQB * QBYTES + NPB * PBYTES + RBYTES + XBYTES + STBYTES + NST * STAGE;
  static constexpr int SMEM_BYTES = 1024 /*alignment slack*/ + TILE_BYTES + 8 * NBAR + 16;
  // tensor memory columns: S buffer b at [128 b, 128 b + 128), O after the S buffers
  static constexpr int O_COL = 128 * NSB;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_QK = idesc_f16_f32(128, 128, 0, 0);
  static constexpr uint32_t IDESC_PV = idesc_f16_f32(128, SC * 64, 0, 1);
  static_assert(NST >= 2, "ring too shallow");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(O_COL + DV <= TMEM_COLS, "tensor memory budget");
  static_assert(QCH % SC == 0 && NCHV % SC == 0, "stage split");
  static_assert(!DSPLIT || (D == 512 && P_TMEM), "head_dim split: D = 512, P in tensor memory");
  static_assert(!SPLITKV || (P_TMEM && !DSPLIT && D != 256), "key-range split: D = 64, 128, 512, P in TMEM");
  static_assert(!SPLITKV || D <= 128 || NCH >= 2 * NCHV, "key-range split at D = 512: Q columns hold the partial");
};

// Static schedule.  With a table (n > 0), CTA c processes items[start[c] .. start[c+1]):
// the host fills it by longest-processing-time-first assignment of item costs (work units
// plus a per-item overhead).  It travels in the kernel parameters, so no device memory is
// involved.  Without a table (problems with more items than it holds), a snake order:
// pass p hands items [p*G, p*G+G) to CTAs 0..G-1, reversed on odd passes.
constexpr int kSchedMaxCtas = 256;
constexpr int kSchedMaxItems = 3072;
struct SchedTable {
  int n;  // items in the table; 0 = snake order
  uint16_t start[kSchedMaxCtas + 1];
  uint16_t items[kSchedMaxItems];
};

struct Sched {
  int cta, G, NI, pass, npass;
  const SchedTable *tbl;
  __device__ Sched(int c, int g, int ni, const SchedTable *t)
      : cta(c), G(g), NI(ni), pass(0), npass((ni + g - 1) / g), tbl(t) {
    if (tbl->n > 0) {
      pass = tbl->start[c];
      npass = tbl->start[c + 1];
    }
  }
  __device__ bool next(int &item) {
    if (tbl->n > 0) {
      if (pass >= npass) return false;
      item = tbl->items[pass++];
      return true;
    }
    while (pass < npass) {
      const int p = pass++;
      const int r = p * G + ((p & 1) ? (G - 1 - cta) : cta);
      if (r < NI) {
        item = r;
        return true;
      }
    }
    return false;
  }
};

template <int DVS, bool CAUSAL>
__device__ __forceinline__ void decode_item(int r, const FwdParams &p, int &bh, int &qt, int &half,
                                            int &ntiles) {
  const int per = p.BH * DVS;
  const int grp = r / per, rem = r - grp * per;
  qt = CAUSAL ? (p.nQ - 1 - grp) : grp;
  bh = rem / DVS;
  half = rem - bh * DVS;
  ntiles = CAUSAL ? qt + 1 : p.nQ;
}

// Work item in a launch with key-range splits: values >= n_items name a split item,
// the query tile of item value - n_items (decoded as above) whose key tiles [0, n) are
// shared by the two CTAs of a cluster: rank 0 takes [0, ceil(n / 2)), rank 1 the rest.
template <int DVS, bool CAUSAL, bool SPLITKV>
__device__ __forceinline__ bool decode_work(int r, const FwdParams &p, uint32_t rank, int &bh, int &qt, int &half,
                                            int &t0, int &t1) {
  const bool split = SPLITKV && r >= p.n_items;
  int n;
  decode_item<DVS, CAUSAL>(split ? r - p.n_items : r, p, bh, qt, half, n);
  t0 = 0;
  t1 = n;
  if (split) {
    const int n0 = (n + 1) / 2;
    if (rank == 0) t1 = n0;
    else t0 = n0;
  }
  return split;
}

// Bounded wait.  Gives up when the abort flag is raised or after `limit` cycles; in the
// latter case records `code` (first error wins) and raises the abort flag.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                             unsigned *status, unsigned code, long long limit) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      atomicCAS(status, 0u, code);
      *abort_flag = 1u;
      return false;
    }
  }
}
// Same, for a barrier that another CTA of the cluster arrives on (acquire at cluster
// scope, so that what it wrote into this CTA's shared memory before arriving is visible).
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                                     unsigned *status, unsigned code, long long limit) {
  if (mbar_try_acquire_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_acquire_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      atomicCAS(status, 0u, code);
      *abort_flag = 1u;
      return false;
    }
  }
}
// Wait for up to three barrier phases at once: first test them all back to back (their
// latencies overlap), and only fall back to bounded waits for those not yet complete.
struct WaitSet {
  uint32_t b0 = 0, p0 = 0, b1 = 0, p1 = 0, b2 = 0, p2 = 0;
  int n = 0;
  __device__ void add(uint32_t b, uint32_t ph) {
    if (n == 0) {
      b0 = b;
      p0 = ph;
    } else if (n == 1) {
      b1 = b;
      p1 = ph;
    } else {
      b2 = b;
      p2 = ph;
    }
    ++n;
  }
  // Non-blocking: the first phase not yet complete (false when all are).
  __device__ bool first_pending(uint32_t &b, uint32_t &ph) const {
    if (!mbar_test(b0, p0)) {
      b = b0;
      ph = p0;
      return true;
    }
    if (n > 1 && !mbar_test(b1, p1)) {
      b = b1;
      ph = p1;
      return true;
    }
    if (n > 2 && !mbar_test(b2, p2)) {
      b = b2;
      ph = p2;
      return true;
    }
    return false;
  }
  // Non-blocking: are all phases complete?
  __device__ bool test() const {
    bool all = mbar_test(b0, p0);
    if (n > 1) all &= mbar_test(b1, p1);
    if (n > 2) all &= mbar_test(b2, p2);
    return all;
  }
  __device__ bool wait(volatile uint32_t *abort_flag, unsigned *status, unsigned code, long long limit) const {
    bool all = mbar_test(b0, p0);
    if (n > 1) all &= mbar_test(b1, p1);
    if (n > 2) all &= mbar_test(b2, p2);
    if (all) return true;
    if (!wait_bounded(b0, p0, abort_flag, status, code, limit)) return false;
    if (n > 1 && !wait_bounded(b1, p1, abort_flag, status, code, limit)) return false;
    if (n > 2 && !wait_bounded(b2, p2, abort_flag, status, code, limit)) return false;
    return true;
  }
};

// Same but ignoring the abort flag: used only while draining in-flight work at exit.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// The order in which the single-tile kernel's MMA issuer consumes ring stages, walked
// identically by the producer (which loads in that order) and the issuer: per key tile g
// (counted across items) the QK, then -- once NSB - 1 PVs wait in the queue -- the oldest
// PV (its S buffer is the next QK's), then PV(g) joins the queue: QK runs NSB - 1 tiles
// ahead of PV.  Before the first QK of an item every PV of an item two back (one back
// without LOOKAHEAD) leaves the queue: that item's epilogue must be able to finish, since
// its Q buffer is its O staging tile and receives the Q of the item after next.
struct PendingPv {
  uint32_t g;
  int il, t, t0, bh, half;  // t0: the item's first key tile (its first PV starts a fresh O)
};
template <int NSB>
struct PvQueue {
  static constexpr int CAP = NSB > 1 ? NSB - 1 : 1;  // at most 2
  static_assert(CAP <= 2, "selects below index at most two entries");
  PendingPv e[CAP];
  int head = 0, size = 0;
  // Entries are picked by selects on constant indices, so the queue stays in registers.
  __device__ void push(const PendingPv &v) {
    int tail = head + size;
    if (tail >= CAP) tail -= CAP;
    if (tail == 0) e[0] = v;
    else e[CAP - 1] = v;
    ++size;
  }
  __device__ PendingPv pop() {
    const PendingPv v = head == 0 ? e[0] : e[CAP - 1];
    head = head + 1 == CAP ? 0 : head + 1;
    --size;
    return v;
  }
  __device__ const PendingPv &front() const { return head == 0 ? e[0] : e[CAP - 1]; }
};

template <int D, bool CAUSAL, bool P_TMEM, bool DSPLIT, bool SPLITKV = false>
__global__ void __launch_bounds__(256, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p, const __grid_constant__ SchedTable tbl) {
  using C = FwdCfg<D, P_TMEM, DSPLIT, SPLITKV>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  // The ring comes first: every tensor-core operand read that starts in a ring stage
  // stays inside this CTA's tiles even at its farthest stride.
  const uint32_t ring_s = base;                             // NST x STAGE
  const uint32_t q_s = ring_s + C::NST * C::STAGE;          // NQB x QBYTES
  const uint32_t p_s = q_s + C::NQB * C::QBYTES;            // NPB x PBYTES
  const uint32_t recv_s = p_s + C::NPB * C::PBYTES;         // RBYTES (head_dim split)
  const uint32_t x_s = recv_s + C::RBYTES;                  // XBYTES (key-range split, D <= 128)
  const uint32_t st_s = x_s + C::XBYTES;                    // STBYTES: rank 1's (m, l) per row
  const uint32_t bar_s = st_s + C::STBYTES;                 // NBAR x 8
  // key-range split: where rank 0 receives rank 1's partial O
  const uint32_t xrecv_s = D <= 128 ? x_s : q_s + C::NCHV * C::CHUNK;
  uint32_t *const tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + (bar_s - base) + 8 * C::NBAR);
  volatile uint32_t *const abort_flag = tmem_slot + 1;
  auto BAR = [&](int i) -> uint32_t { return bar_s + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // head_dim split: the two CTAs of a cluster share every work item; rank r holds Q / K
  // columns [r * D/2, (r + 1) * D/2) and computes the value columns of half r.
  const uint32_t rank = C::CLUSTER ? cluster_ctarank() : 0u;
  const int qc0 = DSPLIT ? static_cast<int>(rank) * C::QCH : 0;  // first 64-column chunk of Q / K held
  const int sched_id = DSPLIT ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int sched_n = DSPLIT ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    if (DSPLIT) {
      mbar_init(BAR(C::B_RECV), 128);   // the peer's 128 softmax threads
      mbar_init(BAR(C::B_RFREE), 128);
    }
    if (SPLITKV) {
      mbar_init(BAR(C::B_READY), 1);    // one thread of rank 0
      mbar_init(BAR(C::B_XRECV), 1);    // this CTA's expect_tx, plus the copied bytes
      mbar_init(BAR(C::B_XACK), 1);     // one thread of rank 0
      mbar_init(BAR(C::B_XSTAGED), 128);
    }
    for (int i = 0; i < C::NQB; ++i) {
      mbar_init(BAR(C::B_QFULL + i), 1);
      mbar_init(BAR(C::B_QEMPTY + i), 1);
    }
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(BAR(C::B_FULL + i), 1);
      mbar_init(BAR(C::B_EMPTY + i), 1);
    }
    for (int i = 0; i < C::NSB; ++i) {
      mbar_init(BAR(C::B_SFULL + i), 1);
      mbar_init(BAR(C::B_PFULL + i), 128);
    }
    mbar_init(BAR(C::B_ODONE), 1);
    mbar_init(BAR(C::B_ODONE + 1), 1);
    mbar_init(BAR(C::B_OFREE), 128);
    mbar_init(BAR(C::B_EPI), 128);
    mbar_init(BAR(C::B_DRAIN), 1);
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
  // Both CTAs of a pair have initialised their barriers before either arrives on the
  // other's (every thread reaches this, unconditionally).
  if constexpr (C::CLUSTER) cluster_sync_all();
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
  const long long LIM = p.wait_limit;

  if (warp == 0) {
    // =============================================================== TMA producer
    if (lane == 0) {
      Sched sc(sched_id, sched_n, p.n_items, &tbl);
      uint32_t it = 0;
      int il = 0, item;
      bool ok = true;
      const uint64_t pol_kv = policy_evict_last();
      auto load_stage = [&](const CUtensorMap *tm, int chunk0, int y, int z) -> bool {
        const uint32_t s = it % C::NST, ph = (it / C::NST) & 1u;
        if (!wait_bounded(BAR(C::B_EMPTY + s), ph ^ 1u, abort_flag, p.status, kDevTimeoutLoad, LIM))
          return false;
        mbar_arrive_expect_tx(BAR(C::B_FULL + s), C::STAGE);
#pragma unroll
        for (int j = 0; j < C::SC; ++j)
          tma_load_3d_hint(ring_s + s * C::STAGE + j * C::CHUNK, tm, (chunk0 + j) * 64, y, z,
                           BAR(C::B_FULL + s), pol_kv);
        ++it;
        return true;
      };
      auto load_v = [&](const PendingPv &v) -> bool {
        for (int vs = 0; vs < C::VST; ++vs)
          if (!load_stage(&tm_v, v.half * C::NCHV + vs * C::SC, v.t * C::BN, v.bh)) return false;
        return true;
      };
      PvQueue<C::NSB> pq;
      uint32_t g = 0;
      while (ok && sc.next(item)) {
        int bh, qt, half, t0, t1;
        decode_work<DSPLIT ? 1 : C::DVS, CAUSAL, SPLITKV>(item, p, rank, bh, qt, half, t0, t1);
        if (DSPLIT) half = static_cast<int>(rank);
        while (ok && pq.size > 0 && pq.front().il < il - (C::LOOKAHEAD ? 1 : 0)) ok = load_v(pq.pop());
        if (!ok) break;
        const int qb = il % C::NQB;
        const uint32_t qph = (il / C::NQB) & 1;
        if (!(ok = wait_bounded(BAR(C::B_QEMPTY + qb), qph ^ 1u, abort_flag, p.status, kDevTimeoutLoad, LIM)))
          break;
        mbar_arrive_expect_tx(BAR(C::B_QFULL + qb), C::QBYTES);
        for (int c = 0; c < C::QCH; ++c)
          tma_load_3d(q_s + qb * C::QBYTES + c * C::CHUNK, &tm_q, (qc0 + c) * 64, qt * C::BM, bh,
                      BAR(C::B_QFULL + qb));
        for (int t = t0; t < t1 && ok; ++t, ++g) {
          for (int ks = 0; ks < C::KST && ok; ++ks) ok = load_stage(&tm_k, qc0 + ks * C::SC, t * C::BN, bh);
          if (ok && pq.size == C::NSB - 1) ok = load_v(pq.pop());
          pq.push(PendingPv{g, il, t, t0, bh, half});
        }
        ++il;
      }
      while (ok && pq.size > 0) ok = load_v(pq.pop());
      // Drain: every load issued must have landed before the CTA may exit.
      const uint32_t first = it > static_cast<uint32_t>(C::NST) ? it - C::NST : 0u;
      for (uint32_t i = first; i < it; ++i)
        wait_drain(BAR(C::B_FULL + (i % C::NST)), (i / C::NST) & 1u, LIM);
      for (int i = (il > C::NQB ? il - C::NQB : 0); i < il; ++i)
        wait_drain(BAR(C::B_QFULL + (i % C::NQB)), (i / C::NQB) & 1, LIM);
    }
    __syncwarp();
  } else if (warp == 1) {
    // =============================================================== MMA issuer
    if (lane == 0) {
      Sched sc(sched_id, sched_n, p.n_items, &tbl);
      uint32_t it = 0, g = 0;
      int il = 0, item;
      bool ok = true;
      auto wait = [&](uint32_t bar, uint32_t ph) -> bool {
        return wait_bounded(bar, ph, abort_flag, p.status, kDevTimeoutMma, LIM);
      };
      auto issue_qk = [&](uint32_t gg, int qb) -> bool {
        const uint32_t sb = gg % C::NSB;
        const uint32_t d_tmem = tmem + sb * 128u;
        for (int ks = 0; ks < C::KST; ++ks) {
          const uint32_t s = it % C::NST;
          if (!wait(BAR(C::B_FULL + s), (it / C::NST) & 1u)) return false;
          tc_fence_after();
          const SDesc a = sdesc_split(sdesc_sw128(q_s + qb * C::QBYTES + ks * C::STAGE, 16, 1024));
          const SDesc b = sdesc_split(sdesc_sw128(ring_s + s * C::STAGE, 16, 1024));
#pragma unroll
          for (int j = 0; j < C::SC; ++j) {
            const int cidx = ks * C::SC + j;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ss_off(d_tmem, a, j * C::CHUNK + kk * 32, b, j * C::CHUNK + kk * 32, C::IDESC_QK,
                          (cidx | kk) != 0 ? 1u : 0u);
          }
          umma_commit(BAR(C::B_EMPTY + s));
          ++it;
        }
        umma_commit(BAR(C::B_SFULL + sb));
        return true;
      };
      auto issue_pv = [&](const PendingPv &v) -> bool {
        const uint32_t sb = v.g % C::NSB;
        const bool first = v.t == v.t0;
        // P, the first V stage and (on an item's first PV) the free O are tested together:
        // their barrier probes' latencies overlap.
        WaitSet ws;
        ws.add(BAR(C::B_PFULL + sb), (v.g / C::NSB) & 1u);
        ws.add(BAR(C::B_FULL + it % C::NST), (it / C::NST) & 1u);
        if (first && v.il > 0) ws.add(BAR(C::B_OFREE), (v.il - 1) & 1);
        if (!ws.wait(abort_flag, p.status, kDevTimeoutMma, LIM)) return false;
        tc_fence_after();
        for (int vs = 0; vs < C::VST; ++vs) {
          const uint32_t s = it % C::NST;
          if (vs > 0 && !wait(BAR(C::B_FULL + s), (it / C::NST) & 1u)) return false;
          tc_fence_after();
          const uint32_t o_tmem = tmem + C::O_COL + vs * C::SC * 64;
          const SDesc b = sdesc_split(sdesc_sw128(ring_s + s * C::STAGE, C::CHUNK, 1024));
          const SDesc a = sdesc_split(sdesc_sw128(p_s + (v.g & 1u) * C::PBYTES, 16, 1024));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t acc = (first && kk == 0) ? 0u : 1u;
            if constexpr (P_TMEM) {
              umma_ts_off(o_tmem, tmem + sb * 128u + kk * 8u, b, kk * 2048, C::IDESC_PV, acc);
            } else {
              umma_ss_off(o_tmem, a, (kk >> 2) * C::CHUNK + (kk & 3) * 32, b, kk * 2048, C::IDESC_PV, acc);
            }
          }
          umma_commit(BAR(C::B_EMPTY + s));
          ++it;
        }
        umma_commit(BAR(C::B_ODONE + (v.g & 1u)));
        return true;
      };
      PvQueue<C::NSB> pq;
      while (ok && sc.next(item)) {
        int bh, qt, half, t0, t1;
        decode_work<DSPLIT ? 1 : C::DVS, CAUSAL, SPLITKV>(item, p, rank, bh, qt, half, t0, t1);
        if (DSPLIT) half = static_cast<int>(rank);
        while (ok && pq.size > 0 && pq.front().il < il - (C::LOOKAHEAD ? 1 : 0)) ok = issue_pv(pq.pop());
        if (!ok) break;
        const int qb = il % C::NQB;
        if (!(ok = wait(BAR(C::B_QFULL + qb), (il / C::NQB) & 1))) break;
        tc_fence_after();
        for (int t = t0; t < t1 && ok; ++t, ++g) {
          ok = issue_qk(g, qb);
          if (ok && pq.size == C::NSB - 1) ok = issue_pv(pq.pop());
          pq.push(PendingPv{g, il, t, t0, bh, half});
        }
        ++il;
      }
      while (ok && pq.size > 0) ok = issue_pv(pq.pop());
      // Drain: all MMAs issued by this thread complete before tensor memory is freed.
      umma_commit(BAR(C::B_DRAIN));
      wait_drain(BAR(C::B_DRAIN), 0, LIM);
    }
    __syncwarp();
  } else if (SPLITKV && warp == 2) {
    // =============================================================== key-range split sender
    // Rank 1: per split item, once its softmax warps have staged the partial and rank 0's
    // receive area is free, copy the partial and the row statistics into rank 0 (one bulk
    // copy per 64-column chunk, completion on rank 0's XRECV), wait until rank 0 has them,
    // then give the item's Q buffer (its staging tile) back to the producer.
    if (lane == 0 && rank == 1) {
      Sched sc(sched_id, sched_n, p.n_items, &tbl);
      int il = 0, ks = 0, item;
      bool ok = true;
      const uint32_t peer_bar = mapa_shared(BAR(C::B_XRECV), 0u);
      while (ok && sc.next(item)) {
        int bh, qt, half, t0, t1;
        if (decode_work<C::DVS, CAUSAL, SPLITKV>(item, p, rank, bh, qt, half, t0, t1)) {
          const int qb = il % C::NQB;
          const uint32_t stage = q_s + qb * C::QBYTES;
          if (!(ok = wait_bounded(BAR(C::B_XSTAGED), ks & 1, abort_flag, p.status, kDevTimeoutEpilogue, LIM)))
            break;
          if (!(ok = wait_bounded_cluster(BAR(C::B_READY), ks & 1, abort_flag, p.status, kDevTimeoutEpilogue, LIM)))
            break;
          for (int j = 0; j < C::NCHV; ++j)
            bulk_s2c(mapa_shared(xrecv_s + j * C::CHUNK, 0u), stage + j * C::CHUNK, C::CHUNK, peer_bar);
          bulk_s2c(mapa_shared(st_s, 0u), st_s, C::STBYTES, peer_bar);
          if (!(ok = wait_bounded_cluster(BAR(C::B_XACK), ks & 1, abort_flag, p.status, kDevTimeoutEpilogue, LIM)))
            break;
          mbar_arrive(BAR(C::B_QEMPTY + qb));
          ++ks;
        }
        ++il;
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // =============================================================== softmax + epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // query row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.c2;
    Sched sc(sched_id, sched_n, p.n_items, &tbl);
    uint32_t g = 0;
    int il = 0, item;
    bool ok = true;
    // Store issuer (warp 4, lane 0) with two Q buffers: the Q buffer whose O store has not
    // yet been waited for (-1: none).  Its release waits until the next item's first
    // softmax tile is done, by when the store has read it, so the softmax never waits for
    // the store; the producer needs that buffer only for the item after next.
    int qempty_pending = -1;
    auto release_pending = [&]() {
      if (qempty_pending >= 0) {
        bulk_wait_read0();
        mbar_arrive(BAR(C::B_QEMPTY + qempty_pending));
        qempty_pending = -1;
      }
    };
    auto wait_warp = [&](uint32_t bar, uint32_t ph) -> bool {
      const bool r = wait_bounded(bar, ph, abort_flag, p.status, kDevTimeoutSoftmax, LIM);
      return __all_sync(0xffffffffu, r);
    };
    auto wait_warp_cluster = [&](uint32_t bar, uint32_t ph) -> bool {
      const bool r = wait_bounded_cluster(bar, ph, abort_flag, p.status, kDevTimeoutSoftmax, LIM);
      return __all_sync(0xffffffffu, r);
    };
    int ks = 0;  // split items so far (the phase of the key-range split barriers)
    int ne = 0;  // items whose O this CTA stores (the phase of EPI; rank 1 stores no split item)
    while (ok && sc.next(item)) {
      int bh, qt, half, t0, t1;
      const bool split = decode_work<DSPLIT ? 1 : C::DVS, CAUSAL, SPLITKV>(item, p, rank, bh, qt, half, t0, t1);
      if (DSPLIT) half = static_cast<int>(rank);
      float m_used = 0.f, l = 0.f;
      for (int t = t0; t < t1; ++t, ++g) {
        const uint32_t sb = g % C::NSB;
        if (!(ok = wait_warp(BAR(C::B_SFULL + sb), (g / C::NSB) & 1u))) break;
        tc_fence_after();
        if (SPLITKV && split && rank == 0 && t == t1 - 1 && warp == 4 && lane == 0) {
          // The last QK of this part is done: Q is no longer read, and the receive area
          // is free.  Expect rank 1's partial and tell it to send.
          mbar_arrive_expect_tx(BAR(C::B_XRECV), C::NCHV * C::CHUNK + C::STBYTES);
          mbar_arrive_cluster(mapa_shared(BAR(C::B_READY), 1u));
        }
        const int lim = CAUSAL ? (t == qt ? row + 1 : 128) : min(128, p.L - t * C::BN);
        // PV(g) completes a phase of ODONE[g & 1] (the (g >> 1)-th).  The softmax waits for
        // PV(g - 1) only before rescaling O (which must not race with it) and for the item's
        // last PV before its epilogue; it skips the phases in between.  A wait for PV(x) is
        // never two phases behind its barrier: that barrier's next phase is PV(x + 2), which
        // needs P of a tile this softmax has not formed yet (in the epilogue: the next
        // item's second PV, which waits for this epilogue's OFREE).  The P stored over S(t)
        // never races with PV(t - 2), which ran before QK(t) wrote S(t).
        auto wait_prev_pv = [&]() -> bool {
          if (!wait_warp(BAR(C::B_ODONE + ((g - 1u) & 1u)), ((g - 1u) >> 1) & 1u)) return false;
          tc_fence_after();
          return true;
        };
        bool rescaled = false;
        if constexpr (DSPLIT) {
          // S = this CTA's partial (its half of head_dim) + the peer's.  Send this row's
          // partial into the peer's buffer once the peer has read the previous one, take
          // the peer's out of this CTA's buffer, add (partial + partial in either CTA: the
          // same sum, so both run the same softmax), and free the buffer for the peer.
          const uint32_t s_row = tmem + lane_base + sb * 128u;
          uint32_t ra[64], rb[64];
          tmem_ld32x64_async(s_row, ra);
          tmem_ld32x64_async(s_row + 64, rb);
          tmem_wait_ld_fence64(ra);
          tmem_wait_ld_fence64(rb);
          if (g > 0 && !(ok = wait_warp_cluster(BAR(C::B_RFREE), (g - 1) & 1u))) break;
          const uint32_t peer_row = mapa_shared(recv_s + row * 512, rank ^ 1u);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            st_cluster_v4(peer_row + ((c ^ (row & 7)) << 4), ra[4 * c], ra[4 * c + 1], ra[4 * c + 2], ra[4 * c + 3]);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            st_cluster_v4(peer_row + (((16 + c) ^ (row & 7)) << 4), rb[4 * c], rb[4 * c + 1], rb[4 * c + 2],
                          rb[4 * c + 3]);
          mbar_arrive_cluster(mapa_shared(BAR(C::B_RECV), rank ^ 1u));
          if (!(ok = wait_warp_cluster(BAR(C::B_RECV), g & 1u))) break;
          const uint32_t my_row = recv_s + row * 512;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const uint4 x = ld_shared_v4(my_row + ((c ^ (row & 7)) << 4));
            ra[4 * c] = __float_as_uint(__uint_as_float(ra[4 * c]) + __uint_as_float(x.x));
            ra[4 * c + 1] = __float_as_uint(__uint_as_float(ra[4 * c + 1]) + __uint_as_float(x.y));
            ra[4 * c + 2] = __float_as_uint(__uint_as_float(ra[4 * c + 2]) + __uint_as_float(x.z));
            ra[4 * c + 3] = __float_as_uint(__uint_as_float(ra[4 * c + 3]) + __uint_as_float(x.w));
          }
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const uint4 x = ld_shared_v4(my_row + (((16 + c) ^ (row & 7)) << 4));
            rb[4 * c] = __float_as_uint(__uint_as_float(rb[4 * c]) + __uint_as_float(x.x));
            rb[4 * c + 1] = __float_as_uint(__uint_as_float(rb[4 * c + 1]) + __uint_as_float(x.y));
            rb[4 * c + 2] = __float_as_uint(__uint_as_float(rb[4 * c + 2]) + __uint_as_float(x.z));
            rb[4 * c + 3] = __float_as_uint(__uint_as_float(rb[4 * c + 3]) + __uint_as_float(x.w));
          }
          mbar_arrive_cluster(mapa_shared(BAR(C::B_RFREE), rank ^ 1u));
          if (!(ok = softmax_regs<C::DV>(ra, rb, s_row, tmem + lane_base + C::O_COL, lim, c2, t == t0, m_used, l,
                                         wait_prev_pv, &rescaled)))
            break;
        } else if constexpr (P_TMEM) {
          if (!(ok = softmax_tile<C::DV>(tmem + lane_base + sb * 128u, tmem + lane_base + C::O_COL, lim, c2, t == t0,
                                         m_used, l, wait_prev_pv, &rescaled)))
            break;
        } else {
          // P through shared memory: run the step into tensor memory, then move the fp16
          // P from the S columns into the swizzled shared-memory operand tile.
          if (!(ok = softmax_tile<C::DV>(tmem + lane_base + sb * 128u, tmem + lane_base + C::O_COL, lim, c2, t == t0,
                                         m_used, l, wait_prev_pv, &rescaled)))
            break;
          uint32_t pk[64];
          tmem_ld32x64(tmem + lane_base + sb * 128u, pk);
          const uint32_t pb = p_s + (g & 1u) * C::PBYTES + row * 128;
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) {
            const uint32_t addr = pb + (ch >> 3) * C::CHUNK + ((((ch & 7) ^ (row & 7))) << 4);
            st_shared_v4(addr, pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(BAR(C::B_PFULL + sb));
        if (t == t0 && warp == 4 && lane == 0) release_pending();
      }
      if (!ok) break;
      // ------------------------------------------------------------- epilogue
      if (!(ok = wait_warp(BAR(C::B_ODONE + ((g - 1u) & 1u)), ((g - 1u) >> 1) & 1u))) break;
      tc_fence_after();
      const int qb = il % C::NQB;
      const uint32_t stage = q_s + qb * C::QBYTES;  // the item's Q tile is no longer read
      const uint32_t o_row = tmem + lane_base + C::O_COL;
      if (SPLITKV && split && rank == 1) {
        // Rank 1 of a split item: its partial O / l (fp16) into its own staging tile and
        // its (m, l) beside it; warp 2 copies both into rank 0's receive area.  The stats
        // area is reused only once rank 0 has the previous split item's copy.
        if (ks > 0 && !(ok = wait_warp_cluster(BAR(C::B_XACK), (ks - 1) & 1))) break;
        stage_o_row<C::DV>(o_row, stage, row, 1.0f / l);
        float *const st = reinterpret_cast<float *>(base_ptr + (st_s - base)) + 2 * row;
        st[0] = m_used;
        st[1] = l;
        tc_fence_before();
        mbar_arrive(BAR(C::B_OFREE));
        fence_proxy_async_smem();
        mbar_arrive(BAR(C::B_XSTAGED));
        ++ks;
        ++il;
        continue;
      }
      float lse2 = m_used + __log2f(l);  // base-2 LSE of the row
      if (SPLITKV && split) {
        // Rank 0 of a split item: merge the two disjoint key ranges (STAGE_D.md, "Merge":
        // valid because no key is in both).  With M = max(m0, m1), the row's sum is
        // L = 2^(m0 - M) l0 + 2^(m1 - M) l1 and O = (2^(m0 - M) O0 + 2^(m1 - M) l1 O1hat) / L,
        // where O0 is this CTA's unnormalised accumulator and O1hat rank 1's O1 / l1.
        if (!(ok = wait_warp(BAR(C::B_XRECV), ks & 1))) break;
        if (warp == 4 && lane == 0) mbar_arrive_cluster(mapa_shared(BAR(C::B_XACK), 1u));
        const float *const st = reinterpret_cast<const float *>(base_ptr + (st_s - base)) + 2 * row;
        const float m1 = st[0], l1 = st[1];
        const float mx = fmaxf(m_used, m1);
        const float a0 = ex2_approx(m_used - mx), a1 = ex2_approx(m1 - mx) * l1;
        const float lsum = a0 * l + a1, inv = 1.0f / lsum;
        merge_o_row<C::DV>(o_row, xrecv_s, stage, row, a0 * inv, a1 * inv);
        lse2 = mx + __log2f(lsum);
        ++ks;
      } else {
        stage_o_row<C::DV>(o_row, stage, row, 1.0f / l);
      }
      tc_fence_before();
      mbar_arrive(BAR(C::B_OFREE));
      const int grow = qt * C::BM + row;
      if (half == 0 && grow < p.L) p.lse[static_cast<long long>(bh) * p.L + grow] = lse2 * 0.69314718055994531f;
      fence_proxy_async_smem();
      mbar_arrive(BAR(C::B_EPI));
      if (warp == 4 && lane == 0) {
        if (wait_bounded(BAR(C::B_EPI), ne & 1, abort_flag, p.status, kDevTimeoutEpilogue, LIM)) {
          for (int j = 0; j < C::NCHV; ++j)
            tma_store_3d(&tm_o, stage + j * C::CHUNK, half * C::DV + j * 64, qt * C::BM, bh);
          bulk_commit();
          qempty_pending = qb;
          // With one Q buffer the next item's Q load needs it back now.
          if (C::NQB < 2) release_pending();
        }
      }
      __syncwarp();
      ++ne;
      ++il;
    }
    if (warp == 4 && lane == 0) {
      release_pending();
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
  // A CTA of a pair stays until the other has stopped writing into its shared memory.
  if constexpr (C::CLUSTER) cluster_sync_all();
}

// Launch with programmatic stream serialization: the kernel may begin (prologue only, see
// grid_wait_prior) while the previous kernel in the stream is still finishing.
template <class Kern, class... Args>
cudaError_t launch_pdl(Kern kern, int grid, int block, int smem, cudaStream_t stream, const Args &...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Launch description shared by the per-head-dim translation units and the ABI.
struct FwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  FwdParams p;
  const SchedTable *tbl;
  int grid;     // CTAs (pairs of CTAs with dsplit; an even number of CTAs with splitkv)
  bool causal;
  bool p_smem;
  bool dsplit;   // head_dim 512 split over the two CTAs of a cluster
  bool splitkv;  // long query tiles' key ranges split over the two CTAs of a cluster
  cudaStream_t stream;
};

// Clusters of two CTAs, `ctas` CTAs in all, with programmatic stream serialization.
template <class Kern>
cudaError_t launch_pairs(Kern kern, int ctas, int smem, const FwdLaunch &a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p, *a.tbl);
}

// Clusters of two CTAs of the key-range split kernel that the current device can hold at
// once (clusters stay within a GPC, so an SM may be left over); -1 if the query fails.
template <int D>
int splitkv_max_clusters() {
  using C = FwdCfg<D, true, false, true>;
  auto *kern = attn_fwd_kernel<D, true, true, false, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess) return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = static_cast<size_t>(C::SMEM_BYTES);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return -1;
  return n;
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_splitkv(const FwdLaunch &a) {
  using C = FwdCfg<D, true, false, true>;
  auto *kern = attn_fwd_kernel<D, CAUSAL, true, false, true>;
  static int configured_mask = 0;  // one bit per device ordinal < 31
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 31 || !(configured_mask & (1 << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 31) configured_mask |= (1 << dev);
  }
  return launch_pairs(kern, a.grid, C::SMEM_BYTES, a);
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_dsplit(const FwdLaunch &a) {
  using C = FwdCfg<D, true, true>;
  auto *kern = attn_fwd_kernel<D, CAUSAL, true, true>;
  static int configured_mask = 0;  // one bit per device ordinal < 31
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 31 || !(configured_mask & (1 << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 31) configured_mask |= (1 << dev);
  }
  return launch_pairs(kern, 2 * a.grid, C::SMEM_BYTES, a);
}

template <int D, bool CAUSAL, bool P_TMEM>
cudaError_t launch_fwd_variant(const FwdLaunch &a) {
  using C = FwdCfg<D, P_TMEM>;
  auto *kern = attn_fwd_kernel<D, CAUSAL, P_TMEM, false>;
  static int configured_mask = 0;  // one bit per device ordinal < 31
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 31 || !(configured_mask & (1 << dev))) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 31) configured_mask |= (1 << dev);
  }
  return launch_pdl(kern, a.grid, 256, C::SMEM_BYTES, a.stream, a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p, *a.tbl);
}

template <int D>
cudaError_t launch_fwd_d(const FwdLaunch &a) {
  if constexpr (D != 256) {
    if (a.splitkv) return a.causal ? launch_fwd_splitkv<D, true>(a) : launch_fwd_splitkv<D, false>(a);
  }
  if constexpr (D <= 128) {
    if (a.p_smem)
      return a.causal ? launch_fwd_variant<D, true, false>(a) : launch_fwd_variant<D, false, false>(a);
  }
  if constexpr (D == 512) {
    if (a.dsplit) return a.causal ? launch_fwd_dsplit<D, true>(a) : launch_fwd_dsplit<D, false>(a);
  }
  return a.causal ? launch_fwd_variant<D, true, true>(a) : launch_fwd_variant<D, false, true>(a);
}

template <int D>
constexpr int fwd_items_per_tile() {
  return FwdCfg<D, true>::DVS;
}

cudaError_t launch_fwd_64(const FwdLaunch &a);
cudaError_t launch_fwd_128(const FwdLaunch &a);
cudaError_t launch_fwd_256(const FwdLaunch &a);
cudaError_t launch_fwd_512(const FwdLaunch &a);
int splitkv_clusters_64();
int splitkv_clusters_128();
int splitkv_clusters_512();

}  // namespace gbattn
