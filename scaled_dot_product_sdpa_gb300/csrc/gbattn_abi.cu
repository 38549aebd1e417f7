// gbattn_abi.cu -- the C ABI of libgbattn.so (declared in include/gbattn.h): argument
// checks, per-device setup, TMA descriptor encoding and kernel launch.  No entry point
// allocates device memory or synchronises (except attn_last_device_error, which is a
// documented host-blocking read of the device status word).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <numeric>
#include <queue>
#include <vector>

#include "attn_bwd.cuh"
#include "attn_decode.cuh"
#include "attn_fwd_kernel.cuh"
#include "attn_fwd_pp.cuh"
#include "gbattn.h"

namespace gbattn {

// One status word per device (each device that loads the module gets its own copy).
// Kernels receive its device address as a parameter; the first error code wins.
__device__ unsigned g_status;

cudaError_t launch_debug_scores(int d, const CUtensorMap &tq, const CUtensorMap &tk, float *s, int BH, int L,
                                float scale, unsigned *status, long long limit, cudaStream_t st);
cudaError_t launch_wait_probe(unsigned *status, long long limit, cudaStream_t st);

namespace {

constexpr long long kWaitLimitCycles = 1LL << 32;  // about two seconds of SM clock
constexpr int kMaxDevices = 64;

struct DevInfo {
  bool init = false;
  int cc_major = 0, cc_minor = 0, sm_count = 0;
  unsigned *status = nullptr;
  int dec_max_ranks[4] = {0, 0, 0, 0};  // decode cluster size limit per head_dim (0: not yet asked)
  int split_ctas[3] = {0, 0, 0};        // CTAs the key-range split kernel can hold at once, d = 64, 128, 512
};
DevInfo g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device setup on first use: capability, SM count, status-word address, and the
// driver's tensor-map encoder (fetched through the runtime, so no -lcuda link).
int device_info(DevInfo **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GBATTN_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return GBATTN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo &d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GBATTN_ERR_LAUNCH;
    if (d.cc_major != 10 || d.cc_minor != 3) return GBATTN_ERR_DEVICE;
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status) != cudaSuccess || addr == nullptr) return GBATTN_ERR_LAUNCH;
    d.status = static_cast<unsigned *>(addr);
    if (g_encode == nullptr) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return GBATTN_ERR_TENSORMAP;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.init = true;
  }
  *out = &d;
  return GBATTN_OK;
}

// [BH, L, D] fp16 viewed as a 3-D tensor (D innermost); box = 64 columns (128 B, the
// swizzle span) x box_rows rows x 1 head.  Rows past L read as zero and are never written.
int encode_bhld(CUtensorMap *tm, const void *ptr, int BH, int L, int D, int box_rows = 128) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2u,
                                 static_cast<cuuint64_t>(L) * static_cast<cuuint64_t>(D) * 2u};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
                              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GBATTN_OK : GBATTN_ERR_TENSORMAP;
}

// ------------------------------------------------------------------ work schedule
// The kernels a launch can use.
// kDSplit: the single-tile kernel at head_dim 512 with head_dim split over the two CTAs
// of a cluster (an option: slower on GB300, whose distributed shared memory moves the
// partial logits at ~17 B per cycle per SM); its schedule deals (head, query tile) items
// to clusters.
// kSplitKV: the single-tile kernel on clusters of two CTAs, the longest query tiles' key
// ranges split over the two CTAs of a cluster and merged by the first; its schedule lists
// such split tiles first, in the same order, for both CTAs of the cluster that runs them.
enum Kind { kSingle = 0, kPair = 1, kDSplit = 2, kSplitKV = 3 };

// Cost of a work item in units of one 128 x 128 tile step of one query tile in the
// two-tile kernel (it runs two such steps at once, one per query tile of its item), plus
// a per-item overhead (fill, drain and epilogue of the item's pipeline).  A tile step of
// the single-tile kernel costs about 1.2 such units.  Measured on GB300.
constexpr double kItemOverheadTwoSlot = 1.7;
constexpr double kSingleStepCost = 1.2;
constexpr double kItemOverheadSingle = 1.0;  // in single-tile steps
// Without a mask every step is a full tile, and a single-tile step costs only about 1.06
// units (non-causal, head_dim 64 and 128, measured on GB300: 1.05-1.07 on six shapes).
constexpr double kSingleStepCostNonCausal = 1.06;
// Key-range split: each part at least 3 key tiles (384 keys: a coarse split, far from the
// one-key splits that measured slowest; parts of 2 tiles made 512-key rows slower, parts of
// at least 4 left 1 x 12 x 1024 x 64 causal 8% slower than 3 on GB300), and each part of a split
// tile costs the handover and merge on top of its steps (in single-tile steps).
constexpr int kSplitMinPart = 3;
constexpr double kSplitOverhead = 1.5;
constexpr double kSplitGain = 0.9;  // taken only below this fraction of the other makespan

struct SchedKey {
  int kind, BH, nQ, nQB, dvs, causal, grid;
  int shortest_first;  // each CTA runs its items shortest first (see build_lpt)
  bool operator==(const SchedKey &o) const {
    return kind == o.kind && BH == o.BH && nQ == o.nQ && nQB == o.nQB && dvs == o.dvs && causal == o.causal &&
           grid == o.grid && shortest_first == o.shortest_first;
  }
};

long long count_items(const SchedKey &k) {
  return k.kind == kPair ? static_cast<long long>(k.BH) * k.nQB : static_cast<long long>(k.BH) * k.nQ * k.dvs;
}
// (kDSplit keys have dvs = 1: one item per head and query tile.)

// Key tiles of single-tile item r (decode_item's order: longest first when causal).
int item_tiles(const SchedKey &k, int r) { return k.causal ? k.nQ - r / (k.BH * k.dvs) : k.nQ; }

// Cost of item r, mirroring the kernels' item decoding (decode_item / pp_decode).
double item_cost(const SchedKey &k, int r) {
  if (k.kind == kPair) {
    if (!k.causal) return 2.0 * k.nQ + kItemOverheadTwoSlot;
    const int qb = k.nQB - 1 - r / k.BH;
    return (2 * qb + 1) + std::min(2 * qb + 2, k.nQ) + kItemOverheadTwoSlot;
  }
  return kSingleStepCost * (item_tiles(k, r) + kItemOverheadSingle);
}

// Schedule with key-range splits: the first `ns` items (the longest) are split; each goes
// to the cluster (CTAs 2c, 2c + 1) where it ends earliest, rank 0 taking ceil(n / 2) key
// tiles and rank 1 the rest; the other items then go longest first to the least-loaded
// CTA.  Returns the makespan; fills `lists` when given.
double split_assign(const SchedKey &k, int ns, std::vector<std::vector<uint16_t>> *lists) {
  const int N = static_cast<int>(count_items(k)), G = k.grid, C = G / 2;
  std::vector<double> load(G, 0.0);
  if (lists) lists->assign(G, {});
  for (int s = 0; s < ns; ++s) {
    const int n = item_tiles(k, s);
    const double c0 = kSingleStepCost * ((n + 1) / 2 + kSplitOverhead);
    const double c1 = kSingleStepCost * (n / 2 + kSplitOverhead);
    int best = 0;
    double best_end = 0.0;
    for (int c = 0; c < C; ++c) {
      const double e = std::max(load[2 * c] + c0, load[2 * c + 1] + c1);
      if (c == 0 || e < best_end) {
        best = c;
        best_end = e;
      }
    }
    load[2 * best] += c0;
    load[2 * best + 1] += c1;
    if (lists) {
      (*lists)[2 * best].push_back(static_cast<uint16_t>(N + s));
      (*lists)[2 * best + 1].push_back(static_cast<uint16_t>(N + s));
    }
  }
  using Slot = std::pair<double, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int c = 0; c < G; ++c) heap.push({load[c], c});
  double makespan = 0.0;
  for (const double x : load) makespan = std::max(makespan, x);
  for (int r = ns; r < N; ++r) {  // r order is longest first (item_tiles is non-increasing)
    const Slot sl = heap.top();
    heap.pop();
    const double w = item_cost(k, r);
    if (lists) (*lists)[sl.second].push_back(static_cast<uint16_t>(r));
    makespan = std::max(makespan, sl.first + w);
    heap.push({sl.first + w, sl.second});
  }
  return makespan;
}

// The split schedule: the number of split tiles (among those whose parts keep at least
// kSplitMinPart key tiles) with the smallest estimated makespan, at most two per cluster.
double build_split(const SchedKey &k, SchedTable &t) {
  std::memset(&t, 0, sizeof(t));
  const long long N = count_items(k);
  if (k.grid < 2 || k.grid % 2 || k.grid > kSchedMaxCtas || N > kSchedMaxItems) return -1.0;
  int cand = 0;
  while (cand < N && item_tiles(k, cand) >= 2 * kSplitMinPart) ++cand;
  const int ns_max = std::min({cand, k.grid, kSchedMaxItems - static_cast<int>(N)});
  const int step = std::max(1, ns_max / 48);
  int best_ns = 0;
  double best = split_assign(k, 0, nullptr);
  for (int ns = step; ns <= ns_max; ns += step) {
    const double m = split_assign(k, ns, nullptr);
    if (m < best - 1e-9) {
      best = m;
      best_ns = ns;
    }
  }
  std::vector<std::vector<uint16_t>> lists;
  split_assign(k, best_ns, &lists);
  int pos = 0;
  for (int c = 0; c < k.grid; ++c) {
    t.start[c] = static_cast<uint16_t>(pos);
    for (uint16_t r : lists[c]) t.items[pos++] = r;
  }
  t.start[k.grid] = static_cast<uint16_t>(pos);
  t.n = pos;
  return best;
}

// Longest-processing-time-first: take items by decreasing cost, give each to the CTA with
// the least accumulated cost (ties: lowest CTA).  Each CTA's list keeps assignment order.
// Returns the largest accumulated cost (the estimated makespan), or -1 with t.n = 0
// (the kernels' fixed snake order) when the items or CTAs do not fit the table.  With at
// most one item per CTA that snake order is the schedule itself: t.n = 0, and the
// makespan is returned.
double build_lpt(const SchedKey &k, SchedTable &t) {
  if (k.kind == kSplitKV) return build_split(k, t);
  std::memset(&t, 0, sizeof(t));
  const long long n_items = count_items(k);
  if (n_items > kSchedMaxItems || k.grid > kSchedMaxCtas || k.grid <= 0) return -1.0;
  std::vector<std::pair<double, int>> order;
  order.reserve(static_cast<size_t>(n_items));
  for (int r = 0; r < n_items; ++r) order.push_back({item_cost(k, r), r});
  std::stable_sort(order.begin(), order.end(),
                   [](const std::pair<double, int> &a, const std::pair<double, int> &b) { return a.first > b.first; });
  // At most one item per CTA (make_key then sets the grid to the item count): the order
  // above, longest first, puts item c on CTA c, which is the kernels' own order, so no
  // table is passed (t.n = 0) and the kernels take their item without reading one.
  if (n_items <= k.grid && (k.kind == kSingle || k.kind == kPair))
    return order.empty() ? 0.0 : order.front().first;
  using Slot = std::pair<double, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int c = 0; c < k.grid; ++c) heap.push({0.0, c});
  std::vector<std::vector<uint16_t>> lists(k.grid);
  double makespan = 0.0;
  for (const auto &w : order) {
    const Slot s = heap.top();
    heap.pop();
    lists[s.second].push_back(static_cast<uint16_t>(w.second));
    makespan = std::max(makespan, s.first + w.first);
    heap.push({s.first + w.first, s.second});
  }
  // A CTA runs its items longest first, except when k.shortest_first (make_key).
  const bool shortest_first = k.shortest_first != 0;
  int pos = 0;
  for (int c = 0; c < k.grid; ++c) {
    t.start[c] = static_cast<uint16_t>(pos);
    if (shortest_first)
      for (auto it = lists[c].rbegin(); it != lists[c].rend(); ++it) t.items[pos++] = *it;
    else
      for (uint16_t r : lists[c]) t.items[pos++] = r;
  }
  t.start[k.grid] = static_cast<uint16_t>(pos);
  t.n = static_cast<int>(n_items);
  return makespan;
}

struct SchedEntry {
  bool valid = false;
  unsigned long long stamp = 0;
  SchedKey key{};
  double makespan = 0.0;
  SchedTable tbl;
};
SchedEntry g_sched_cache[16];
unsigned long long g_sched_clock = 0;
std::mutex g_sched_mu;

// The schedule for `k`, built and cached on a miss; copies the table into `out` when
// given.  Returns the estimated makespan (< 0: no table, snake order).
double get_schedule(const SchedKey &k, SchedTable *out) {
  std::lock_guard<std::mutex> lock(g_sched_mu);
  SchedEntry *victim = &g_sched_cache[0];
  for (SchedEntry &e : g_sched_cache) {
    if (e.valid && e.key == k) {
      e.stamp = ++g_sched_clock;
      if (out) *out = e.tbl;
      return e.makespan;
    }
    if (!e.valid || e.stamp < victim->stamp) victim = &e;
  }
  victim->makespan = build_lpt(k, victim->tbl);
  victim->key = k;
  victim->valid = true;
  victim->stamp = ++g_sched_clock;
  if (out) *out = victim->tbl;
  return victim->makespan;
}

// ------------------------------------------------------------------ launch plan
// The kernel and grid of a launch.  Options force a kernel; otherwise head_dim > 128
// takes the single-tile kernel, and head_dim <= 128 the two-tile kernel, unless that has
// fewer than two items per SM: then whichever of the two has the smaller estimated
// makespan (measured on GB300 at 1x16x512x64 causal 7.6 vs 11.2 us, 1x32x1024x128
// causal 15.9 vs 23.7 us, both for the single-tile kernel).
// Whether each CTA runs its items shortest first: in the two-tile kernel at head_dim 128
// when every item lies within one 512-query block (items of at most 7 tile steps, two to
// four per CTA), which measured faster on GB300 (8x32x512x128 causal 30.8 -> 30.1 us,
// 16x16x512x128 30.8 -> 30.2), while head_dim 64 (8x32x512x64 26.1 -> 26.6), longer rows
// and the single-tile kernel were flat or up to 2% slower.
int shortest_first_rule(int kind, int nQB, int d) { return kind == kPair && nQB <= 2 && d == 128 ? 1 : 0; }

SchedKey make_key(int kind, int BH, int L, int d, int causal, int grid) {
  const int nQ = (L + 127) / 128, nQB = (L + 255) / 256, dvs = d > 256 ? d / 256 : 1;
  SchedKey k{kind, BH, nQ, nQB, kind == kSingle || kind == kSplitKV ? dvs : 1, causal != 0 ? 1 : 0, grid,
             shortest_first_rule(kind, nQB, d)};
  const long long n = count_items(k);
  if (kind == kSplitKV) {
    // An even number of CTAs (clusters of two), at most two per item.
    k.grid = static_cast<int>(std::min<long long>(grid, 2 * n)) & ~1;
    if (k.grid < 2) k.grid = 2;
  } else if (n < grid) {
    k.grid = static_cast<int>(n);
  }
  return k;
}

// head_dims the key-range split is built for
bool split_kv_dim(int d) { return d == 64 || d == 128 || d == 512; }

// `split_ctas`: CTAs (clusters of two) the key-range split kernel can hold at once.
int choose_plan(int BH, int L, int d, int causal, int sm_count, int flags, int grid_limit, SchedKey &out,
                double &makespan, int split_ctas) {
  int grid = sm_count;
  if (grid_limit > 0 && grid_limit < grid) grid = grid_limit;
  const int split_grid = std::max(2, std::min(grid, split_ctas));
  int kind;
  if (flags & GBATTN_FLAG_DSPLIT) {
    kind = kDSplit;  // clusters of two CTAs: the schedule's lanes are the clusters
    grid = std::max(1, grid / 2);
  } else if (flags & GBATTN_FLAG_SPLIT_KV) {
    kind = kSplitKV;
    grid = split_grid;
  } else if (flags & (GBATTN_FLAG_P_SMEM | GBATTN_FLAG_SINGLE_TILE) || d > 128) {
    kind = kSingle;
  } else if (flags & GBATTN_FLAG_TWO_TILE) {
    kind = kPair;
  } else {
    const SchedKey pair = make_key(kPair, BH, L, d, causal, grid);
    if (count_items(pair) > INT_MAX) return GBATTN_ERR_DIMS;
    if (count_items(pair) >= 2LL * grid) {
      kind = kPair;
      if (!causal) {
        // Non-causal items are all alike, so either kernel's makespan is its busiest
        // CTA's whole items: ceil(items / grid) of them.  The two-tile kernel's items are
        // half as many and twice as long, and when its count leaves the last round of
        // items thinly spread the single-tile kernel's is the shorter (GB300, non-causal
        // head_dim 64, 512 two-tile items: 4 x 16 x 2048 103.0 -> 97.1 us, 2 x 16 x 4096
        // 197.3 -> 182.5).
        const SchedKey single = make_key(kSingle, BH, L, d, causal, grid);
        const double rp = std::ceil(static_cast<double>(count_items(pair)) / grid);
        const double rs = std::ceil(static_cast<double>(count_items(single)) / grid);
        const double mp = rp * (2.0 * pair.nQ + kItemOverheadTwoSlot);
        const double ms = rs * kSingleStepCostNonCausal * (single.nQ + kItemOverheadSingle);
        if (ms < mp) kind = kSingle;
      }
    } else {
      double best = 0.0;
      kind = -1;
      for (int cand : {kSingle, kPair}) {
        const double m = get_schedule(make_key(cand, BH, L, d, causal, grid), nullptr);
        if (m >= 0.0 && (kind < 0 || m < best)) {
          best = m;
          kind = cand;
        }
      }
      if (kind < 0) kind = kPair;
    }
  }
  // Without options, key-range splits replace the choice above when their schedule is
  // clearly shorter (few query tiles, some much longer than the average load); not when
  // the two-tile kernel has enough items (that kernel's grid is full).
  if (flags == 0 && split_kv_dim(d) && grid >= 2 && (kind == kSingle || count_items(make_key(kPair, BH, L, d, causal, grid)) < 2LL * grid)) {
    const double cur = get_schedule(make_key(kind, BH, L, d, causal, grid), nullptr);
    const double split = get_schedule(make_key(kSplitKV, BH, L, d, causal, split_grid), nullptr);
    if (cur >= 0.0 && split >= 0.0 && split < kSplitGain * cur) {
      kind = kSplitKV;
      grid = split_grid;
    }
  }
  out = make_key(kind, BH, L, d, causal, grid);
  if (count_items(out) > INT_MAX) return GBATTN_ERR_DIMS;
  makespan = get_schedule(out, nullptr);
  return GBATTN_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The option bits of attn_fwd_ex: known bits only, the two-tile kernel not together with
// a single-tile option, and the two-tile kernel and shared-memory P only for d <= 128.
int check_flags(int flags, int d) {
  if (flags & ~(GBATTN_FLAG_P_SMEM | GBATTN_FLAG_SINGLE_TILE | GBATTN_FLAG_TWO_TILE | GBATTN_FLAG_DSPLIT |
                GBATTN_FLAG_SPLIT_KV))
    return GBATTN_ERR_FLAGS;
  if ((flags & GBATTN_FLAG_SPLIT_KV) && (flags & ~GBATTN_FLAG_SPLIT_KV)) return GBATTN_ERR_FLAGS;
  if ((flags & GBATTN_FLAG_SPLIT_KV) && !split_kv_dim(d)) return GBATTN_ERR_HEAD_DIM;
  if ((flags & GBATTN_FLAG_TWO_TILE) && (flags & (GBATTN_FLAG_SINGLE_TILE | GBATTN_FLAG_P_SMEM)))
    return GBATTN_ERR_FLAGS;
  if ((flags & GBATTN_FLAG_DSPLIT) && (flags & ~GBATTN_FLAG_DSPLIT)) return GBATTN_ERR_FLAGS;
  if ((flags & (GBATTN_FLAG_P_SMEM | GBATTN_FLAG_TWO_TILE)) && d > 128) return GBATTN_ERR_HEAD_DIM;
  if ((flags & GBATTN_FLAG_DSPLIT) && d != 512) return GBATTN_ERR_HEAD_DIM;
  return GBATTN_OK;
}

int check_shape(int B, int H, int L, int d) {
  if (B <= 0 || H <= 0 || L <= 0) return GBATTN_ERR_DIMS;
  const long long rows = static_cast<long long>(B) * H * L;
  if (rows > INT_MAX || static_cast<long long>(B) * H > INT_MAX) return GBATTN_ERR_DIMS;
  if (d != 64 && d != 128 && d != 256 && d != 512) return GBATTN_ERR_HEAD_DIM;
  return GBATTN_OK;
}

// Decode launch plan: the CTAs per head (one cluster, a power of two) and the keys each
// one streams (whole key tiles).  The widest cluster that keeps the launch within one wave
// of two CTAs per SM, at most max_ranks (and the head_dim's own bound), at least one key
// tile per CTA, and one CTA per head when the heads alone fill that wave.  (Measured on
// GB300 at L = 8192, same box, against the earlier rule of two such waves: 64 heads 54.0
// -> 40.8 us, 128 heads 84.9 -> 77.3, 256 heads 158.9 -> 150.6 (at d = 64 83.8 -> 76.9),
// 512 heads 312 -> 297; fewer, longer CTAs stream faster than more, shorter ones.)
// When the widest cluster still leaves the SMs short of CTAs (few heads) and a workspace
// is given, each head's keys are also split over `groups` clusters: clusters of two CTAs,
// as many per head as one wave of two CTAs per SM holds, when that is at most
// kDecMaxGroups and leaves every CTA a key tile; otherwise clusters of at most 8 CTAs, as
// many as that wave holds, at most kDecMaxGroups.  Clusters of two fill the SMs' two CTA
// slots evenly; wider ones leave some SMs with one CTA (and so half the keys of the rest)
// and, past one wave, a tail.  (Measured on GB300 at d = 128, same box: 1 x 8 heads x 1M
// keys 8 x 4 clusters of 8 CTAs 619-629 us, 2 x 19 of 2 584 us; 1 x 12 x 256K 315 -> 224
// us; 1 x 16 x 256K 344 -> 296; 1 x 32 x 128K 299 -> 296; 1 x 6 x 512K at d = 64 151 ->
// 117; 320 CTAs in clusters of 4 or 8, just past one wave, 800-830 us on the 1M shape.)
void decode_plan(long long BH, int L, int d, int sm_count, int max_ranks, bool grouped, int &ranks, int &groups,
                 int &keys_per_rank) {
  max_ranks = std::min(max_ranks, dec_max_ranks_for(d));
  const int kt = dec_key_tile(d);
  const long long tiles = (static_cast<long long>(L) + kt - 1) / kt;
  const long long want = std::max(1LL, 2LL * sm_count / BH);  // CTAs per head in that wave
  int r = 1;
  while (2 * r <= want && 2 * r <= max_ranks && 2 * r <= tiles) r *= 2;
  long long g = 1;
  if (grouped && r < want) {
    // Clusters of two CTAs, as many per head as one wave of two CTAs per SM holds, when
    // that fits the workspace's rows per head; otherwise wider clusters.
    const long long g2 = 2LL * sm_count / (BH * 2);
    if (g2 >= 2 && g2 <= kDecMaxGroups && tiles >= 2 * g2) {
      r = 2;
      g = g2;
    } else {
      r = std::min(r, kDecGroupedRanks);
      g = std::max(1LL, 2LL * sm_count / (BH * r));
      g = std::min({g, static_cast<long long>(kDecMaxGroups), std::max(1LL, tiles / r)});
    }
  }
  ranks = r;
  groups = static_cast<int>(g);
  keys_per_rank = static_cast<int>((tiles + g * r - 1) / (g * r)) * kt;
}

int dec_dim_index(int d) { return d == 64 ? 0 : d == 128 ? 1 : d == 256 ? 2 : 3; }

}  // namespace
}  // namespace gbattn

using namespace gbattn;

extern "C" int attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int L,
                           int d, int causal, float scale, void *stream, int flags, int grid_limit) {
  if (!q || !k || !v || !o || !lse) return GBATTN_ERR_NULL;
  int rc = check_shape(B, H, L, d);
  if (rc != GBATTN_OK) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return GBATTN_ERR_ALIGN;
  if (!std::isfinite(scale) || !(scale > 0.f)) return GBATTN_ERR_SCALE;
  const bool p_smem = (flags & GBATTN_FLAG_P_SMEM) != 0;
  if ((rc = check_flags(flags, d)) != GBATTN_OK) return rc;
  if (grid_limit < 0) return GBATTN_ERR_DIMS;
  const long long rows = static_cast<long long>(B) * H * L;
  const size_t tbytes = static_cast<size_t>(rows) * static_cast<size_t>(d) * 2u;
  const size_t lbytes = static_cast<size_t>(rows) * 4u;
  if (overlaps(o, tbytes, q, tbytes) || overlaps(o, tbytes, k, tbytes) || overlaps(o, tbytes, v, tbytes) ||
      overlaps(lse, lbytes, q, tbytes) || overlaps(lse, lbytes, k, tbytes) || overlaps(lse, lbytes, v, tbytes) ||
      overlaps(lse, lbytes, o, tbytes))
    return GBATTN_ERR_ALIAS;

  DevInfo *di = nullptr;
  if ((rc = device_info(&di)) != GBATTN_OK) return rc;

  const int BH = B * H;
  int split_ctas = di->sm_count;
  if (split_kv_dim(d)) {
    int &sc = di->split_ctas[d == 64 ? 0 : d == 128 ? 1 : 2];
    if (sc == 0) {
      const int n = d == 64 ? splitkv_clusters_64() : d == 128 ? splitkv_clusters_128() : splitkv_clusters_512();
      sc = n > 0 ? std::min(2 * n, di->sm_count & ~1) : (di->sm_count & ~1);
    }
    split_ctas = sc;
  }
  SchedKey key;
  double makespan = 0.0;
  if ((rc = choose_plan(BH, L, d, causal, di->sm_count, flags, grid_limit, key, makespan, split_ctas)) != GBATTN_OK)
    return rc;
  const bool two_tile = key.kind == kPair;

  FwdLaunch a;
  SchedTable tbl;
  a.tbl = &tbl;
  if (encode_bhld(&a.tm_q, q, BH, L, d) || encode_bhld(&a.tm_k, k, BH, L, d) || encode_bhld(&a.tm_v, v, BH, L, d) ||
      encode_bhld(&a.tm_o, o, BH, L, d))
    return GBATTN_ERR_TENSORMAP;
  a.grid = key.grid;
  get_schedule(key, &tbl);
  a.causal = causal != 0;
  a.p_smem = p_smem;
  a.dsplit = key.kind == kDSplit;
  a.splitkv = key.kind == kSplitKV;
  a.stream = static_cast<cudaStream_t>(stream);
  a.p.lse = lse;
  a.p.status = di->status;
  a.p.wait_limit = kWaitLimitCycles;
  a.p.BH = BH;
  a.p.L = L;
  a.p.nQ = key.nQ;
  a.p.nQB = key.nQB;
  a.p.n_items = static_cast<int>(count_items(key));
  a.p.c2 = scale * 1.4426950408889634f;

  cudaError_t e;
  if (two_tile) {
    e = d == 64 ? launch_fwd_pp_64(a) : launch_fwd_pp_128(a);
    return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_LAUNCH;
  }
  switch (d) {
    case 64: e = launch_fwd_64(a); break;
    case 128: e = launch_fwd_128(a); break;
    case 256: e = launch_fwd_256(a); break;
    default: e = launch_fwd_512(a); break;
  }
  return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_LAUNCH;
}

extern "C" int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int L, int d,
                        int causal, float scale, void *stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, H, L, d, causal, scale, stream, 0, 0);
}

// ------------------------------------------------------------------ host buffers
namespace gbattn {
namespace {

// Heads per chunk of attn_fwd_host: chunks of about 24 MB of Q+K+V, at least 4 chunks
// when there are enough heads.  On GB300 every host-link copy costs ~2 us of ramp on top
// of its bytes (4 MB copies reach ~177 GB/s, 32 MB ones ~206), and only the copy out of
// the last chunk is not hidden behind the copies in, so a few large chunks with a short
// final one beat many small chunks.
long long host_chunk_heads(long long BH, int L, int d) {
  const long long head_qkv = 3LL * L * d * 2;
  long long ch = std::max(1LL, (24LL << 20) / head_qkv);
  ch = std::min(ch, std::max(1LL, (BH + 3) / 4));
  return std::min(ch, BH);
}
// Size of the chunk of attn_fwd_host that starts at head h0: `ch` heads, except that the
// last `ch` or fewer heads are cut 3:1 (when there are at least 4) so that the final
// kernel and copy out, which nothing overlaps, are short.
long long host_chunk_at(long long BH, long long ch, long long h0) {
  const long long r = BH - (BH - 1) / ch * ch;  // heads of the last full-size slot, 1..ch
  const long long tail = BH - r;
  if (h0 < tail) return ch;
  if (h0 == tail && r >= 4) return r - r / 4;
  return BH - h0;
}
size_t host_chunk_bytes(long long ch, int L, int d) {
  auto up = [](size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); };
  const size_t t = static_cast<size_t>(ch) * L * d * 2u;
  return 4u * up(t) + up(static_cast<size_t>(ch) * L * 4u);  // q, k, v, o, lse
}

// Streams and events of the host-buffer pipeline, created once per device.
struct HostPipe {
  bool init = false;
  cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
  cudaEvent_t start = nullptr, in_done[2] = {}, comp_done[2] = {}, out_done[2] = {};
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;

int host_pipe(HostPipe **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GBATTN_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return GBATTN_ERR_DEVICE;
  HostPipe &hp = g_pipe[dev];
  if (!hp.init) {
    const unsigned f = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.s_comp, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.start, f) != cudaSuccess)
      return GBATTN_ERR_LAUNCH;
    for (int i = 0; i < 2; ++i)
      if (cudaEventCreateWithFlags(&hp.in_done[i], f) != cudaSuccess ||
          cudaEventCreateWithFlags(&hp.comp_done[i], f) != cudaSuccess ||
          cudaEventCreateWithFlags(&hp.out_done[i], f) != cudaSuccess)
        return GBATTN_ERR_LAUNCH;
    hp.init = true;
  }
  *out = &hp;
  return GBATTN_OK;
}

}  // namespace
}  // namespace gbattn

extern "C" size_t attn_fwd_host_workspace_size(int B, int H, int L, int d) {
  if (check_shape(B, H, L, d) != GBATTN_OK) return 0;
  const long long BH = static_cast<long long>(B) * H;
  return 2u * host_chunk_bytes(host_chunk_heads(BH, L, d), L, d);
}

extern "C" int attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int L,
                             int d, int causal, float scale, void *workspace, size_t workspace_bytes, void *stream) {
  if (!q || !k || !v || !o || !lse || !workspace) return GBATTN_ERR_NULL;
  int rc = check_shape(B, H, L, d);
  if (rc != GBATTN_OK) return rc;
  if (!std::isfinite(scale) || !(scale > 0.f)) return GBATTN_ERR_SCALE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GBATTN_ERR_ALIGN;
  const long long BH = static_cast<long long>(B) * H;
  const long long ch = host_chunk_heads(BH, L, d);
  const size_t slot_bytes = host_chunk_bytes(ch, L, d);
  if (workspace_bytes < 2u * slot_bytes) return GBATTN_ERR_WORKSPACE;
  const size_t rows = static_cast<size_t>(BH) * L;
  const size_t tbytes = rows * d * 2u, lbytes = rows * 4u;
  if (overlaps(o, tbytes, q, tbytes) || overlaps(o, tbytes, k, tbytes) || overlaps(o, tbytes, v, tbytes) ||
      overlaps(lse, lbytes, q, tbytes) || overlaps(lse, lbytes, k, tbytes) || overlaps(lse, lbytes, v, tbytes) ||
      overlaps(lse, lbytes, o, tbytes))
    return GBATTN_ERR_ALIAS;
  DevInfo *di = nullptr;
  if ((rc = device_info(&di)) != GBATTN_OK) return rc;
  HostPipe *hp = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    if ((rc = host_pipe(&hp)) != GBATTN_OK) return rc;
    const cudaStream_t user = static_cast<cudaStream_t>(stream);
    auto up = [](size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); };
    const size_t t_ch = up(static_cast<size_t>(ch) * L * d * 2u);
    // Everything starts after the work already queued on the caller's stream.
    if (cudaEventRecord(hp->start, user) != cudaSuccess || cudaStreamWaitEvent(hp->s_in, hp->start, 0) != cudaSuccess)
      return GBATTN_ERR_LAUNCH;
    const size_t head_t = static_cast<size_t>(L) * d * 2u, head_l = static_cast<size_t>(L) * 4u;
    int c = 0;
    for (long long h0 = 0, nh = 0; h0 < BH; h0 += nh, ++c) {
      nh = host_chunk_at(BH, ch, h0);
      const int slot = c & 1;
      char *base = static_cast<char *>(workspace) + slot * slot_bytes;
      char *dq = base, *dk = base + t_ch, *dv = base + 2 * t_ch, *dO = base + 3 * t_ch;
      float *dl = reinterpret_cast<float *>(base + 4 * t_ch);
      const size_t nb = static_cast<size_t>(nh) * head_t, nl = static_cast<size_t>(nh) * head_l;
      const size_t off = static_cast<size_t>(h0) * head_t, offl = static_cast<size_t>(h0) * head_l;
      // The slot is free once the chunk two back has been copied out (its kernel read
      // the inputs before that).
      if (c >= 2 && cudaStreamWaitEvent(hp->s_in, hp->out_done[slot], 0) != cudaSuccess) return GBATTN_ERR_LAUNCH;
      if (cudaMemcpyAsync(dq, static_cast<const char *>(q) + off, nb, cudaMemcpyHostToDevice, hp->s_in) != cudaSuccess ||
          cudaMemcpyAsync(dk, static_cast<const char *>(k) + off, nb, cudaMemcpyHostToDevice, hp->s_in) != cudaSuccess ||
          cudaMemcpyAsync(dv, static_cast<const char *>(v) + off, nb, cudaMemcpyHostToDevice, hp->s_in) != cudaSuccess ||
          cudaEventRecord(hp->in_done[slot], hp->s_in) != cudaSuccess ||
          cudaStreamWaitEvent(hp->s_comp, hp->in_done[slot], 0) != cudaSuccess)
        return GBATTN_ERR_LAUNCH;
      if ((rc = attn_fwd(dq, dk, dv, dO, dl, 1, static_cast<int>(nh), L, d, causal, scale, hp->s_comp)) != GBATTN_OK)
        return rc;
      if (cudaEventRecord(hp->comp_done[slot], hp->s_comp) != cudaSuccess ||
          cudaStreamWaitEvent(hp->s_out, hp->comp_done[slot], 0) != cudaSuccess ||
          cudaMemcpyAsync(static_cast<char *>(o) + off, dO, nb, cudaMemcpyDeviceToHost, hp->s_out) != cudaSuccess ||
          cudaMemcpyAsync(reinterpret_cast<char *>(lse) + offl, dl, nl, cudaMemcpyDeviceToHost, hp->s_out) !=
              cudaSuccess ||
          cudaEventRecord(hp->out_done[slot], hp->s_out) != cudaSuccess)
        return GBATTN_ERR_LAUNCH;
    }
    // The caller's stream continues once the last copy out is done (the copies out run
    // in order on one stream).
    if (cudaStreamWaitEvent(user, hp->out_done[(c - 1) & 1], 0) != cudaSuccess) return GBATTN_ERR_LAUNCH;
  }
  return GBATTN_OK;
}

extern "C" long long attn_bwd_workspace_bytes(int B, int H, int L) {
  if (B <= 0 || H <= 0 || L <= 0) return GBATTN_ERR_DIMS;
  const long long BH = static_cast<long long>(B) * H, Lp = (static_cast<long long>(L) + 127) / 128 * 128;
  if (BH * Lp > INT_MAX) return GBATTN_ERR_DIMS;
  return 8 * BH * Lp;
}

namespace gbattn {
// Every check of attn_bwd's arguments (no CUDA call), in attn_bwd's order: NULL pointers,
// shape, head_dim, alignment, scale, overlaps.  `workspace` may be NULL only when
// `check_workspace` is false (attn_bwd_noalloc, whose workspace is the library's own).
int bwd_check_args(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
                   const void *dq, const void *dk, const void *dv, const void *workspace, bool check_workspace, int B,
                   int H, int L, int d, float scale) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || (check_workspace && !workspace))
    return GBATTN_ERR_NULL;
  int rc = check_shape(B, H, L, d);
  if (rc != GBATTN_OK) return rc;
  if (d != 64 && d != 128) return GBATTN_ERR_HEAD_DIM;
  const long long wsb = attn_bwd_workspace_bytes(B, H, L);
  if (wsb < 0) return GBATTN_ERR_DIMS;
  const void *ins[6] = {q, k, v, o, lse, dout};
  const void *outs[4] = {dq, dk, dv, workspace};
  const int n_out = check_workspace ? 4 : 3;
  for (const void *x : ins)
    if (!aligned16(x)) return GBATTN_ERR_ALIGN;
  for (int i = 0; i < n_out; ++i)
    if (!aligned16(outs[i])) return GBATTN_ERR_ALIGN;
  if (!std::isfinite(scale) || !(scale > 0.f)) return GBATTN_ERR_SCALE;
  const long long BH = static_cast<long long>(B) * H;
  const size_t tb = static_cast<size_t>(BH) * L * d * 2u, lb = static_cast<size_t>(BH) * L * 4u;
  const size_t in_sz[6] = {tb, tb, tb, tb, lb, tb};
  const size_t out_sz[4] = {tb, tb, tb, static_cast<size_t>(wsb)};
  for (int i = 0; i < n_out; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlaps(outs[i], out_sz[i], ins[j], in_sz[j])) return GBATTN_ERR_ALIAS;
    for (int j = i + 1; j < n_out; ++j)
      if (overlaps(outs[i], out_sz[i], outs[j], out_sz[j])) return GBATTN_ERR_ALIAS;
  }
  return GBATTN_OK;
}
}  // namespace gbattn

extern "C" int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                        const void *dout, void *dq, void *dk, void *dv, void *workspace, int B, int H, int L, int d,
                        int causal, float scale, void *stream) {
  int rc = bwd_check_args(q, k, v, o, lse, dout, dq, dk, dv, workspace, true, B, H, L, d, scale);
  if (rc != GBATTN_OK) return rc;
  const long long BH = static_cast<long long>(B) * H;
  DevInfo *di = nullptr;
  if ((rc = device_info(&di)) != GBATTN_OK) return rc;
  BwdLaunch a;
  const int bh = static_cast<int>(BH);
  if (encode_bhld(&a.tm_q128, q, bh, L, d) || encode_bhld(&a.tm_do128, dout, bh, L, d) ||
      encode_bhld(&a.tm_k128, k, bh, L, d) || encode_bhld(&a.tm_v128, v, bh, L, d) ||
      encode_bhld(&a.tm_dq128, dq, bh, L, d) || encode_bhld(&a.tm_dk128, dk, bh, L, d) ||
      encode_bhld(&a.tm_dv128, dv, bh, L, d))
    return GBATTN_ERR_TENSORMAP;
  a.p.lse = lse;
  a.p.o = static_cast<const __half *>(o);
  a.p.status = di->status;
  a.p.wait_limit = kWaitLimitCycles;
  a.p.BH = bh;
  a.p.L = L;
  a.p.n128 = (L + 127) / 128;
  a.p.Lp = a.p.n128 * 128;
  a.p.ws_lse2 = static_cast<float *>(workspace);
  a.p.ws_d = a.p.ws_lse2 + static_cast<long long>(bh) * a.p.Lp;
  a.p.items = bh * a.p.n128;
  a.p.c2 = scale * 1.4426950408889634f;
  a.p.scale = scale;
  a.grid = std::min(a.p.items, di->sm_count);
  a.causal = causal != 0;
  a.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t e = d == 64 ? launch_bwd_64(a) : launch_bwd_128(a);
  return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_LAUNCH;
}

extern "C" long long attn_decode_workspace_bytes(int B, int H, int d) {
  if (B <= 0 || H <= 0) return GBATTN_ERR_DIMS;
  if (d != 64 && d != 128 && d != 256 && d != 512) return GBATTN_ERR_HEAD_DIM;
  return dec_workspace_bytes(static_cast<long long>(B) * H, d);
}

extern "C" int attn_decode(const void *q, const void *k, const void *v, void *o, float *lse, void *workspace, int B,
                           int H, int L, int d, float scale, void *stream) {
  if (!q || !k || !v || !o || !lse) return GBATTN_ERR_NULL;
  int rc = check_shape(B, H, L, d);
  if (rc != GBATTN_OK) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(workspace))
    return GBATTN_ERR_ALIGN;
  if (!std::isfinite(scale) || !(scale > 0.f)) return GBATTN_ERR_SCALE;
  const long long BH = static_cast<long long>(B) * H;
  const size_t qbytes = static_cast<size_t>(BH) * d * 2u, kvbytes = qbytes * static_cast<size_t>(L),
               lbytes = static_cast<size_t>(BH) * 4u;
  if (overlaps(o, qbytes, q, qbytes) || overlaps(o, qbytes, k, kvbytes) || overlaps(o, qbytes, v, kvbytes) ||
      overlaps(lse, lbytes, q, qbytes) || overlaps(lse, lbytes, k, kvbytes) || overlaps(lse, lbytes, v, kvbytes) ||
      overlaps(lse, lbytes, o, qbytes))
    return GBATTN_ERR_ALIAS;
  if (workspace) {
    const size_t wb = static_cast<size_t>(dec_workspace_bytes(BH, d));
    if (overlaps(workspace, wb, q, qbytes) || overlaps(workspace, wb, k, kvbytes) ||
        overlaps(workspace, wb, v, kvbytes) || overlaps(workspace, wb, o, qbytes) || overlaps(workspace, wb, lse, lbytes))
      return GBATTN_ERR_ALIAS;
  }
  DevInfo *di = nullptr;
  if ((rc = device_info(&di)) != GBATTN_OK) return rc;
  int &max_ranks = di->dec_max_ranks[dec_dim_index(d)];
  if (max_ranks == 0) {
    const int mr = decode_max_ranks(d);
    if (mr <= 0) return GBATTN_ERR_LAUNCH;
    max_ranks = mr;
  }
  DecLaunch a;
  const int kt = dec_key_tile(d);
  if (encode_bhld(&a.tm_k, k, static_cast<int>(BH), L, d, kt) || encode_bhld(&a.tm_v, v, static_cast<int>(BH), L, d, kt))
    return GBATTN_ERR_TENSORMAP;
  decode_plan(BH, L, d, di->sm_count, max_ranks, workspace != nullptr, a.p.ranks, a.p.groups, a.p.keys_per_rank);
  a.p.ws = static_cast<float *>(workspace);
  a.p.q = q;
  a.p.o = o;
  a.p.lse = lse;
  a.p.status = di->status;
  a.p.wait_limit = kWaitLimitCycles;
  a.p.BH = static_cast<int>(BH);
  a.p.L = L;
  a.p.c2 = scale * 1.4426950408889634f;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (d) {
    case 64: e = launch_decode_64(a); break;
    case 128: e = launch_decode_128(a); break;
    case 256: e = launch_decode_256(a); break;
    default: e = launch_decode_512(a); break;
  }
  return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_LAUNCH;
}

extern "C" int attn_debug_decode_plan(int B, int H, int L, int d, int sm_count, int max_ranks, int grouped,
                                      int *out) {
  if (!out) return GBATTN_ERR_NULL;
  const int rc = check_shape(B, H, L, d);
  if (rc != GBATTN_OK) return rc;
  if (sm_count <= 0 || max_ranks < 1 || max_ranks > kDecMaxRanks) return GBATTN_ERR_DIMS;
  decode_plan(static_cast<long long>(B) * H, L, d, sm_count, max_ranks, grouped != 0, out[0], out[2], out[1]);
  return GBATTN_OK;
}

extern "C" int attn_debug_scores(const void *q, const void *k, float *s, int B, int H, int L, int d, float scale,
                                 void *stream) {
  if (!q || !k || !s) return GBATTN_ERR_NULL;
  int rc = check_shape(B, H, L, d);
  if (rc != GBATTN_OK) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(s)) return GBATTN_ERR_ALIGN;
  if (!std::isfinite(scale)) return GBATTN_ERR_SCALE;
  const long long BH = static_cast<long long>(B) * H;
  const long long nQ = (L + 127) / 128;
  if (BH > 65535 || nQ * nQ > INT_MAX) return GBATTN_ERR_DIMS;
  const size_t tbytes = static_cast<size_t>(BH) * L * d * 2u;
  const size_t sbytes = static_cast<size_t>(BH) * L * L * 4u;
  if (overlaps(s, sbytes, q, tbytes) || overlaps(s, sbytes, k, tbytes)) return GBATTN_ERR_ALIAS;
  DevInfo *di = nullptr;
  if ((rc = device_info(&di)) != GBATTN_OK) return rc;
  CUtensorMap tq, tk;
  if (encode_bhld(&tq, q, static_cast<int>(BH), L, d) || encode_bhld(&tk, k, static_cast<int>(BH), L, d))
    return GBATTN_ERR_TENSORMAP;
  const cudaError_t e = launch_debug_scores(d, tq, tk, s, static_cast<int>(BH), L, scale, di->status,
                                            kWaitLimitCycles, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GBATTN_OK : GBATTN_ERR_LAUNCH;
}

extern "C" int attn_debug_wait_probe(long long limit_cycles, void *stream) {
  DevInfo *di = nullptr;
  const int rc = device_info(&di);
  if (rc != GBATTN_OK) return rc;
  long long lim = limit_cycles < 1000 ? 1000 : limit_cycles;
  if (lim > 100000000LL) lim = 100000000LL;
  return launch_wait_probe(di->status, lim, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GBATTN_OK
                                                                                               : GBATTN_ERR_LAUNCH;
}

extern "C" int attn_last_device_error(void) {
  DevInfo *di = nullptr;
  const int rc = device_info(&di);
  if (rc != GBATTN_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return GBATTN_ERR_LAUNCH;
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) return GBATTN_ERR_LAUNCH;
  if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return GBATTN_ERR_LAUNCH;
  return static_cast<int>(v);
}

extern "C" const char *attn_strerror(int code) {
  switch (code) {
    case GBATTN_OK: return "success";
    case GBATTN_ERR_NULL: return "a required pointer is NULL";
    case GBATTN_ERR_DIMS: return "bad dimensions (B, H, L must be > 0 and B*H*L must fit in int32)";
    case GBATTN_ERR_HEAD_DIM: return "unsupported head_dim (64, 128, 256 or 512; shared-memory P only for <= 128)";
    case GBATTN_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case GBATTN_ERR_LAUNCH: return "a CUDA call or the kernel launch failed";
    case GBATTN_ERR_DEVICE: return "the current device is not compute capability 10.3 (sm_103)";
    case GBATTN_ERR_SCALE: return "scale must be finite and > 0";
    case GBATTN_ERR_ALIAS: return "an output overlaps an input or the other output";
    case GBATTN_ERR_TENSORMAP: return "the driver rejected a TMA tensor-map descriptor";
    case GBATTN_ERR_FLAGS: return "flags holds bits that name no option";
    case GBATTN_ERR_WORKSPACE: return "the device workspace is smaller than attn_fwd_host_workspace_size()";
    case GBATTN_ERR_SCRATCH: return "the shape needs more workspace than attn_bwd_noalloc's fixed buffer holds";
    case GBATTN_DEV_TIMEOUT_LOAD: return "device: the TMA producer's wait timed out";
    case GBATTN_DEV_TIMEOUT_MMA: return "device: the MMA issuer's wait timed out";
    case GBATTN_DEV_TIMEOUT_SOFTMAX: return "device: a softmax warp's wait timed out";
    case GBATTN_DEV_TIMEOUT_EPILOGUE: return "device: the epilogue's wait timed out";
    case GBATTN_DEV_TIMEOUT_PROBE: return "device: the wait-probe barrier timed out (expected)";
    case GBATTN_DEV_TIMEOUT_MERGE: return "device: decode's wait for the other CTAs' partial results timed out";
    case GBATTN_DEV_SMEM_ALIGN: return "device: the backward kernel's shared memory was not 1 KB aligned; it did nothing";
    default: return "unknown gbattn status code";
  }
}

extern "C" int attn_debug_schedule(int B, int H, int L, int d, int causal, int grid, int flags, int *start,
                                   int *items, int max_items) {
  int rc = check_shape(B, H, L, d);
  if (rc != GBATTN_OK) return rc;
  if (grid <= 0 || grid > kSchedMaxCtas) return GBATTN_ERR_DIMS;
  if (!start || !items) return GBATTN_ERR_NULL;
  // The schedule of the kernel the flags name (no flag, d <= 128: the two-tile kernel;
  // the head_dim split's `grid` lanes are clusters of two CTAs; the automatic choice of
  // attn_fwd is not applied here).
  if ((rc = check_flags(flags, d)) != GBATTN_OK) return rc;
  const int kind = (flags & GBATTN_FLAG_DSPLIT)     ? kDSplit
                   : (flags & GBATTN_FLAG_SPLIT_KV) ? kSplitKV
                   : ((flags & (GBATTN_FLAG_P_SMEM | GBATTN_FLAG_SINGLE_TILE)) || d > 128) ? kSingle
                                                                                           : kPair;
  if (kind == kSplitKV && grid % 2) return GBATTN_ERR_DIMS;
  SchedKey key{kind, B * H, (L + 127) / 128, (L + 255) / 256,
               (kind == kSingle || kind == kSplitKV) && d > 256 ? d / 256 : 1, causal != 0 ? 1 : 0, grid,
               shortest_first_rule(kind, (L + 255) / 256, d)};
  if (count_items(key) > INT_MAX) return GBATTN_ERR_DIMS;
  static SchedTable t;  // large; this is a test hook, not thread-safe
  get_schedule(key, &t);
  if (t.n == 0) return 0;
  if (t.n > max_items) return GBATTN_ERR_DIMS;
  for (int c = 0; c <= grid; ++c) start[c] = t.start[c];
  for (int i = 0; i < t.n; ++i) items[i] = t.items[i];
  return t.n;
}

extern "C" int attn_debug_plan(int B, int H, int L, int d, int causal, int sm_count, int flags, int grid_limit,
                               int *out) {
  if (!out) return GBATTN_ERR_NULL;
  int rc = check_shape(B, H, L, d);
  if (rc != GBATTN_OK) return rc;
  if (sm_count <= 0 || sm_count > kSchedMaxCtas || grid_limit < 0) return GBATTN_ERR_DIMS;
  if ((rc = check_flags(flags, d)) != GBATTN_OK) return rc;
  SchedKey key;
  double makespan = 0.0;
  if ((rc = choose_plan(B * H, L, d, causal, sm_count, flags, grid_limit, key, makespan, sm_count & ~1)) !=
      GBATTN_OK)
    return rc;
  out[0] = key.kind;
  out[1] = static_cast<int>(count_items(key));
  out[2] = key.grid;
  out[3] = static_cast<int>(makespan * 100.0);
  return GBATTN_OK;
}

extern "C" int attn_version(void) { return 10100; }
