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
// swizzle span) x 128 rows x 1 head.  Rows past L read as zero and are never written.
int encode_bhld(CUtensorMap *tm, const void *ptr, int BH, int L, int D) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2u,
                                 static_cast<cuuint64_t>(L) * static_cast<cuuint64_t>(D) * 2u};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
                              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GBATTN_OK : GBATTN_ERR_TENSORMAP;
}

// ------------------------------------------------------------------ work schedule
// Cost of a work item in 128 x 128 tile units plus a per-item overhead (fill, drain and
// epilogue of the item's pipeline), the latter measured on GB300 for each kernel.
constexpr double kItemOverheadTwoTile = 1.7;
constexpr double kItemOverheadSingle = 1.0;

struct SchedKey {
  int two_tile, BH, nQ, nQB, dvs, causal, grid;
  bool operator==(const SchedKey &o) const {
    return two_tile == o.two_tile && BH == o.BH && nQ == o.nQ && nQB == o.nQB && dvs == o.dvs &&
           causal == o.causal && grid == o.grid;
  }
};

// Work units of item r, mirroring the kernels' item decoding (pp_decode / decode_item).
int item_units(const SchedKey &k, int r) {
  if (k.two_tile) {
    if (!k.causal) return 2 * k.nQ;
    const int qb = k.nQB - 1 - r / k.BH;
    return (2 * qb + 1) + std::min(2 * qb + 2, k.nQ);
  }
  if (!k.causal) return k.nQ;
  const int qt = k.nQ - 1 - r / (k.BH * k.dvs);
  return qt + 1;
}

// Longest-processing-time-first: take items by decreasing cost, give each to the CTA with
// the least accumulated cost (ties: lowest CTA).  Each CTA's list keeps assignment order.
void build_lpt(const SchedKey &k, int n_items, SchedTable &t) {
  std::memset(&t, 0, sizeof(t));
  if (n_items > kSchedMaxItems || k.grid > kSchedMaxCtas || k.grid <= 0) return;  // snake order
  const double over = k.two_tile ? kItemOverheadTwoTile : kItemOverheadSingle;
  std::vector<int> order(n_items);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return item_units(k, a) > item_units(k, b); });
  using Slot = std::pair<double, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int c = 0; c < k.grid; ++c) heap.push({0.0, c});
  std::vector<std::vector<uint16_t>> lists(k.grid);
  for (int r : order) {
    const Slot s = heap.top();
    heap.pop();
    lists[s.second].push_back(static_cast<uint16_t>(r));
    heap.push({s.first + item_units(k, r) + over, s.second});
  }
  int pos = 0;
  for (int c = 0; c < k.grid; ++c) {
    t.start[c] = static_cast<uint16_t>(pos);
    for (uint16_t r : lists[c]) t.items[pos++] = r;
  }
  t.start[k.grid] = static_cast<uint16_t>(pos);
  t.n = n_items;
}

struct SchedEntry {
  bool valid = false;
  unsigned long long stamp = 0;
  SchedKey key{};
  SchedTable tbl;
};
SchedEntry g_sched_cache[8];
unsigned long long g_sched_clock = 0;
std::mutex g_sched_mu;

// Copy the schedule for `k` into `out`, building and caching it on a miss.
void get_schedule(const SchedKey &k, int n_items, SchedTable &out) {
  std::lock_guard<std::mutex> lock(g_sched_mu);
  SchedEntry *victim = &g_sched_cache[0];
  for (SchedEntry &e : g_sched_cache) {
    if (e.valid && e.key == k) {
      e.stamp = ++g_sched_clock;
      out = e.tbl;
      return;
    }
    if (!e.valid || e.stamp < victim->stamp) victim = &e;
  }
  build_lpt(k, n_items, victim->tbl);
  victim->key = k;
  victim->valid = true;
  victim->stamp = ++g_sched_clock;
  out = victim->tbl;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int B, int H, int L, int d) {
  if (B <= 0 || H <= 0 || L <= 0) return GBATTN_ERR_DIMS;
  const long long rows = static_cast<long long>(B) * H * L;
  if (rows > INT_MAX || static_cast<long long>(B) * H > INT_MAX) return GBATTN_ERR_DIMS;
  if (d != 64 && d != 128 && d != 256 && d != 512) return GBATTN_ERR_HEAD_DIM;
  return GBATTN_OK;
}

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
  if (p_smem && d > 128) return GBATTN_ERR_HEAD_DIM;
  if (flags & ~(GBATTN_FLAG_P_SMEM | GBATTN_FLAG_SINGLE_TILE | GBATTN_FLAG_TWO_TILE)) return GBATTN_ERR_FLAGS;
  if ((flags & GBATTN_FLAG_TWO_TILE) && (flags & (GBATTN_FLAG_SINGLE_TILE | GBATTN_FLAG_P_SMEM)))
    return GBATTN_ERR_FLAGS;
  if ((flags & GBATTN_FLAG_TWO_TILE) && d > 128) return GBATTN_ERR_HEAD_DIM;
  // d <= 128: the two-tile kernel (two 128-row query tiles per item) unless an option asks
  // for the single-tile kernel, or unless it would get fewer than two items per SM: then
  // the single-tile kernel's twice-as-many, half-as-long items balance the SMs better
  // (measured on GB300: 1x16x512x64 causal 7.7 vs 10.5 us, 1x32x1024x128 causal 15.0 vs
  // 19.2 us), while the two-tile kernel is faster once every SM has several items.
  bool two_tile = d <= 128 && !(flags & (GBATTN_FLAG_P_SMEM | GBATTN_FLAG_SINGLE_TILE));
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
  const int nQ = (L + 127) / 128;
  const int nQB = (L + 255) / 256;
  const int dvs = d > 256 ? d / 256 : 1;
  if (two_tile && !(flags & GBATTN_FLAG_TWO_TILE) && static_cast<long long>(BH) * nQB < 2LL * di->sm_count)
    two_tile = false;
  const long long n_items = two_tile ? static_cast<long long>(BH) * nQB : static_cast<long long>(BH) * nQ * dvs;
  if (n_items > INT_MAX) return GBATTN_ERR_DIMS;

  FwdLaunch a;
  SchedTable tbl;
  a.tbl = &tbl;
  if (encode_bhld(&a.tm_q, q, BH, L, d) || encode_bhld(&a.tm_k, k, BH, L, d) || encode_bhld(&a.tm_v, v, BH, L, d) ||
      encode_bhld(&a.tm_o, o, BH, L, d))
    return GBATTN_ERR_TENSORMAP;
  int grid = di->sm_count;
  if (grid_limit > 0 && grid_limit < grid) grid = grid_limit;
  if (n_items < grid) grid = static_cast<int>(n_items);
  a.grid = grid;
  get_schedule(SchedKey{two_tile ? 1 : 0, BH, nQ, nQB, two_tile ? 1 : dvs, causal != 0 ? 1 : 0, grid},
               static_cast<int>(n_items), tbl);
  a.causal = causal != 0;
  a.p_smem = p_smem;
  a.stream = static_cast<cudaStream_t>(stream);
  a.p.o = o;
  a.p.lse = lse;
  a.p.status = di->status;
  a.p.wait_limit = kWaitLimitCycles;
  a.p.BH = BH;
  a.p.L = L;
  a.p.nQ = nQ;
  a.p.nQB = nQB;
  a.p.n_items = static_cast<int>(n_items);
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
    case GBATTN_DEV_TIMEOUT_LOAD: return "device: the TMA producer's wait timed out";
    case GBATTN_DEV_TIMEOUT_MMA: return "device: the MMA issuer's wait timed out";
    case GBATTN_DEV_TIMEOUT_SOFTMAX: return "device: a softmax warp's wait timed out";
    case GBATTN_DEV_TIMEOUT_EPILOGUE: return "device: the epilogue's wait timed out";
    case GBATTN_DEV_TIMEOUT_PROBE: return "device: the wait-probe barrier timed out (expected)";
    default: return "unknown gbattn status code";
  }
}

extern "C" int attn_debug_schedule(int B, int H, int L, int d, int causal, int grid, int flags, int *start,
                                   int *items, int max_items) {
  int rc = check_shape(B, H, L, d);
  if (rc != GBATTN_OK) return rc;
  if (grid <= 0 || grid > kSchedMaxCtas) return GBATTN_ERR_DIMS;
  if (!start || !items) return GBATTN_ERR_NULL;
  // The schedule of the kernel the flags name: the two-tile kernel when d <= 128 and no
  // single-tile option is set (the automatic choice of attn_fwd is not applied here).
  const bool two_tile = d <= 128 && !(flags & (GBATTN_FLAG_P_SMEM | GBATTN_FLAG_SINGLE_TILE));
  const int BH = B * H, nQ = (L + 127) / 128, nQB = (L + 255) / 256, dvs = d > 256 ? d / 256 : 1;
  const long long n_items = two_tile ? static_cast<long long>(BH) * nQB : static_cast<long long>(BH) * nQ * dvs;
  if (n_items > INT_MAX) return GBATTN_ERR_DIMS;
  static SchedTable t;  // large; this is a test hook, not thread-safe
  get_schedule(SchedKey{two_tile ? 1 : 0, BH, nQ, nQB, two_tile ? 1 : dvs, causal != 0 ? 1 : 0, grid},
               static_cast<int>(n_items), t);
  if (t.n == 0) return 0;
  if (t.n > max_items) return GBATTN_ERR_DIMS;
  for (int c = 0; c <= grid; ++c) start[c] = t.start[c];
  for (int i = 0; i < t.n; ++i) items[i] = t.items[i];
  return t.n;
}

extern "C" int attn_version(void) { return 100; }
