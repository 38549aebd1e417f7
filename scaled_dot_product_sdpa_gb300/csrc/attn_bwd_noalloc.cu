// attn_bwd_noalloc -- the backward pass for callers that cannot allocate device memory.
//
// attn_bwd needs a small device workspace (8 bytes per query row) that its caller
// allocates.  Some callers cannot do that: a plug-in running inside a host application
// that owns every device allocation, or a latency-critical path where cudaMalloc (which
// may synchronise the device) is not allowed.  This entry point runs the same two kernels
// with the workspace taken from one fixed buffer compiled into the library: a file-scope
// __device__ array of kBwdScratchBytes bytes, which every GPU that loads the library holds
// until the process exits.  Nothing here calls cudaMalloc, cudaFree or any allocating
// routine.
//
// In host code the array's name only stands for the device symbol; its device address is
// looked up with cudaGetSymbolAddress on the first call on each device (with that device
// current) and cached per device.  The cache does not survive cudaDeviceReset (the
// buffer gets a new address in the new context): a process that resets a device must not
// call this entry point on it afterwards.  Every call on a device shares the one buffer: calls
// whose kernels can run at the same time on the GPU (streams not ordered against each
// other) race on it and must be serialised by the caller.  The buffer keeps the last
// call's contents, and nothing in it needs to start at zero: the first kernel writes every
// workspace row the second kernel reads.
#include <cuda_runtime.h>

#include <mutex>

#include "gbattn.h"

namespace {

constexpr long long kBwdScratchBytes = 16ll << 20;  // 16 MiB: 2,097,152 padded query rows

static __device__ __align__(256) unsigned char g_bwd_scratch[kBwdScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch buffer on the current device (looked up once per device).
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GBATTN_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return GBATTN_ERR_LAUNCH;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GBATTN_OK;
}

}  // namespace

namespace gbattn {
int bwd_check_args(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
                   const void *dq, const void *dk, const void *dv, const void *workspace, bool check_workspace, int B,
                   int H, int L, int d, float scale);  // gbattn_abi.cu
}

extern "C" long long attn_bwd_noalloc_max_bytes(void) { return kBwdScratchBytes; }

extern "C" int attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse,
                                const void *dout, void *dq, void *dk, void *dv, int B, int H, int L, int d,
                                int causal, float scale, void *stream) {
  // attn_bwd's own checks first (no CUDA call), so that errors come in its order; then
  // the buffer's size; only then the address lookup.
  int rc = gbattn::bwd_check_args(q, k, v, o, lse, dout, dq, dk, dv, nullptr, false, B, H, L, d, scale);
  if (rc != GBATTN_OK) return rc;
  if (attn_bwd_workspace_bytes(B, H, L) > kBwdScratchBytes) return GBATTN_ERR_SCRATCH;
  void *ws = nullptr;
  if ((rc = scratch_address(&ws)) != GBATTN_OK) return rc;
  return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, ws, B, H, L, d, causal, scale, stream);
}
