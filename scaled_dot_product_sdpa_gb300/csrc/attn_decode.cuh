// attn_decode.cuh -- decode (one query row per head against a long key/value sequence)
// on sm_103a: parameters and launch entry points shared with the C ABI.
//
// What it computes ("Validating Memory-Optimal Transformer Kernels on Real Hardware",
// section 5, "Paper III: Inference (Decode)": one new token attends to the whole cached
// sequence, at a cost linear in its length):
//     o[bh, :] = sum_j softmax_j(scale * q[bh] . k[bh, j]) v[bh, j, :]   (every key j < L)
//     lse[bh]  = log sum_j exp(scale * q[bh] . k[bh, j])
// Each head's keys are split over the CTAs of one thread-block cluster (its "ranks"); every
// rank streams its key range once and the partial results are merged in the cluster's
// shared memory.  When a head's keys are also split over several clusters ("groups": few
// heads, so that one cluster per head would leave SMs idle), each cluster writes its
// merged, normalised partial (o_g, lse_g) to a workspace and a small merge kernel combines
// the groups: o = sum_g 2^(lse_g - M) o_g / sum_g 2^(lse_g - M), M = max_g lse_g.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace gbattn {

constexpr unsigned kDevTimeoutMerge = 6;  // rank 0's wait for the other ranks' partials
constexpr int kDecMaxRanks = 16;          // CTAs per cluster at most
constexpr int kDecMaxGroups = 32;         // clusters per head at most (workspace rows per head)
constexpr int kDecGroupedRanks = 8;      // CTAs per cluster when a head spans several clusters
// CTAs per head for head_dim d: rank 0 keeps every rank's partial o[d] in shared memory,
// and this bound keeps that buffer small enough for two CTAs per SM.
constexpr int dec_max_ranks_for(int d) { return d <= 128 ? 16 : d == 256 ? 8 : 4; }

struct DecParams {
  const void *q;           // [BH, D] fp16
  void *o;                 // [BH, D] fp16
  float *lse;              // [BH] fp32
  unsigned *status;        // device status word (first error code wins)
  long long wait_limit;    // SM clock cycles a single wait may take before it gives up
  int BH, L;               // heads, keys per head
  int ranks;               // CTAs per cluster
  int groups;              // clusters per head (> 1: partials go to ws, then the merge kernel)
  int keys_per_rank;       // a multiple of the key tile
  float *ws;               // [BH, groups, D + 2] fp32: o_g (normalised), lse_g (base 2), unused
  float c2;                // scale * log2(e)
};

struct DecLaunch {
  CUtensorMap tm_k, tm_v;  // [BH, L, D] viewed as 3-D, box 64 columns x key-tile rows
  DecParams p;
  cudaStream_t stream;
};

// Keys per tile for head_dim d (one tile of K is 16 KB).
constexpr int dec_key_tile(int d) { return 8192 / d; }

cudaError_t launch_decode_64(const DecLaunch &a);
cudaError_t launch_decode_128(const DecLaunch &a);
cudaError_t launch_decode_256(const DecLaunch &a);
cudaError_t launch_decode_512(const DecLaunch &a);
// Workspace bytes of a decode launch over BH heads at head_dim d (kDecMaxGroups rows per head).
constexpr long long dec_workspace_bytes(long long BH, int d) { return BH * kDecMaxGroups * (d + 2) * 4LL; }

// Largest cluster size the decode kernel for head_dim d can be launched with on the
// current device (16 if allowed, else 8); negative on a CUDA error.
int decode_max_ranks(int d);

}  // namespace gbattn
