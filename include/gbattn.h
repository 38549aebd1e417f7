/*
 * gbattn.h -- C ABI of libgbattn.so: exact scaled-dot-product attention forward on one
 * GB300 (sm_103a), FP16 inputs, FP32 accumulation, FP16 output plus FP32 row LSE.
 *
 * The operation ("An Optimal Mapper Meets a Real GPU", sections "Ground rules" and
 * "Experiment one", Cases table; STAGE_D.md of nvfp4-megamoe-kernel, sections 2, 4
 * and 6):
 *     O[b,h,i,:] = sum_j softmax_j(scale * q_i . k_j + mask_ij) * v[b,h,j,:]
 *     LSE[b,h,i] = log sum_j exp(scale * q_i . k_j + mask_ij)       (natural log)
 * with query length = key/value length = L, mask_ij = -inf for j > i when causal, else 0.
 * The QK reduction over head_dim d is summed in full (in logit space) before the
 * softmax, also when d is wider than one 256-wide sub-tile.
 *
 * Conventions shared by every entry point:
 *   - Tensors are contiguous row-major [B, H, L, d] (PyTorch SDPA layout); q, k, v, o
 *     hold IEEE fp16 values, lse holds fp32 [B, H, L].
 *   - Every pointer is a DEVICE pointer owned by the caller (for example memory that
 *     PyTorch allocated).  No entry point allocates or frees device memory, and none
 *     synchronises (attn_last_device_error excepted); the library caches only host-side
 *     schedules, per-device attributes and the host-buffer pipeline's streams.  The one
 *     piece of device memory the library itself holds is attn_bwd_noalloc's fixed
 *     16 MiB buffer (plus a 4-byte status word): a file-scope __device__ array, so every
 *     GPU that loads the library holds it until the process exits, also in processes
 *     that never call attn_bwd_noalloc.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Work is enqueued asynchronously on it; on return the outputs are not yet written.
 *   - Return value: 0 if the work was enqueued, otherwise one of the negative
 *     GBATTN_ERR_* codes below; on an error nothing is enqueued and no output is touched.
 *   - Outputs must not overlap inputs or each other.
 *   - Not thread-safe for concurrent first calls on a new device (the per-device setup
 *     is done once); later calls from several host threads are safe.
 */
#ifndef GBATTN_H
#define GBATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GBATTN_OK 0
#define GBATTN_ERR_NULL (-1)        /* a required pointer is NULL                            */
#define GBATTN_ERR_DIMS (-2)        /* B, H or L <= 0, or B*H*L*d too large                  */
#define GBATTN_ERR_HEAD_DIM (-3)    /* d not in {64, 128, 256, 512}                          */
#define GBATTN_ERR_ALIGN (-4)       /* a pointer is not 16-byte aligned                      */
#define GBATTN_ERR_LAUNCH (-5)      /* a CUDA call or the kernel launch failed               */
#define GBATTN_ERR_DEVICE (-6)      /* the current device is not compute capability 10.3     */
#define GBATTN_ERR_SCALE (-7)       /* scale is not a finite number > 0                      */
#define GBATTN_ERR_ALIAS (-8)       /* an output overlaps an input or the other output       */
#define GBATTN_ERR_TENSORMAP (-9)   /* the driver rejected a TMA descriptor                  */
#define GBATTN_ERR_FLAGS (-10)      /* attn_fwd_ex: unknown bits in flags                    */
#define GBATTN_ERR_WORKSPACE (-11)  /* attn_fwd_host: device workspace too small             */
#define GBATTN_ERR_SCRATCH (-12)    /* attn_bwd_noalloc: shape needs more than its fixed buffer */

/* Device-side status codes reported by attn_last_device_error() (positive). */
#define GBATTN_DEV_TIMEOUT_LOAD 1    /* the TMA producer's wait for a free buffer timed out  */
#define GBATTN_DEV_TIMEOUT_MMA 2     /* the MMA issuer's wait for data or P timed out        */
#define GBATTN_DEV_TIMEOUT_SOFTMAX 3 /* the softmax warps' wait for S or O timed out         */
#define GBATTN_DEV_TIMEOUT_EPILOGUE 4 /* the epilogue's wait for its staging tile timed out   */
#define GBATTN_DEV_TIMEOUT_PROBE 5   /* the self-test wait of attn_debug_wait_probe ran out */
#define GBATTN_DEV_TIMEOUT_MERGE 6   /* attn_decode: waiting for the other CTAs' partials ran out */
#define GBATTN_DEV_SMEM_ALIGN 7      /* attn_bwd: dynamic shared memory not 1 KB aligned (kernel skipped) */

/*
 * attn_fwd -- the fused forward pass.
 *   q, k, v : const fp16 [B, H, L, d], device, 16-byte aligned.
 *   o       : fp16 [B, H, L, d] output, device, 16-byte aligned.
 *   lse     : fp32 [B, H, L] output (natural-log LSE of the scaled, masked logits).
 *   B, H, L : > 0.  d : 64, 128, 256 or 512.  causal : 0 or 1 (nonzero = 1).
 *   scale   : the logit scale (usually 1/sqrt(d)), finite and > 0.
 * Rounding: O is rounded to fp16 to nearest even; P (the softmax weights) is rounded to
 * fp16 before the PV product, as the FP16-in/FP32-accumulate convention implies.
 * A wait inside the kernel that exceeds about two seconds (a fault, never expected)
 * ends the kernel early with a code readable through attn_last_device_error().
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
             int L, int d, int causal, float scale, void *stream);

/*
 * attn_fwd_ex -- attn_fwd with design options (same arguments, same errors, plus
 * GBATTN_ERR_FLAGS for unknown or conflicting flag bits).  Two kernels exist:
 *   two-tile kernel (d <= 128 only): each work item is a 256-row query block whose two
 *     128-row halves share every K/V tile and have their own softmax warpgroup;
 *   single-tile kernel (every d): each work item is one 128-row query tile.
 * With flags = 0: d > 128 uses the single-tile kernel; d <= 128 the two-tile kernel when
 * it has at least two items per SM, else whichever of the two kernels has the shorter
 * estimated schedule; for d = 64, 128 and 512 the single-tile kernel with key-range splits
 * (bit 4) replaces that choice when its estimated schedule is clearly shorter (query
 * tiles with many more key tiles than the average CTA's load).  Options:
 *   flags bit 0 (GBATTN_FLAG_P_SMEM): single-tile kernel, with P staged through shared
 *     memory instead of tensor memory before the PV product (the SMEM-P path of the
 *     STAGE_D.md notes, section 4); only for d <= 128, otherwise GBATTN_ERR_HEAD_DIM.
 *   flags bit 1 (GBATTN_FLAG_SINGLE_TILE): single-tile kernel, P in tensor memory.
 *   flags bit 2 (GBATTN_FLAG_TWO_TILE): two-tile kernel whatever the item count; only for
 *     d <= 128 (else GBATTN_ERR_HEAD_DIM) and not with bits 0 or 1 (GBATTN_ERR_FLAGS).
 *   flags bit 3 (GBATTN_FLAG_DSPLIT): the single-tile kernel with head_dim split over the
 *     two CTAs of a thread-block cluster: each CTA computes the logits over half of
 *     head_dim, the two exchange their partial S tiles through distributed shared memory,
 *     and each produces half of O, so no QK product is computed twice (without it each of
 *     the two value halves of a d = 512 tile recomputes the full QK product).  Only for
 *     d = 512 (else GBATTN_ERR_HEAD_DIM) and alone (else GBATTN_ERR_FLAGS).  Slower on
 *     GB300: moving a 64 KB partial S tile between SMs takes longer than the QK work it
 *     saves.
 *   flags bit 4 (GBATTN_FLAG_SPLIT_KV): the single-tile kernel on clusters of two CTAs,
 *     where the longest query tiles are split into two disjoint key ranges, each at least
 *     3 key tiles (384 keys), one per CTA of a cluster; the second CTA hands its partial
 *     O (normalised, fp16) and each row's running maximum and sum to the first through
 *     shared memory (one bulk copy per 64 columns), and the first merges the two with the
 *     log-sum-exp weights (exact for disjoint key ranges: "An Optimal Mapper Meets a Real
 *     GPU", "Experiment one", and STAGE_D.md, section 2, "Merge") and writes O and LSE.
 *     Query tiles whose split would leave a part shorter than 3 key tiles are not split.
 *     Only for d = 64, 128, 512 (else GBATTN_ERR_HEAD_DIM) and alone (else
 *     GBATTN_ERR_FLAGS); the launch uses an even number of CTAs (at least 2).
 *   grid_limit: 0 = one persistent CTA per SM; n > 0 = at most n CTAs (scheduler tests).
 * Every option gives the same results up to rounding.
 */
#define GBATTN_FLAG_P_SMEM 1
#define GBATTN_FLAG_SINGLE_TILE 2
#define GBATTN_FLAG_TWO_TILE 4
#define GBATTN_FLAG_DSPLIT 8
#define GBATTN_FLAG_SPLIT_KV 16
int attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                int H, int L, int d, int causal, float scale, void *stream, int flags,
                int grid_limit);

/*
 * attn_fwd_host -- attn_fwd on inputs and outputs in HOST memory, for callers whose
 * tensors are not on the GPU.  Same operation, arguments and errors as attn_fwd, except:
 *   q, k, v, o, lse : HOST pointers (page-locked memory -- e.g. cudaHostAlloc or
 *                     PyTorch pin_memory -- for the copies to overlap; other host
 *                     memory works, the driver then stages the copies), any alignment.
 *   workspace       : DEVICE memory of at least attn_fwd_host_workspace_size(B, H, L, d)
 *                     bytes, 256-byte aligned (else GBATTN_ERR_ALIGN), owned by the caller;
 *                     too small: GBATTN_ERR_WORKSPACE.  Launches that share a workspace
 *                     must not overlap on the GPU (give them one stream).
 * The heads are cut into chunks of about 12 MB of Q+K+V; chunk by chunk, the library's
 * own streams copy Q, K, V in, run the forward pass, and copy O and LSE out, through two
 * alternating halves of the workspace, so that the copies in, the kernels and the copies
 * out of different chunks overlap (the host link is the bound: ~0.2 TB/s each way on
 * GB300).  The work starts after what is already queued on `stream`, and `stream` waits
 * for its end: synchronise `stream` before reading o and lse.  The streams and events are
 * created on the first call per device and kept; calls from several host threads are
 * serialised.
 */
int attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                  int L, int d, int causal, float scale, void *workspace, size_t workspace_bytes,
                  void *stream);

/* Device workspace bytes attn_fwd_host needs for this shape (0 for invalid arguments). */
size_t attn_fwd_host_workspace_size(int B, int H, int L, int d);

/*
 * attn_bwd -- the backward pass: gradients of O = SDPA(q, k, v) (as attn_fwd computes it)
 * for an upstream gradient dout ("Validating Memory-Optimal Transformer Kernels on Real
 * Hardware", section 4, "Paper II: Backward Pass and Fused Forward+Backward"):
 *     P = softmax(scale * q k^T + mask),  D_i = dout_i . o_i,
 *     dv = P^T dout,  dS = P * (dout v^T - D),  dq = scale dS k,  dk = scale dS^T q.
 *   q, k, v, o, dout : const fp16 [B, H, L, d], device, 16-byte aligned (o: attn_fwd's output).
 *   lse              : const fp32 [B, H, L] (attn_fwd's LSE output).
 *   dq, dk, dv       : fp16 [B, H, L, d] outputs, device, 16-byte aligned, overlapping no
 *                      input and no other output (else GBATTN_ERR_ALIAS).
 *   workspace        : device memory of attn_bwd_workspace_bytes(B, H, L) bytes, 16-byte
 *                      aligned, overlapping no input and no output (GBATTN_ERR_NULL,
 *                      GBATTN_ERR_ALIGN, GBATTN_ERR_ALIAS); owned by the caller, its
 *                      contents on entry do not matter and are overwritten.
 *   d : 64 or 128 (else GBATTN_ERR_HEAD_DIM).  causal, scale, stream, errors: as attn_fwd.
 * Two persistent kernels without atomics, enqueued on `stream`: the first computes dq one
 * 128-row query tile at a time and writes each query row's statistics LSE log2(e) and
 * D_i to the workspace (8 bytes per row); the second computes dk and dv one 128-row key
 * tile at a time, streaming the query rows with those statistics.  P is recomputed from
 * lse; nothing is allocated or kept.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
             void *dq, void *dk, void *dv, void *workspace, int B, int H, int L, int d, int causal, float scale,
             void *stream);

/*
 * attn_bwd_workspace_bytes -- bytes of workspace attn_bwd needs for B x H heads of L rows:
 * 8 * B * H * Lp with Lp = L rounded up to a multiple of 128.  Host-only; returns a
 * negative GBATTN_ERR_DIMS when B, H or L is not positive or the shape is too large.
 */
long long attn_bwd_workspace_bytes(int B, int H, int L);

/*
 * attn_bwd_noalloc -- attn_bwd for callers that cannot allocate device memory (a plug-in
 * inside a host application that owns every device allocation, or a latency-critical
 * path where cudaMalloc, which may synchronise the device, is not allowed).  The paper
 * has no counterpart: this is a deployment variant, not part of the method.
 *   Same arguments, results and errors as attn_bwd, without `workspace`: the workspace is
 *   a fixed buffer of attn_bwd_noalloc_max_bytes() = 16 MiB compiled into the library
 *   (every GPU that loads it holds the buffer until the process exits).  Shapes whose
 *   attn_bwd_workspace_bytes(B, H, L) exceeds it (more than 2,097,152 query rows after
 *   padding L to a multiple of 128) return GBATTN_ERR_SCRATCH before anything is enqueued.
 *   No device memory is allocated or freed.
 *   Arguments are checked first, in attn_bwd's order (so the same errors come back for
 *   the same mistakes), then the size, and only then is any CUDA call made.
 *   The first call on each device looks up the buffer's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make that first call
 *   before any stream capture.  The cached address does not survive cudaDeviceReset: do
 *   not call this entry point on a device after resetting it in the same process.  All calls on a device share the one buffer: calls that can run at the
 *   same time on the GPU (on streams not ordered against each other) race and must be
 *   serialised by the caller.  Nothing in the buffer needs to start at zero.
 */
int attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse,
                     const void *dout, void *dq, void *dk, void *dv, int B, int H, int L, int d, int causal,
                     float scale, void *stream);

/* attn_bwd_noalloc_max_bytes -- the size in bytes of attn_bwd_noalloc's fixed buffer. */
long long attn_bwd_noalloc_max_bytes(void);

/*
 * attn_decode -- decoding: one query row per (b, h) against all L cached keys, every key
 * visible ("Validating Memory-Optimal Transformer Kernels on Real Hardware", section 5,
 * "Paper III: Inference (Decode)"):
 *     o[b,h,:] = sum_j softmax_j(scale * q[b,h] . k[b,h,j]) v[b,h,j,:]
 *     lse[b,h] = log sum_j exp(scale * q[b,h] . k[b,h,j])                (natural log)
 *   q         : const fp16 [B, H, d] (the [B, H, 1, d] query), device, 16-byte aligned.
 *   k, v      : const fp16 [B, H, L, d], device, 16-byte aligned.
 *   o         : fp16 [B, H, d] output;  lse : fp32 [B, H] output.
 *   workspace : NULL, or device memory of attn_decode_workspace_bytes(B, H, d) bytes,
 *               16-byte aligned, overlapping no input or output; owned by the caller, its
 *               contents on entry do not matter.
 *   B, H, L : > 0.  d : 64, 128, 256 or 512.  scale : finite and > 0.
 * Ownership, stream, return values and errors as for attn_fwd.  Each head's keys are
 * split over the CTAs of one thread-block cluster (a power of two, up to 16: the widest
 * that keeps the launch within one wave of two CTAs per SM, so one CTA per head once the
 * heads alone fill it), which merge their partial results in distributed shared memory.
 * When no such cluster fills that wave (fewer than about 40 heads) and a workspace is
 * given, each head's keys are instead split over several clusters (of two CTAs, or of up
 * to 8 when a head would need more than 32 clusters), each cluster writes its normalised
 * partial (o, lse) to the workspace, and a second small kernel merges them.  Without a
 * workspace the launch keeps one cluster per head.  The work is bound by the HBM reads of
 * K and V.
 */
int attn_decode(const void *q, const void *k, const void *v, void *o, float *lse, void *workspace, int B, int H,
                int L, int d, float scale, void *stream);

/*
 * attn_decode_workspace_bytes -- bytes of the optional attn_decode workspace for B x H heads
 * at head_dim d: B * H * 32 * (d + 2) * 4 (at most 32 clusters per head).  Host-only;
 * negative GBATTN_ERR_DIMS or GBATTN_ERR_HEAD_DIM on bad arguments.
 */
long long attn_decode_workspace_bytes(int B, int H, int d);

/*
 * attn_debug_decode_plan -- test hook (host-only): the split attn_decode uses for this
 * shape on a GPU with `sm_count` SMs whose clusters hold at most `max_ranks` CTAs (1..16),
 * with a workspace (`grouped` != 0) or without: out[0] = CTAs per cluster (a power of
 * two; at most 16, 8, 4 for d <= 128, 256, 512), out[1] = keys per CTA (whole key tiles
 * of 8192 / d keys), out[2] = clusters per head (1 without a workspace; at most 32).
 * Returns 0 or a negative GBATTN_ERR_* code.
 */
int attn_debug_decode_plan(int B, int H, int L, int d, int sm_count, int max_ranks, int grouped, int *out);

/*
 * attn_debug_scores -- test hook: the raw scaled logits s[b,h,i,j] = scale * q_i . k_j
 * (fp32 [B, H, L, L], no mask), with the head_dim reduction done the same way as in
 * attn_fwd (tensor-core products accumulated over every 64-wide slice of d before any
 * read-out).  It exists to check the QK stage alone ("no-softmax mode", STAGE_D.md,
 * option 2 of the closing list).  Not a production path.
 */
int attn_debug_scores(const void *q, const void *k, float *s, int B, int H, int L, int d,
                      float scale, void *stream);

/*
 * attn_last_device_error -- read and clear the device status word of the current
 * device.  Returns 0 if every kernel since the last call finished normally, otherwise
 * the first GBATTN_DEV_* code recorded.  Synchronises the current device first (it is
 * a host-blocking call); returns GBATTN_ERR_LAUNCH if that fails.
 */
int attn_last_device_error(void);

/*
 * attn_debug_wait_probe -- self-test of the bounded waits: launches one tiny kernel
 * that waits on a shared-memory barrier that nothing completes, giving up after
 * `limit_cycles` SM clock cycles (clamped to [1000, 100000000]) and recording
 * GBATTN_DEV_TIMEOUT_PROBE.  Lets a test check, without hanging the GPU, that a wait
 * that runs out turns into a status the host can read.
 */
int attn_debug_wait_probe(long long limit_cycles, void *stream);

/*
 * attn_debug_schedule -- test hook: the static work schedule attn_fwd_ex would use for
 * this shape, `grid` CTAs (clusters of two CTAs with GBATTN_FLAG_DSPLIT) and `flags`.
 * With GBATTN_FLAG_SPLIT_KV (`grid` even: CTAs 2c and 2c + 1 form cluster c) a value
 * v >= (number of query tiles x value-column halves) in items[] names a split query tile
 * (the tile of item v - that number), listed by both CTAs of a cluster, first, in the
 * same order; the table then has one entry per CTA for each split tile.
 * Returns the number of entries n and fills
 * start[0..grid] (CTA c runs items[start[c] .. start[c+1]) in order) and items[0..n), or
 * returns 0 when the kernels take no table and use their fixed snake order: the problem
 * is too large for a table, or (single-tile and two-tile kernels) no CTA has more than one
 * item, where that order is the schedule; or a negative GBATTN_ERR_* code
 * (GBATTN_ERR_DIMS if n > max_items).
 * Host-only; needs no GPU.  Not thread-safe.
 */
int attn_debug_schedule(int B, int H, int L, int d, int causal, int grid, int flags, int *start, int *items,
                        int max_items);

/*
 * attn_debug_plan -- test hook: the kernel attn_fwd_ex would launch for this shape,
 * `flags` and `grid_limit` on a GPU with `sm_count` SMs (host-only; needs no GPU).
 * Fills out[0] = kernel (0 single-tile, 1 two-tile, 2 single-tile with the head_dim split,
 * 3 single-tile with key-range splits), out[1] = work items (query tiles x value-column
 * halves, before any split), out[2] = CTAs (clusters of two CTAs for kernel 2, CTAs in
 * clusters of two for kernel 3),
 * out[3] = estimated makespan x 100 (in units of one tile step of a query tile in the
 * two-tile kernel; -100 when the kernels use their fixed order).
 * Returns 0 or a negative GBATTN_ERR_* code.
 */
int attn_debug_plan(int B, int H, int L, int d, int causal, int sm_count, int flags, int grid_limit,
                    int *out);

/* Human-readable text for a GBATTN_ERR_* or GBATTN_DEV_* code (static storage). */
const char *attn_strerror(int code);

/* Library version as major*10000 + minor*100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GBATTN_H */
