"""GB300-native (sm_103a) exact scaled-dot-product attention forward.

O = softmax(scale * Q K^T + causal mask) V with FP16 inputs, FP32 accumulation, FP16 O
and FP32 row log-sum-exp, computed by one fused persistent CUDA kernel (TMA, tcgen05
tensor cores, tensor memory) behind the C ABI of include/gbattn.h; and decoding (one
query row per head against a long cached key/value sequence, attn_decode) by a
cluster-split streaming kernel.  This package is the
thin Python binding of that library; every step of the computation runs on the GPU.
"""
from ._binding import (FLAG_DSPLIT, FLAG_P_SMEM, FLAG_SINGLE_TILE, FLAG_SPLIT_KV, FLAG_TWO_TILE, LIB_PATH, GbattnError, attn_debug_decode_plan,
                       attn_bwd, attn_bwd_workspace_bytes, attn_debug_plan, attn_debug_schedule, attn_debug_scores, attn_debug_wait_probe, attn_decode,
                       attn_fwd, attn_fwd_host, attn_last_device_error, attn_strerror, attn_version, load_library)

__all__ = ["attn_fwd", "attn_fwd_host", "attn_bwd", "attn_bwd_workspace_bytes", "attn_decode", "attn_debug_plan", "attn_debug_decode_plan",
           "attn_debug_scores", "attn_debug_schedule", "attn_debug_wait_probe",
           "attn_last_device_error", "attn_strerror", "attn_version", "load_library", "GbattnError", "FLAG_P_SMEM",
           "FLAG_SINGLE_TILE", "FLAG_TWO_TILE", "FLAG_DSPLIT", "FLAG_SPLIT_KV", "LIB_PATH"]
