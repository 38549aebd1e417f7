"""The five SDPA-forward workloads, their seeds and their algorithmic work.

Cases A-D are the four SDPA shapes of "An Optimal Mapper Meets a Real GPU",
"Experiment one" (Cases table): FP16 in, FP32 accumulate, query length = key/value
length.  The fifth is the head_dim-512 shape of the STAGE_D.md notes
(nvfp4-megamoe-kernel), section 6, whose QK reduction is wider than one 256-wide
sub-tile.  Inputs are i.i.d. N(0, sigma^2) cast to fp16 (sigma = 0.5 for head_dim 512),
drawn with seed = the workload's index.
"""
from __future__ import annotations

import math
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    d: int
    causal: bool
    seed: int
    sigma: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self) -> float:
        """Algorithmic FLOPs: 4*B*H*L^2*d, halved when causal (QK^T and PV each 2*L^2*d)."""
        f = 4.0 * self.B * self.H * self.L * self.L * self.d
        return f * 0.5 if self.causal else f

    def bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V once, write O (2 B each) and LSE (4 B/row)."""
        n = self.B * self.H * self.L
        return 2 * 4 * n * self.d + 4 * n

    def describe(self) -> str:
        return (f"B={self.B} H={self.H} L={self.L} d={self.d} "
                f"{'causal' if self.causal else 'non-causal'} seed={self.seed} sigma={self.sigma}")


WORKLOADS = {
    "caseA": Workload("caseA", 1, 8, 128, 64, False, 1),
    "caseB": Workload("caseB", 1, 16, 512, 64, True, 2),
    "caseC": Workload("caseC", 1, 32, 1024, 128, True, 3),
    "caseD": Workload("caseD", 8, 32, 512, 128, True, 4),
    "hd512": Workload("hd512", 1, 8, 2048, 512, True, 5, 0.5),
}

# Shapes beyond the five, for profiling the paths the five do not take: few heads of long
# causal rows, where the planner splits the longest query tiles' key ranges over clusters
# of two CTAs (split-KV).  bench.py --workload accepts these names; per_config times only
# the five workloads above.
EXTRA_WORKLOADS = {
    "long4": Workload("long4", 1, 4, 4096, 128, True, 8),
}


@dataclass(frozen=True)
class DecodeWorkload:
    """Decoding: one query row per (b, h) against L cached keys, every key visible
    ("Validating Memory-Optimal Transformer Kernels on Real Hardware", section 5, "Paper
    III: Inference (Decode)"; the pages scale the sequence length from 1,024 to 1,048,576
    and give no batch, head or head_dim sizes)."""
    name: str
    B: int
    H: int
    L: int
    d: int
    seed: int
    sigma: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self) -> float:
        """Algorithmic FLOPs: 4*B*H*L*d (q.K^T and p.V, 2*L*d each per head)."""
        return 4.0 * self.B * self.H * self.L * self.d

    def bytes(self) -> int:
        """Algorithmic HBM bytes: read K, V (and q) once, write o (2 B each) and LSE (4 B)."""
        bh = self.B * self.H
        return 2 * bh * self.d * (2 * self.L + 2) + 4 * bh

    def describe(self) -> str:
        return f"decode B={self.B} H={self.H} L={self.L} d={self.d} seed={self.seed} sigma={self.sigma}"


# A batched decode step (B x H = 256 sequences of 8192 cached tokens, 1.07 GB of K and V)
# and the pages' longest sequence, 1,048,576 tokens, for 8 heads (4.3 GB of K and V).
DECODE_WORKLOADS = {
    "decB": DecodeWorkload("decB", 8, 32, 8192, 128, 6),
    "dec1M": DecodeWorkload("dec1M", 1, 8, 1048576, 128, 7),
}
