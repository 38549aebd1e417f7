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
