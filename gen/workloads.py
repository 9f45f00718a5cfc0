"""The synthetic workloads of the quantized MoE expert layer.

Each is named by what it is and its sizes.  Shapes, formats, top-k, shared
expert and router-bias recipes follow the layer shapes the engine pages speak
of (512 experts with top-10 and one shared expert in the hybrid-attention
family; 256 experts with top-8 in the larger family; NVFP4 with an e4m3 scale
per 16 weights and FP6 e2m3 with a power-of-two scale per 128 weights, from
the knivesysl README, "formats").
"""
from __future__ import annotations

from dataclasses import dataclass

FMT_NVFP4 = 1
FMT_FP6 = 2
FMT_MXFP4 = 3


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    I: int
    E: int
    k: int
    shared: int
    T: int
    fmt: int
    bias: str            # "none" | "zipf" | "normal"
    bias_param: float = 0.0   # Zipf exponent
    bias_scale: float = 0.0   # Zipf multiplier, or the normal bias' sigma
    seed: int = 0

    @property
    def n_experts_total(self) -> int:
        return self.E + (1 if self.shared else 0)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny-h256-i128-e8-k2-t4-nvfp4", 256, 128, 8, 2, 0, 4, FMT_NVFP4, "none", seed=0),
        Workload("decode-h2048-i512-e512-k10-s1-t1-nvfp4", 2048, 512, 512, 10, 1, 1, FMT_NVFP4,
                 "zipf", 1.1, 0.5, seed=0),
        Workload("decode-h6144-i2048-e256-k8-s1-t1-fp6", 6144, 2048, 256, 8, 1, 1, FMT_FP6, "none",
                 seed=0),
        Workload("batched-h2048-i512-e512-k10-s1-t64-nvfp4", 2048, 512, 512, 10, 1, 64, FMT_NVFP4,
                 "zipf", 1.1, 0.5, seed=0),
        Workload("prefill-h2048-i512-e512-k10-s1-t4096-nvfp4", 2048, 512, 512, 10, 1, 4096,
                 FMT_NVFP4, "normal", 0.0, 0.1, seed=0),
        # MXFP4 and the DeepSeek-V4 expert shape (256 routed + 1 shared, top-6).
        # The pages give no H or I; ~167 GB over 43 layers of 257 fp4 experts
        # bounds a matrix at ~9.5M weights, and H = 4096, I = 2048 (8.4M) is
        # the reading taken
        Workload("tiny-h256-i128-e8-k2-t4-mxfp4", 256, 128, 8, 2, 0, 4, FMT_MXFP4, "none", seed=1),
        Workload("decode-h4096-i2048-e256-k6-s1-t1-mxfp4", 4096, 2048, 256, 6, 1, 1, FMT_MXFP4,
                 "normal", 0.0, 0.1, seed=0),
        Workload("prefill-h4096-i2048-e256-k6-s1-t4096-mxfp4", 4096, 2048, 256, 6, 1, 4096,
                 FMT_MXFP4, "normal", 0.0, 0.1, seed=0),
    ]
}

ORDER = list(WORKLOADS)


def get_workload(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[ORDER[name_or_index]]
    return WORKLOADS[name_or_index]
