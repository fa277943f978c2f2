"""Shapes of the synthetic decode workloads.

Stand-ins for the decode points of "Serving Kolibri-1 with a 4-bit KV cache" (section
"Throughput": decode only, every step decoding every session, 64k and 256k context;
Kolibri-1 has 50 attention layers, 40 of them sliding-window with window 513 and 10 with
full attention, 20 query and 4 KV heads of 128). The pages' workloads are Kolibri-1
serving runs; these configurations reproduce their shapes with seeded synthetic data
(see synth/__init__.py). Context L = positions cached before the step; the step appends
S rows at positions L .. L+S-1, so row r attends to L + r + 1 positions.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import context_lengths


@dataclass
class Workload:
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    S: int
    ctx: np.ndarray                 # int64[B]
    bf16: bool                      # q/k/v dtype (False: fp32)
    int4_layers: int = 1
    swa_layers: int = 0
    window: int = 513
    ring_capacity: int = 576
    page_order: str = "random"      # "ordered" or "random" physical page order
    steps: int = 1                  # consecutive decode steps the workload is quoted on
    extra: dict = field(default_factory=dict)

    @property
    def G(self):
        return self.Hq // self.Hkv

    def max_pages(self, extra_steps: int = 0) -> int:
        return int((int(self.ctx.max()) + self.S * (1 + extra_steps) + 63) // 64)

    def kv_bytes_int4(self) -> int:
        """Algorithmic int4 cache bytes one attention launch reads: 136 B per token-head
        (64 B K codes + 4 B K scale/offset + the same for V), over L + S positions."""
        return int(((self.ctx + self.S).sum()) * self.Hkv * 136)


def config(n: int) -> Workload:
    """The five configurations (1-based)."""
    if n == 1:  # tiny oracle check
        return Workload("tiny 1x512 ctx, 4/1 heads, fp32", 1, 1, 4, 1, 1, np.array([512]), False, page_order="ordered")
    if n == 2:  # single layer, 16 x 8k
        return Workload("16 x 8192 ctx, one int4 layer, 20/4 heads, bf16", 2, 16, 20, 4, 1,
                        np.full(16, 8192, np.int64), True, page_order="ordered")
    if n == 3:  # the 64k point: ragged 32k..64k
        return Workload("32 x U[32768,65536] ctx, one int4 layer, paged random order, bf16", 3, 32, 20, 4, 1,
                        context_lengths(3, 32, 32768, 65536), True)
    if n == 4:  # speculative verify
        return Workload("64 x 16384 ctx, S=4/8 verify, one int4 layer, bf16", 4, 64, 20, 4, 8,
                        np.full(64, 16384, np.int64), True, extra={"S_values": (4, 8)})
    if n == 5:  # the 256k point: full decode step over 50 layers
        return Workload("8 x 262144 ctx, 10 int4 + 40 FP8 window-513 layers, bf16", 5, 8, 20, 4, 1,
                        np.full(8, 262144, np.int64), True, int4_layers=10, swa_layers=40, steps=512)
    raise ValueError(n)


# fp8 per-tensor scales of the sliding-window layers: the generator's support [-6, 6]
# mapped onto the e4m3 range (keys and values are plain normals there).
SWA_K_SCALE = 6.0 / 448.0
SWA_V_SCALE = 6.0 / 448.0
