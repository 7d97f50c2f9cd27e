"""The workloads: shapes and input recipes of the MoE layer configurations.

Each workload is seeded and synthetic. No dataset is involved, and the pages measure none
for this path.
  tiny     T=16, d=256, f=128, E=16, top-2, no shared expert; router N(0, 0.02)
  decode   T=4 (one token plus three drafts), d=2048, f=768, E=512, top-10 + 1 shared; router N(0, 1)
  stack    48 decode layers, router columns scaled for Zipf(1.1) popularity, residual stream
  prefill  T=8192 chunk, d=2048, f=768, E=512, top-10 + 1 shared, Zipf(1.1) routing
  tiered   the stack with a 4,500-slot device pool, the rest in pinned host memory
  decode_q2, tiered_q2   decode and tiered with 2-bit expert records (2.5 bits per weight); the
           tiered pool has the same bytes (22.56 GB), so 15,300 slots
Experts are N(0, 0.02) quantised to int8 blocks of 32 with fp16 scales (or to the 2-bit format).
Activations are N(0, 1) rounded to bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

from . import (FMT_INT8, FMT_Q2, activations_bf16, activations_f32, bf16_bits_to_f32, expert_arrays,
               expert_arrays_q2, record_layout, router_weights)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    n_shared: int
    router_sigma: float
    zipf_s: float | None = None
    layers: int = 1
    residual: bool = False
    slots: int | None = None       # device slot pool size (tiered); None = every expert resident
    seed: int = 0
    expert_sigma: float = 0.02
    fmt: int = FMT_INT8            # expert record format: FMT_INT8 or FMT_Q2 (2-bit codes)

    @property
    def P(self) -> int:
        return self.T * self.k

    @property
    def record_bytes(self) -> int:
        return record_layout(self.d, self.f, self.fmt).record_bytes

    def describe(self) -> str:
        s = f"{self.name}: T={self.T} d={self.d} f={self.f} E={self.E} top-{self.k}"
        s += f" + {self.n_shared} shared" if self.n_shared else ""
        if self.layers > 1:
            s += f", {self.layers} layers"
        if self.zipf_s:
            s += f", Zipf({self.zipf_s}) routing"
        if self.fmt == FMT_Q2:
            s += ", 2-bit block-32 experts (2.5 bits per weight)"
        return s

    # ---- inputs -------------------------------------------------------------------------
    def x_bits(self, batch: int = 0) -> np.ndarray:
        """bf16 bit patterns [T][d] of input batch `batch`."""
        return activations_bf16(self.seed, batch, self.T, self.d)

    def x_f64(self, batch: int = 0) -> np.ndarray:
        return bf16_bits_to_f32(self.x_bits(batch)).astype(np.float64)

    def x_f32(self, batch: int = 0) -> np.ndarray:
        """fp32 activations (the fp32 debug mode's input)."""
        return activations_f32(self.seed, batch, self.T, self.d)

    def router(self, layer: int = 0) -> np.ndarray:
        return router_weights(self.seed, layer, self.d, self.E, self.router_sigma, self.zipf_s, self.k)

    def expert(self, layer: int, e: int):
        """Routed expert e < E, or shared expert s as e = E + s."""
        gen = expert_arrays_q2 if self.fmt == FMT_Q2 else expert_arrays
        return gen(self.seed, layer, e, self.d, self.f, self.expert_sigma)


WORKLOADS = {
    "tiny": Workload("tiny", 16, 256, 128, 16, 2, 0, 0.02),
    "decode": Workload("decode", 4, 2048, 768, 512, 10, 1, 1.0),
    "stack": Workload("stack", 4, 2048, 768, 512, 10, 1, 1.0, zipf_s=1.1, layers=48, residual=True),
    "prefill": Workload("prefill", 8192, 2048, 768, 512, 10, 1, 1.0, zipf_s=1.1),
    "tiered": Workload("tiered", 4, 2048, 768, 512, 10, 1, 1.0, zipf_s=1.1, layers=48, residual=True, slots=4500),
    # the same device pool bytes (4,500 x 5,013,504 B) holding 2-bit records of 1,474,560 B
    "tiered_q2": Workload("tiered_q2", 4, 2048, 768, 512, 10, 1, 1.0, zipf_s=1.1, layers=48, residual=True,
                          slots=15300, fmt=FMT_Q2),
    "decode_q2": Workload("decode_q2", 4, 2048, 768, 512, 10, 1, 1.0, fmt=FMT_Q2),
}


def custom(base: str, **kw) -> Workload:
    return replace(WORKLOADS[base], **kw)
