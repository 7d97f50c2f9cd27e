"""A layer's synthetic inputs placed in device memory (torch tensors), for tests and the bench.

The expert pool holds the E routed experts' records in slots 0..E-1, followed by the
n_shared shared experts' records. The records are written on the device by
libsynth_b300.so, or copied from the numpy generator with fill="host"; both give the
same bytes. slot_of is the identity (every routed expert resident).
"""
from __future__ import annotations

import numpy as np
import torch

from . import pack_record
from .workloads import Workload


class DeviceLayer:
    def __init__(self, w: Workload, layer: int = 0, device: str = "cuda", fill: str = "device"):
        self.w, self.layer, self.device = w, layer, device
        self.slot_bytes = w.record_bytes
        n = w.E + w.n_shared
        self.pool = torch.empty(n * self.slot_bytes, dtype=torch.uint8, device=device)
        if fill == "device":
            from .gpu import fill_expert_records
            fill_expert_records(w.seed, layer, 0, n, w.d, w.f, self.pool.data_ptr(), self.slot_bytes,
                                w.expert_sigma, fmt=w.fmt)
        else:
            for e in range(n):
                rec = pack_record(w.expert(layer, e), self.slot_bytes)
                self.pool[e * self.slot_bytes:(e + 1) * self.slot_bytes].copy_(torch.from_numpy(rec))
        self.slot_of = torch.arange(w.E, dtype=torch.int32, device=device)
        self.router = torch.from_numpy(w.router(layer)).to(device)

    @property
    def n_slots(self) -> int:
        """Slots of the routed-expert pool (the shared records follow them)."""
        return self.w.E

    @property
    def shared_ptr(self) -> int | None:
        return self.pool.data_ptr() + self.w.E * self.slot_bytes if self.w.n_shared else None

    def record_bytes_of(self, e: int) -> np.ndarray:
        """The bytes of record e (routed e < E, shared E + s) as they sit on the device."""
        return self.pool[e * self.slot_bytes:(e + 1) * self.slot_bytes].cpu().numpy()

    def x(self, batch: int = 0, dtype=torch.bfloat16) -> torch.Tensor:
        if dtype == torch.float32:
            return torch.from_numpy(self.w.x_f32(batch)).to(self.device)
        bits = self.w.x_bits(batch).astype(np.int16)
        return torch.from_numpy(bits).view(torch.bfloat16).to(self.device)
