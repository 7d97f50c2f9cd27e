"""ctypes loader of libsynth_b300.so: the device half of the seeded input generator."""
from __future__ import annotations

import ctypes as C
import os

_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsynth_b300.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_PATH):
            raise RuntimeError(f"{_PATH} is missing: build it with `python -m routed_expert_ffn_bucketing_b300.build`")
        _lib = C.CDLL(_PATH)
        _lib.synth_fill_expert_records.restype = C.c_int
        _lib.synth_fill_expert_records.argtypes = [C.c_uint64, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                                   C.c_float, C.c_void_p, C.c_uint64, C.c_void_p]
        _lib.synth_fill_expert_records_fmt.restype = C.c_int
        _lib.synth_fill_expert_records_fmt.argtypes = [C.c_uint64, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                                       C.c_float, C.c_void_p, C.c_uint64, C.c_int, C.c_void_p]
    return _lib


def fill_expert_records(seed: int, layer: int, expert0: int, n_experts: int, d: int, f: int, dst: int,
                        stride: int, sigma: float = 0.02, stream: int | None = None, fmt: int = 0) -> None:
    """Writes the records of experts expert0 .. expert0+n-1 of `layer` to device address dst,
    one every `stride` bytes; the same bytes as synth.pack_record(synth.expert_arrays(...)), or of
    expert_arrays_q2 with fmt 1."""
    if stream is None:
        import torch
        stream = torch.cuda.current_stream().cuda_stream
    rc = _load().synth_fill_expert_records_fmt(seed, layer, expert0, n_experts, d, f, sigma, dst, stride, fmt,
                                               stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_expert_records failed with CUDA error {rc}")
