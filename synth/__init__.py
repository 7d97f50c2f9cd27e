"""Seeded synthetic inputs for the sparse MoE layer: test and benchmark infrastructure.

This module prepares inputs and nothing else. It holds:

* a counter-based random stream: SplitMix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014), where draw i of a stream with key K is
  mix64(K + (i + 1) * 0x9E3779B97F4A7C15 mod 2^64);
* an approximately normal draw built from one 64-bit value without transcendental
  functions (Irwin-Hall sum of four 16-bit uniforms, rescaled to unit variance), so that
  a CUDA implementation of the same draw (synth/csrc/synth_fill.cu) is bit-identical;
* the block-32 weight quantiser that turns N(0, sigma) weights into int8 codes plus one
  fp16 scale per 32 consecutive elements of the reduction dimension (the weight format
  of the workloads: s = fp16_rne(amax / 127), q = clamp(rint(w / s), -127, 127)), and the
  2.5-bit one of the sub-4-bit format (2-bit codes c with w = s (c - 1.5): s = fp16_rne(amax /
  1.5), c = clamp(rint(w / s + 1.5), 0, 3));
* the packing of one expert's six arrays into its byte record;
* the router columns' Zipf(s) popularity recipe.

None of the layer's own arithmetic (router logits, softmax, top-k, bucketing, SwiGLU,
combine) lives here. The oracle and the CUDA path both consume these inputs; neither
implements them, and this module imports neither of them.
"""
from __future__ import annotations

import functools
from dataclasses import dataclass

import numpy as np

M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB

# fp32 sqrt(3) * 2^-16: the unit-variance rescale of a sum of four 16-bit uniforms.
ZSCALE = np.float32(np.sqrt(3.0)) * np.float32(2.0 ** -16)
assert int(np.float32(ZSCALE).view(np.uint32)) == 0x37DDB3D7

BLOCK = 32  # elements per quantisation block along the reduction dimension

# stream tags (the first component of every stream key)
TAG_GATE, TAG_UP, TAG_DOWN, TAG_X, TAG_ROUTER, TAG_PERM, TAG_ZIPF_MC, TAG_DRIFT = 1, 2, 3, 4, 5, 6, 7, 8


def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (mod 2^64)."""
    z &= M64
    z = ((z ^ (z >> 30)) * _MIX1) & M64
    z = ((z ^ (z >> 27)) * _MIX2) & M64
    return z ^ (z >> 31)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= np.uint64(_MIX1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(_MIX2)
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, tag: int, a: int = 0, b: int = 0) -> int:
    """Key of the stream (seed, tag, a, b); a and b are below 2^24, tag below 2^16."""
    assert 0 <= a < (1 << 24) and 0 <= b < (1 << 24) and 0 <= tag < (1 << 16)
    return mix64_int((mix64_int(seed) + ((tag << 48) ^ (a << 24) ^ b)) & M64)


def draws_u64(key: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of the stream with this key (uint64)."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        ctr = np.uint64(key) + i * np.uint64(GOLDEN)
    return _mix64(ctr)


def normal_f32(key: int, start: int, count: int, sigma: float) -> np.ndarray:
    """Approximately N(0, sigma) fp32 values: (sum of four 16-bit fields - 131070)
    * fp32(sqrt 3) * 2^-16, then * fp32(sigma); each product rounded once (IEEE fp32)."""
    r = draws_u64(key, start, count)
    m = np.uint64(0xFFFF)
    s = (r & m) + ((r >> np.uint64(16)) & m) + ((r >> np.uint64(32)) & m) + (r >> np.uint64(48))
    z = (s.astype(np.int64) - 131070).astype(np.float32) * ZSCALE
    return (z * np.float32(sigma)).astype(np.float32)


def quantize_block32(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """int8 codes and fp16 scales of fp32 w [R][C] in blocks of 32 along C.

    s = fp16_rne(amax / 127) (fp32 division), q = clamp(rint(w / s), -127, 127) with
    round-half-even and fp32 division; a block whose scale is 0 gets q = 0."""
    R, C = w.shape
    assert C % BLOCK == 0
    wb = w.astype(np.float32).reshape(R, C // BLOCK, BLOCK)
    amax = np.abs(wb).max(axis=2)
    s16 = (amax / np.float32(127.0)).astype(np.float32).astype(np.float16)
    sf = s16.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        qf = np.rint(wb / sf)
    qf = np.where(sf == 0, np.float32(0), qf)
    q = np.clip(qf, -127, 127).astype(np.int8).reshape(R, C)
    return q, s16


def quantize_q2_block32(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """2-bit codes (uint8, 0..3) and fp16 scales of fp32 w [R][C] in blocks of 32 along C, for
    the format w = s * (c - 1.5): s = fp16_rne(amax / 1.5) (fp32 division), c = clamp(rint(w / s
    + 1.5), 0, 3) with the division and the addition in fp32 and round-half-even; a block whose
    scale is 0 gets c = 0."""
    R, C = w.shape
    assert C % BLOCK == 0
    wb = w.astype(np.float32).reshape(R, C // BLOCK, BLOCK)
    amax = np.abs(wb).max(axis=2)
    s16 = (amax / np.float32(1.5)).astype(np.float32).astype(np.float16)
    sf = s16.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        cf = np.rint((wb / sf).astype(np.float32) + np.float32(1.5))
    cf = np.where(sf == 0, np.float32(0), cf)
    c = np.clip(cf, 0, 3).astype(np.uint8).reshape(R, C)
    return c, s16


def fp32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns.
    Inputs are finite (the generator never produces NaN or Inf)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------------------
# expert records
# --------------------------------------------------------------------------------------

def _align256(n: int) -> int:
    return (n + 255) // 256 * 256


@dataclass(frozen=True)
class RecordLayout:
    """Byte offsets of one expert record: gate_q [f][d] i8, up_q [f][d] i8, down_q [d][f]
    i8 (each row in the stored order of interleave_codes), gate_s [f][d/32] f16, up_s [f][d/32]
    f16, down_s [d][f/32] f16, each section starting on a 256-byte boundary."""
    d: int
    f: int
    gate_q: int
    up_q: int
    down_q: int
    gate_s: int
    up_s: int
    down_s: int
    record_bytes: int


FMT_INT8, FMT_Q2 = 0, 1  # record formats: int8 codes, or 2-bit codes (4 per byte)


def record_layout(d: int, f: int, fmt: int = FMT_INT8) -> RecordLayout:
    """fmt FMT_INT8: one byte per code; FMT_Q2: four codes per byte (d and f multiples of 256)."""
    assert d % BLOCK == 0 and f % BLOCK == 0
    cb = 1 if fmt == FMT_INT8 else 4  # codes per byte
    if fmt == FMT_Q2:
        assert d % 256 == 0 and f % 256 == 0
    sizes = [f * d // cb, f * d // cb, d * f // cb, f * (d // BLOCK) * 2, f * (d // BLOCK) * 2,
             d * (f // BLOCK) * 2]
    offs, o = [], 0
    for n in sizes:
        offs.append(o)
        o = _align256(o + n)
    return RecordLayout(d, f, *offs, o)


@dataclass
class ExpertArrays:
    """One expert's quantised weights (the oracle's view of a record). fmt "int8": codes are int8;
    fmt "q2": codes are 2-bit values 0..3 (uint8 arrays) of the format w = s (c - 1.5)."""
    gate_q: np.ndarray  # int8 [f][d]
    gate_s: np.ndarray  # fp16 [f][d/32]
    up_q: np.ndarray    # int8 [f][d]
    up_s: np.ndarray    # fp16 [f][d/32]
    down_q: np.ndarray  # int8 [d][f]
    down_s: np.ndarray  # fp16 [d][f/32]
    fmt: str = "int8"


def expert_arrays(seed: int, layer: int, expert: int, d: int, f: int,
                  sigma: float = 0.02) -> ExpertArrays:
    """Expert `expert` of layer `layer`: N(0, sigma) weights quantised in blocks of 32 along
    the reduction dimension (d for gate/up, f for down). Shared experts use ids E, E+1, ..."""
    g = normal_f32(stream_key(seed, TAG_GATE, layer, expert), 0, f * d, sigma).reshape(f, d)
    u = normal_f32(stream_key(seed, TAG_UP, layer, expert), 0, f * d, sigma).reshape(f, d)
    w = normal_f32(stream_key(seed, TAG_DOWN, layer, expert), 0, d * f, sigma).reshape(d, f)
    gq, gs = quantize_block32(g)
    uq, us = quantize_block32(u)
    dq, ds = quantize_block32(w)
    return ExpertArrays(gq, gs, uq, us, dq, ds)


def expert_arrays_q2(seed: int, layer: int, expert: int, d: int, f: int,
                     sigma: float = 0.02) -> ExpertArrays:
    """The same N(0, sigma) weights as expert_arrays, quantised to the 2-bit format."""
    g = normal_f32(stream_key(seed, TAG_GATE, layer, expert), 0, f * d, sigma).reshape(f, d)
    u = normal_f32(stream_key(seed, TAG_UP, layer, expert), 0, f * d, sigma).reshape(f, d)
    w = normal_f32(stream_key(seed, TAG_DOWN, layer, expert), 0, d * f, sigma).reshape(d, f)
    gq, gs = quantize_q2_block32(g)
    uq, us = quantize_q2_block32(u)
    dq, ds = quantize_q2_block32(w)
    return ExpertArrays(gq, gs, uq, us, dq, ds, fmt="q2")


# stored position of code j (0..7) of a lane's 8 consecutive codes in the 2-bit format: the
# order (0, 2, 1, 3, 4, 6, 5, 7), two bits each
_Q2_SLOT = np.array([0, 2, 1, 3, 4, 6, 5, 7])


def pack_codes_q2(c: np.ndarray) -> np.ndarray:
    """Rows of 2-bit codes [R][K] (K a multiple of 256) to their stored bytes [R][K/4]: in each
    group of 8 blocks (256 codes, 64 bytes), 16-byte chunk q holds for block b = 0..7 one 16-bit
    little-endian word with codes 8q..8q+7 of block b, code j at bits 2 * slot(j), slot the
    order (0, 2, 1, 3, 4, 6, 5, 7)."""
    R, K = c.shape
    assert K % 256 == 0
    v = c.astype(np.uint32).reshape(R, K // 256, 8, 4, 8)        # [r][group][block][q][j]
    words = np.zeros((R, K // 256, 8, 4), dtype=np.uint32)
    for j in range(8):
        words |= v[..., j] << np.uint32(2 * _Q2_SLOT[j])
    words = words.transpose(0, 1, 3, 2).astype(np.uint16)       # [r][group][q][block]
    return np.ascontiguousarray(words).view(np.uint8).reshape(R, K // 4)


def unpack_codes_q2(b: np.ndarray) -> np.ndarray:
    """The inverse of pack_codes_q2."""
    R, KB = b.shape
    K = KB * 4
    words = np.ascontiguousarray(b).view(np.uint16).reshape(R, K // 256, 4, 8).transpose(0, 1, 3, 2)
    out = np.zeros((R, K // 256, 8, 4, 8), dtype=np.uint8)
    for j in range(8):
        out[..., j] = (words.astype(np.uint32) >> np.uint32(2 * _Q2_SLOT[j])) & 3
    return out.reshape(R, K)


def interleave_codes(q: np.ndarray) -> np.ndarray:
    """Rows of int8 codes [R][K] in the stored order: in each 64-code span (two blocks of 32)
    chunk c (16 bytes) holds codes 8c..8c+7 of the first block, then 8c..8c+7 of the second;
    a trailing block without a partner stays as it is."""
    R, K = q.shape
    K64 = K // 64 * 64
    out = q.copy()
    out[:, :K64] = q[:, :K64].reshape(R, K64 // 64, 2, 4, 8).transpose(0, 1, 3, 2, 4).reshape(R, K64)
    return out


def deinterleave_codes(q: np.ndarray) -> np.ndarray:
    """The inverse of interleave_codes."""
    R, K = q.shape
    K64 = K // 64 * 64
    out = q.copy()
    out[:, :K64] = q[:, :K64].reshape(R, K64 // 64, 4, 2, 8).transpose(0, 1, 3, 2, 4).reshape(R, K64)
    return out


def pack_record(a: ExpertArrays, slot_bytes: int | None = None) -> np.ndarray:
    """Byte record (uint8) of one expert in the layout of record_layout (codes in the stored
    order of interleave_codes, or of pack_codes_q2 for the 2-bit format); zero padding."""
    f, d = a.gate_q.shape
    q2 = a.fmt == "q2"
    L = record_layout(d, f, FMT_Q2 if q2 else FMT_INT8)
    n = L.record_bytes if slot_bytes is None else slot_bytes
    assert n >= L.record_bytes
    rec = np.zeros(n, dtype=np.uint8)
    pk = pack_codes_q2 if q2 else interleave_codes
    for off, arr in ((L.gate_q, pk(a.gate_q)), (L.up_q, pk(a.up_q)), (L.down_q, pk(a.down_q)),
                     (L.gate_s, a.gate_s), (L.up_s, a.up_s), (L.down_s, a.down_s)):
        b = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
        rec[off:off + b.size] = b
    return rec


def unpack_record(rec: np.ndarray, d: int, f: int, fmt: int = FMT_INT8) -> ExpertArrays:
    L = record_layout(d, f, fmt)
    r = np.ascontiguousarray(rec, dtype=np.uint8)

    def take(off, n, dt, shape):
        return r[off:off + n * np.dtype(dt).itemsize].view(dt).reshape(shape).copy()
    nb_d, nb_f = d // BLOCK, f // BLOCK
    if fmt == FMT_Q2:
        return ExpertArrays(unpack_codes_q2(take(L.gate_q, f * d // 4, np.uint8, (f, d // 4))),
                            take(L.gate_s, f * nb_d, np.float16, (f, nb_d)),
                            unpack_codes_q2(take(L.up_q, f * d // 4, np.uint8, (f, d // 4))),
                            take(L.up_s, f * nb_d, np.float16, (f, nb_d)),
                            unpack_codes_q2(take(L.down_q, d * f // 4, np.uint8, (d, f // 4))),
                            take(L.down_s, d * nb_f, np.float16, (d, nb_f)), fmt="q2")
    return ExpertArrays(deinterleave_codes(take(L.gate_q, f * d, np.int8, (f, d))),
                        take(L.gate_s, f * nb_d, np.float16, (f, nb_d)),
                        deinterleave_codes(take(L.up_q, f * d, np.int8, (f, d))),
                        take(L.up_s, f * nb_d, np.float16, (f, nb_d)),
                        deinterleave_codes(take(L.down_q, d * f, np.int8, (d, f))),
                        take(L.down_s, d * nb_f, np.float16, (d, nb_f)))


# --------------------------------------------------------------------------------------
# activations and router weights
# --------------------------------------------------------------------------------------

def activations_bf16(seed: int, batch: int, T: int, d: int, sigma: float = 1.0) -> np.ndarray:
    """Token activations x [T][d] ~ N(0, sigma), rounded to bf16; returned as uint16 bits."""
    v = normal_f32(stream_key(seed, TAG_X, batch, 0), 0, T * d, sigma)
    return fp32_to_bf16_bits(v).reshape(T, d)


def activations_f32(seed: int, batch: int, T: int, d: int, sigma: float = 1.0) -> np.ndarray:
    return normal_f32(stream_key(seed, TAG_X, batch, 0), 0, T * d, sigma).reshape(T, d)


def expert_rank_permutation(seed: int, layer: int, E: int) -> np.ndarray:
    """perm[r] = expert holding popularity rank r in this layer (a seeded shuffle)."""
    r = draws_u64(stream_key(seed, TAG_PERM, layer, 0), 0, E)
    return np.argsort(r, kind="stable").astype(np.int64)


DRIFT_EVERY = 10      # steps between two drift epochs of the hot set
DRIFT_SWAPS = 5       # adjacent-rank transpositions per epoch


def drift_rank_permutation(perm: np.ndarray, seed: int, layer: int, epoch: int) -> np.ndarray:
    """One drift epoch of a layer's popularity ranking: DRIFT_SWAPS transpositions of
    adjacent ranks (r, r + 1), r drawn uniformly from 0 .. E-2 by the counter generator
    keyed (seed, layer, epoch). Returns the new rank -> expert permutation (a copy)."""
    E = perm.size
    out = perm.copy()
    r = draws_u64(stream_key(seed, TAG_DRIFT, layer, epoch), 0, DRIFT_SWAPS) % np.uint64(E - 1)
    for j in r.astype(np.int64):
        out[j], out[j + 1] = out[j + 1], out[j]
    return out


def router_column_scales(perm: np.ndarray, E: int, k: int, s: float, seed: int = 0) -> np.ndarray:
    """fp32 [E]: the Zipf scale of each expert's column under the ranking perm."""
    c, _ = zipf_column_scales(E, k, s, seed)
    col = np.empty(E, dtype=np.float32)
    col[perm] = c
    return col


@functools.lru_cache(maxsize=None)
def zipf_column_scales(E: int, k: int, s: float, seed: int = 0, n_mc: int = 4096,
                       iters: int = 60) -> tuple[np.ndarray, np.ndarray]:
    """Scales c[r] (fp32) for the router column of popularity rank r, so that top-k over
    logits c[r] * z_r with z_r iid N(0, 1) (the law of x . w_e for fixed x and N(0, 1)
    columns) includes rank r with frequency close to k r^-s / H, H = sum_r r^-s.

    A Gaussian logit is negative half the time, so no rank can be included more often
    than about half of the tokens: targets are capped at 0.45 and the excess is spread
    over the other ranks. Calibrated by a seeded Monte Carlo with a fixed number of damped
    multiplicative updates, kept non-increasing in r. Returns (c, realised inclusion
    frequency per rank in the last Monte-Carlo pass)."""
    ranks = np.arange(1, E + 1, dtype=np.float64)
    target = k * ranks ** (-s) / np.sum(ranks ** (-s))
    for _ in range(8):
        target = np.minimum(target, 0.45)
        target *= k / target.sum()
    target = np.minimum(target, 0.45)
    z = normal_f32(stream_key(seed, TAG_ZIPF_MC, E, k), 0, n_mc * E, 1.0).reshape(n_mc, E).astype(np.float64)
    logc = np.zeros(E)
    freq = None
    for it in range(iters):
        lg = z * np.exp(logc)[None, :]
        sel = np.argpartition(-lg, k - 1, axis=1)[:, :k]
        freq = np.bincount(sel.reshape(-1), minlength=E) / n_mc
        step = 0.05 + 0.35 * (1.0 - it / iters)
        logc += step * (np.log(target) - np.log(np.maximum(freq, 0.5 / n_mc)))
        logc = np.minimum.accumulate(logc)
        logc -= logc.max()
    c = np.exp(logc).astype(np.float32)
    return c, freq


def router_weights(seed: int, layer: int, d: int, E: int, sigma: float,
                   zipf_s: float | None = None, k: int | None = None) -> np.ndarray:
    """Router weights w_router [d][E] fp32 ~ N(0, sigma). With zipf_s, column e is further
    multiplied (one fp32 rounding) by the scale of its popularity rank in this layer."""
    w = normal_f32(stream_key(seed, TAG_ROUTER, layer, 0), 0, d * E, sigma).reshape(d, E)
    if zipf_s is None:
        return w
    col = router_column_scales(expert_rank_permutation(seed, layer, E), E, k, zipf_s, seed)
    return (w * col[None, :]).astype(np.float32)


def router_weights_unscaled(seed: int, layer: int, d: int, E: int, sigma: float) -> np.ndarray:
    """The N(0, sigma) draws of router_weights before the Zipf column scales."""
    return normal_f32(stream_key(seed, TAG_ROUTER, layer, 0), 0, d * E, sigma).reshape(d, E)
