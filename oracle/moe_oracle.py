"""CPU oracle for one sparse MoE layer's forward pass (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this module. The
product path never imports it, and it shares no code with the CUDA library. It is written
for a reader checking it against its sources, not for speed: numpy in float64, one
library matmul or sort per step, and no blocking, fusion or reordering.

What it computes comes from two sources:
* the pages on the Strata engine. "单张RTX 5090跑125B大模型：Strata实测Qwen3.8 Flash Next",
  section "MoE专家按需调度" (MoE explainer): a light router picks the top-K experts per
  token, and the other experts take no part. "Strata 工作原理图解GPU内存SSD三级存储如何让125B
  模型塞进消费级显卡", section "三级存储分工": the router and a shared expert stay in VRAM,
  and the shared expert is applied to every token. Section "专家缓存": experts stay resident in a slot cache.
* the workload definition those pages leave open. It fixes the dequantise, fp32
  router, softmax, top-k with lowest-index tie-break, renormalise, SwiGLU and weighted-sum steps.

Readings taken where the pages are silent (each also listed in the design notes):
* The expert FFN is SwiGLU without biases: y = W_d (silu(W_g x) * W_u x), silu(z) = z / (1 + e^-z).
* The shared expert is added with weight 1 and takes no part in the renormalised sum.
* Ties in the top-k go to the lowest expert index, and -0.0 and +0.0 compare equal.
* A logit is x . w_router accumulated exactly (float64 here) and rounded once to fp32. That
  fp32 value decides the top-k on both sides.
* The gate is the softmax over all E logits, restricted to the selected k and renormalised.
* Output is out[t] = sum_j w[t, j] y_{e_j}(x_t) + sum_s y_shared_s(x_t) (+ x_t as a residual
  when asked), rounded once at the end to bf16 (or kept in float64 for the fp32 debug mode).
* In a stack of layers each layer is a pre-norm residual block: x_{l+1} = x_l + MoE_l(n(x_l))
  with n the RMS normalisation without a learned gain, n(x) = x / sqrt(mean(x^2) + eps),
  eps = 1e-6. With no normalisation the residual stream of N(0, 0.02) SwiGLU experts grows
  without bound (SwiGLU is quadratic for large inputs) and overflows within a few dozen layers.

Parity status: each function here is pinned by tests/test_oracle_pins.py against brute
force, closed forms, hand-computed examples or invariants.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable, Sequence

import numpy as np

BLOCK = 32


# ---------------------------------------------------------------------------------------
# dequantisation: W[r, i] = q[r, i] * s[r, i // 32]
# ---------------------------------------------------------------------------------------

def dequantize(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Dense float64 weights from int8 codes q [R][C] and fp16 block scales s [R][C/32].
    Exact: an int8 times an fp16 needs at most 8 + 11 significant bits."""
    R, C = q.shape
    assert s.shape == (R, C // BLOCK)
    scale = np.repeat(s.astype(np.float64), BLOCK, axis=1)
    return q.astype(np.float64) * scale


def dequantize_q2(c: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Dense float64 weights of the sub-4-bit format: 2-bit codes c [R][C] (values 0..3) and
    fp16 block scales s [R][C/32], W[r, i] = s[r, i // 32] * (c[r, i] - 1.5): four levels
    symmetric about zero, 2.5 bits per weight with the scale. Exact in float64."""
    R, C = c.shape
    assert s.shape == (R, C // BLOCK)
    assert np.all((c >= 0) & (c <= 3))
    scale = np.repeat(s.astype(np.float64), BLOCK, axis=1)
    return (c.astype(np.float64) - 1.5) * scale


# ---------------------------------------------------------------------------------------
# RMS normalisation of a layer's input (pre-norm residual block of a layer stack)
# ---------------------------------------------------------------------------------------

RMS_EPS = 1e-6


def rms_norm(x: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """n(x)[t] = x[t] / sqrt(mean_i x[t, i]^2 + eps), per row, in float64 (no learned gain)."""
    x = x.astype(np.float64)
    return x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps)


# ---------------------------------------------------------------------------------------
# router, top-k and gate
# ---------------------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_router: np.ndarray) -> np.ndarray:
    """logit[t, e] = sum_i x[t, i] * w_router[i, e], summed in float64 and rounded once to fp32."""
    return (x.astype(np.float64) @ w_router.astype(np.float64)).astype(np.float32)


def select_topk(logits32: np.ndarray, k: int) -> np.ndarray:
    """Indices [T][k] of the k largest fp32 logits per token. Order: descending logit, then
    ascending expert index, so ties go to the lowest index. -0.0 counts as +0.0 and NaN as -inf."""
    T, E = logits32.shape
    assert 1 <= k <= E
    v = logits32.astype(np.float64) + 0.0          # -0.0 + 0.0 = +0.0
    v = np.where(np.isnan(v), -np.inf, v)
    out = np.empty((T, k), dtype=np.int32)
    experts = np.arange(E)
    for t in range(T):
        order = np.lexsort((experts, -v[t]))        # primary: -logit, secondary: index
        out[t] = order[:k]
    return out


def gate_weights(logits32: np.ndarray, topk_idx: np.ndarray) -> np.ndarray:
    """Renormalised gate weights [T][k]: p = softmax over all E logits (float64, max-subtracted),
    w[t, j] = p[t, e_j] / sum_j' p[t, e_j']."""
    v = logits32.astype(np.float64)
    m = np.max(v, axis=1, keepdims=True)
    p = np.exp(v - m)
    p = p / np.sum(p, axis=1, keepdims=True)
    sel = np.take_along_axis(p, topk_idx.astype(np.int64), axis=1)
    return sel / np.sum(sel, axis=1, keepdims=True)


# ---------------------------------------------------------------------------------------
# expert FFN (SwiGLU)
# ---------------------------------------------------------------------------------------

@dataclass
class DenseExpert:
    """One expert's dequantised float64 weights: gate [f][d], up [f][d], down [d][f]."""
    gate: np.ndarray
    up: np.ndarray
    down: np.ndarray


def dense_expert(a) -> DenseExpert:
    """Dequantise the six arrays of one expert (any object with gate_q, gate_s, up_q, up_s,
    down_q and down_s attributes; fmt "q2" for the 2-bit format, int8 codes otherwise)."""
    deq = dequantize_q2 if getattr(a, "fmt", "int8") == "q2" else dequantize
    return DenseExpert(deq(a.gate_q, a.gate_s), deq(a.up_q, a.up_s), deq(a.down_q, a.down_s))


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def swiglu_ffn(xrows: np.ndarray, ex: DenseExpert) -> np.ndarray:
    """y = W_d (silu(W_g x) * W_u x) for each row x of xrows [n][d]; float64 throughout."""
    g = xrows @ ex.gate.T
    u = xrows @ ex.up.T
    h = silu(g) * u
    return h @ ex.down.T


# ---------------------------------------------------------------------------------------
# bucketing: stable counting sort of flat pair ids p = t*k + j by expert
# ---------------------------------------------------------------------------------------

@dataclass
class Buckets:
    counts: np.ndarray       # int32 [E]: pairs routed to each expert
    offsets: np.ndarray      # int32 [E+1]: exclusive prefix sum of counts
    sorted_pair: np.ndarray  # int32 [T*k]: pair ids grouped by expert, ascending within a group
    inv_pos: np.ndarray      # int32 [T*k]: position of pair p in sorted_pair
    active: np.ndarray       # int32 [n_active]: experts with count > 0, ascending


def bucketing(topk_idx: np.ndarray, E: int) -> Buckets:
    """Group the (token, slot) pairs by expert so that each expert's rows form one contiguous
    run, in ascending pair order within the run."""
    e_of_pair = topk_idx.reshape(-1).astype(np.int64)
    P = e_of_pair.size
    counts = np.bincount(e_of_pair, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    sorted_pair = np.empty(P, dtype=np.int64)
    fill = offsets[:-1].copy()
    for p in range(P):                       # counting sort, stable by construction
        e = e_of_pair[p]
        sorted_pair[fill[e]] = p
        fill[e] += 1
    inv_pos = np.empty(P, dtype=np.int64)
    inv_pos[sorted_pair] = np.arange(P)
    active = np.nonzero(counts)[0]
    return Buckets(counts.astype(np.int32), offsets.astype(np.int32), sorted_pair.astype(np.int32),
                   inv_pos.astype(np.int32), active.astype(np.int32))


# ---------------------------------------------------------------------------------------
# bf16 rounding of the layer output
# ---------------------------------------------------------------------------------------

def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values once to the nearest bf16 value (8 significant bits), ties to even.
    Written from the definition: v = m * 2^e with 0.5 <= |m| < 1, keep 8 bits of m.
    Finite inputs inside the normal bf16 range; zero stays zero."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)
    r = np.rint(m * 256.0)                   # np.rint rounds half to even
    return np.ldexp(r, e - 8)


# ---------------------------------------------------------------------------------------
# the whole layer
# ---------------------------------------------------------------------------------------

@dataclass
class LayerResult:
    out: np.ndarray           # float64 [n][d] before the final rounding
    logits: np.ndarray        # fp32 [n][E]
    topk_idx: np.ndarray      # int32 [n][k] (forced or selected)
    topk_w: np.ndarray        # float64 [n][k]
    tokens: np.ndarray        # int64 [n]: which tokens of the batch these rows are


def moe_layer(x: np.ndarray, w_router: np.ndarray, k: int,
              expert: Callable[[int], object], shared: Sequence[object] = (),
              residual: bool = False, forced_idx: np.ndarray | None = None,
              tokens: np.ndarray | None = None) -> LayerResult:
    """Forward pass of one MoE layer for the rows `tokens` of x [T][d] (all rows by default).

    expert(e) returns routed expert e's quantised arrays. `shared` holds the always-on shared
    experts. forced_idx [T][k] replaces the top-k selection (forced routing: used where
    two logits are too close to decide). Each token is computed on its own, as the
    definition is per token.
    """
    T, d = x.shape
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    xs = x[tok].astype(np.float64)
    logits = router_logits(xs, w_router)
    idx = select_topk(logits, k) if forced_idx is None else np.asarray(forced_idx)[tok].astype(np.int32)
    w = gate_weights(logits, idx)
    out = np.zeros((tok.size, d), dtype=np.float64)
    for e in np.unique(idx):
        ex = dense_expert(expert(int(e)))
        rows, slots = np.nonzero(idx == e)
        y = swiglu_ffn(xs[rows], ex)
        contrib = np.zeros_like(out)
        contrib[rows] = w[rows, slots][:, None] * y
        out += contrib
    for sh in shared:
        out += swiglu_ffn(xs, dense_expert(sh))
    if residual:
        out += xs
    return LayerResult(out, logits, idx, w, tok)


def moe_layer_reference_order(x: np.ndarray, w_router: np.ndarray, k: int,
                              expert: Callable[[int], object], shared: Sequence[object] = (),
                              residual: bool = False) -> np.ndarray:
    """The same layer as a token-by-token loop, summing each token's terms in the fixed order
    j = 0..k-1, then the shared experts, then the residual. Used to pin moe_layer on small cases."""
    T, d = x.shape
    xs = x.astype(np.float64)
    logits = router_logits(xs, w_router)
    idx = select_topk(logits, k)
    w = gate_weights(logits, idx)
    out = np.zeros((T, d))
    for t in range(T):
        acc = np.zeros(d)
        for j in range(k):
            acc = acc + w[t, j] * swiglu_ffn(xs[t:t + 1], dense_expert(expert(int(idx[t, j]))))[0]
        for sh in shared:
            acc = acc + swiglu_ffn(xs[t:t + 1], dense_expert(sh))[0]
        if residual:
            acc = acc + xs[t]
        out[t] = acc
    return out


def rms(v: np.ndarray) -> float:
    v = np.asarray(v, dtype=np.float64)
    return float(math.sqrt(np.mean(v * v))) if v.size else 0.0


def logit_gap(logits32: np.ndarray, k: int) -> np.ndarray:
    """Per token, the k-th largest minus the (k+1)-th largest fp32 logit (+inf when k == E)."""
    T, E = logits32.shape
    if k >= E:
        return np.full(T, np.inf)
    s = -np.sort(-logits32.astype(np.float64), axis=1)
    return s[:, k - 1] - s[:, k]
