"""Helpers of the GPU parity tests: run one layer through the C-ABI and compare with the oracle."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from oracle import moe_oracle as O
from routed_expert_ffn_bucketing_b300 import _lib as L
from routed_expert_ffn_bucketing_b300 import layer as lay
from synth.device import DeviceLayer
from synth.workloads import Workload

GAP = 1e-4              # index parity holds where the k-th to (k+1)-th logit gap exceeds this
TOL_BF16 = 2e-2         # max |err| <= TOL_BF16 * rms(oracle output), bf16 path
TOL_F32 = 1e-4          # max |err| <= TOL_F32 * rms(oracle output), fp32 debug mode


@dataclass
class GpuRun:
    buf: lay.LayerBuffers
    status: int
    x_np: np.ndarray      # float64 [T][d] (the exact values the GPU saw)


def run_layer(dl: DeviceLayer, batch: int = 0, mode: int = L.MOE_MODE_AUTO, f32: bool = False,
              ydt: int = L.MOE_F32, residual: bool = False, slot_of: torch.Tensor | None = None) -> GpuRun:
    w = dl.w
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    odt = L.MOE_F32 if f32 else L.MOE_BF16
    buf = lay.alloc_buffers(s, ydt=L.MOE_F32 if f32 else ydt, odt=odt)
    x = dl.x(batch, torch.float32 if f32 else torch.bfloat16)
    table = L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of if slot_of is None else slot_of,
                           dl.shared_ptr, fmt=w.fmt)
    lay.forward(buf, x, dl.router, table, mode, residual=x if residual else None)
    status = L.moe_read_status(buf.ws)
    torch.cuda.synchronize()
    x_np = x.float().cpu().numpy().astype(np.float64)
    return GpuRun(buf, status, x_np)


_EXPERTS: dict = {}


def cached_expert(w: Workload, layer: int, e: int):
    key = (w.seed, w.d, w.f, w.expert_sigma, w.fmt, layer, e)
    if key not in _EXPERTS:
        if len(_EXPERTS) > 256:
            _EXPERTS.pop(next(iter(_EXPERTS)))
        _EXPERTS[key] = w.expert(layer, e)
    return _EXPERTS[key]


def oracle_layer(w: Workload, layer: int, x_np: np.ndarray, forced_idx=None, tokens=None, residual=False):
    shared = [cached_expert(w, layer, w.E + s) for s in range(w.n_shared)]

    def expert(e):
        return cached_expert(w, layer, e)
    return O.moe_layer(x_np, w.router(layer), w.k, expert, shared, residual=residual, forced_idx=forced_idx,
                       tokens=tokens)


def check_routing(run: GpuRun, w: Workload, layer: int = 0):
    """Index parity where the gap exceeds GAP; weights against the oracle's gate for the GPU's
    indices; returns (oracle logits fp32, gpu idx)."""
    logits_o = O.router_logits(run.x_np, w.router(layer))
    idx_g = run.buf.topk_idx.cpu().numpy()
    idx_o = O.select_topk(logits_o, w.k)
    gap = O.logit_gap(logits_o, w.k)
    srt = -np.sort(-logits_o.astype(np.float64), axis=1)
    n_checked = 0
    for t in range(w.T):
        if gap[t] > GAP:
            assert set(idx_g[t]) == set(idx_o[t]), (t, idx_g[t], idx_o[t], gap[t])
            n_checked += 1
        # order inside the top-k wherever adjacent selected logits are GAP apart
        for j in range(w.k):
            left = srt[t, j - 1] - srt[t, j] if j > 0 else np.inf
            right = srt[t, j] - srt[t, j + 1] if j + 1 < w.E else np.inf
            if left > GAP and right > GAP:
                assert idx_g[t, j] == idx_o[t, j], (t, j, idx_g[t], idx_o[t])
    wts_o = O.gate_weights(logits_o, idx_g)
    wts_g = run.buf.topk_w.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(wts_g - wts_o)) <= 5e-5, np.max(np.abs(wts_g - wts_o))
    assert np.allclose(wts_g.sum(axis=1), 1.0, atol=1e-5)
    if run.buf.logits.numel():
        # fp32 summation error bound with an addition depth of at most 100 (both router kernels
        # add each logit's 2048 terms in a tree of depth <= 96): |err| <= 100 u sum_i |x_i w_ie|
        lg = run.buf.logits.cpu().numpy().astype(np.float64)
        bound = 100 * 2.0 ** -24 * (np.abs(run.x_np) @ np.abs(w.router(layer).astype(np.float64)))
        assert np.all(np.abs(lg - logits_o) <= bound + 1e-30), np.max(np.abs(lg - logits_o) - bound)
    return logits_o, idx_g, n_checked


def check_bucketing(run: GpuRun, w: Workload):
    idx_g = run.buf.topk_idx.cpu().numpy()
    b = O.bucketing(idx_g, w.E)
    P = w.P
    assert np.array_equal(run.buf.counts.cpu().numpy(), b.counts)
    assert np.array_equal(run.buf.offsets.cpu().numpy(), b.offsets)
    assert np.array_equal(run.buf.sorted_pair.cpu().numpy()[:P], b.sorted_pair)
    assert np.array_equal(run.buf.inv_pos.cpu().numpy()[:P], b.inv_pos)
    act = run.buf.active.cpu().numpy()
    assert act[0] == b.active.size and np.array_equal(act[1:1 + act[0]], b.active)


def check_expert_rows(run: GpuRun, w: Workload, experts, layer: int = 0, tol: float = TOL_BF16,
                      rows: dict | None = None):
    """Whole experts' y_perm rows against the oracle's SwiGLU FFN of the same tokens: for a
    routed expert e < E its rows offsets[e]..offsets[e+1] (tokens sorted_pair // k), for shared
    expert s = e - E its T rows (token order). rows[e] may name a sub-range of an expert's
    rows (relative to its first row). max |y - y_oracle| <= tol * rms(y_oracle) per expert.
    Returns {e: (n_rows, err / rms)}."""
    offs = run.buf.offsets.cpu().numpy()
    sp = run.buf.sorted_pair.cpu().numpy()
    out = {}
    for e in experts:
        e = int(e)
        if e < w.E:
            r0, r1 = int(offs[e]), int(offs[e + 1])
            toks = sp[r0:r1] // w.k
        else:
            r0 = w.P + (e - w.E) * w.T
            r1 = r0 + w.T
            toks = np.arange(w.T)
        if rows and e in rows:
            a, b = rows[e]
            toks = toks[a:b]
            r0, r1 = r0 + a, r0 + b
        assert r1 > r0, (e, r0, r1)
        y = run.buf.y_perm[r0:r1].float().cpu().numpy().astype(np.float64)
        ref = O.swiglu_ffn(run.x_np[toks], O.dense_expert(cached_expert(w, layer, e)))
        err, r = float(np.max(np.abs(y - ref))), O.rms(ref)
        assert err <= tol * r, (e, r1 - r0, err, r)
        out[e] = (r1 - r0, err / r)
    return out


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (8 significant bits)."""
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, e - 8)


def check_output(run: GpuRun, w: Workload, layer: int = 0, f32: bool = False, residual: bool = False,
                 tokens=None):
    """max |out - oracle| <= tol * rms(oracle), with the oracle's exact (float64) output.

    The bf16 output is rounded once, so its error against the exact value includes that
    rounding (at most half a bf16 ulp). Comparing two rounded values instead would turn a
    rounding flip at the largest elements into a whole ulp: 2^-7 relative, which for
    Gaussian-like outputs (max ~ 4.5 rms) is ~2-3.5% of rms on its own. In bf16 mode every
    element of magnitude >= rms must also be the correctly rounded oracle value or one of
    its bf16 neighbours (near zero an ulp is far below the fp32 summation error)."""
    idx_g = run.buf.topk_idx.cpu().numpy()
    ref = oracle_layer(w, layer, run.x_np, forced_idx=idx_g, tokens=tokens, residual=residual)
    out_g = run.buf.out.float().cpu().numpy().astype(np.float64)
    if tokens is not None:
        out_g = out_g[tokens]
    if not ref.out.size:
        return 0.0
    err = np.max(np.abs(out_g - ref.out))
    r = O.rms(ref.out)
    tol = (TOL_F32 if f32 else TOL_BF16) * r
    assert err <= tol, (err, r, err / max(r, 1e-30))
    if not f32:
        rounded = O.round_to_bf16(ref.out)
        big = np.abs(ref.out) >= r
        assert np.all(np.abs(out_g - rounded)[big] <= bf16_ulp(rounded)[big] * 1.0000001)
    return err / max(r, 1e-30)
