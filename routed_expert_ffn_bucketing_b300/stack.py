"""Multi-layer drivers over the C-ABI: a decode stack with every expert resident, and a tiered
stack whose experts live in pinned host memory and are cached in a device slot pool.

Both only order the library's calls and hold buffers in torch tensors; every step of every
layer runs in the library's kernels. Each layer is a pre-norm residual block,
x_{l+1} = x_l + MoE_l(n(x_l)) with n the RMS normalisation (no gain, eps 1e-6): moe_rms_norm
writes n(x_l), the layer routes and runs its experts on it, and the combine adds the residual
x_l in fp32 and rounds once to bf16, in place.
"""
from __future__ import annotations

import os
import time

import ctypes as C
from dataclasses import dataclass

import numpy as np
import torch

from . import _lib as L
from . import layer as lay

RMS_EPS = 1e-6


@dataclass
class LayerWeights:
    """Device weights of one layer: router fp32 [d][E], and the expert table the FFN reads."""
    router: torch.Tensor
    table: L.moe_expert_table


class DecodeStack:
    """L MoE layers run one after another on a residual stream of T tokens."""

    def __init__(self, shape: L.moe_shape, layers: list[LayerWeights], device="cuda", native: bool = True):
        self.shape, self.layers = shape, layers
        self.buf = lay.alloc_buffers(shape, device=device, ydt=L.MOE_F32, odt=L.MOE_BF16, keep_logits=False)
        self.resid = torch.empty((shape.T, shape.d), dtype=torch.bfloat16, device=device)
        self.xn = torch.empty_like(self.resid)
        # native: one moe_stack_forward call runs every layer (one chain of programmatic
        # dependents); otherwise a moe_rms_norm and a moe_layer_forward call per layer
        self.native = native

    def forward(self, x: torch.Tensor, stream=None, keep: list | None = None) -> torch.Tensor:
        """Runs every layer on x (bf16 [T][d], left unchanged); returns the residual stream after
        the last layer. With keep (a list), appends a copy of each layer's input and output
        (that runs the per-layer calls)."""
        self.resid.copy_(x)
        s, b = self.shape, self.buf
        if self.native and keep is None:
            L.moe_stack_forward(s, [lw.router for lw in self.layers], [lw.table for lw in self.layers],
                                L.MOE_MODE_AUTO, self.resid, L.MOE_BF16, RMS_EPS, self.xn, b.topk_idx, b.topk_w,
                                b.counts, b.offsets, b.sorted_pair, b.inv_pos, b.active, b.y_perm, b.ydt, b.ws,
                                b.ws_bytes, stream)
            return self.resid
        for lw in self.layers:
            if keep is not None:
                keep.append(("in", self.resid.clone()))
            L.moe_rms_norm(s, self.resid, L.MOE_BF16, self.xn, L.MOE_BF16, RMS_EPS, stream)
            # the whole layer in one call; out aliases the residual: resid <- resid + MoE(n(resid))
            L.moe_layer_forward(s, self.xn, L.MOE_BF16, lw.router, lw.table, L.MOE_MODE_AUTO, b.topk_idx, b.topk_w,
                                None, b.counts, b.offsets, b.sorted_pair, b.inv_pos, b.active, b.y_perm, b.ydt,
                                self.resid, self.resid, L.MOE_BF16, b.ws, b.ws_bytes, stream)
            if keep is not None:
                keep.append(("idx", b.topk_idx.clone()))
                keep.append(("out", self.resid.clone()))
        return self.resid


class TieredStack:
    """L layers whose E routed experts per layer live in pinned host memory; a pool of n_slots
    device slots caches them (the library's slot table, misses copied on a side stream). Shared
    experts stay resident. The replacement policy is LRU, or with policy=MOE_SLOT_FREQ the
    decayed use count (half-life in steps, one step = one pass over the L layers); profile
    (float32 [L*E] use weights) seeds the counts and fills the empty pool before the first step.

    Per layer: route and bucket on the compute stream; read the active list on the host; update
    the slot table (miss copies on the copy stream, `ready` recorded after them). With overlap
    (the default) the expert FFN runs in two calls: the hit experts (those resident before the
    update, listed on the device by moe_filter_resident) and the shared expert are launched right
    after the routing, before the host has read the active list, so they compute during the host's
    wait and the miss copies; the missed experts follow once the compute stream has waited on
    `ready`. Without overlap one FFN call runs after the wait. Then the combine.

    With prefetch (early routing): right after layer l's routing, layer l+1's router is run on
    layer l's normalised input, which is close to layer l+1's own (the residual stream changes
    by one MoE output per layer). Its active list comes back with layer l's, and the experts it
    names that are not resident are copied after layer l's misses (slot_table_prefetch, never
    evicting layer l's experts), so that PCIe works on layer l+1 while layer l computes. Layer
    l+1's expert FFN waits for those copies (an event per layer); where the prediction was
    right its experts are then hits.

    With pcie_frac < 1 (the pages' bandwidth split of the miss path): of a layer's missed experts
    only the first pcie_frac share is copied; the host computes the rest from their pinned
    records (moe_host_expert_ffn) while the GPU runs the others, and their output rows are copied
    into y_perm before the combine. Host-computed experts do not become resident.

    fmt: the record format of every expert (MOE_FMT_INT8, or MOE_FMT_Q2: 2-bit codes, 2.5 bits
    per weight, so that the same pool bytes hold 3.4x more experts and a miss copies 3.4x fewer
    bytes). slot_bytes is at least the format's record size.

    native: forward() runs the library's executor (moe_tiered_forward: the same steps, overlap
    mode, bit for bit, with the per-layer host work in C++) instead of this class's loop; keep,
    prefetch and overlap=False need the loop."""

    def __init__(self, shape: L.moe_shape, n_layers: int, routers: list[torch.Tensor], h_records: list[int],
                 n_slots: int, slot_bytes: int, shared: list[torch.Tensor], device="cuda",
                 policy: int = L.MOE_SLOT_LRU, half_life_steps: float = 50.0, profile=None,
                 fmt: int = L.MOE_FMT_INT8, native: bool = False):
        self.shape, self.L, self.routers = shape, n_layers, routers
        self.fmt = fmt
        self.shape_routed = L.shape(shape.T, shape.d, shape.f, shape.E, shape.k, 0)
        self.n_slots, self.slot_bytes = n_slots, slot_bytes
        self.pool = torch.empty(n_slots * slot_bytes, dtype=torch.uint8, device=device)
        self.slot_of = torch.full((n_layers, shape.E), -1, dtype=torch.int32, device=device)
        self.shared = shared  # per layer: n_shared records (device, uint8)
        self.table = L.slot_table_create(n_layers, shape.E, n_slots, slot_bytes, self.pool, self.slot_of, h_records)
        self.buf = lay.alloc_buffers(shape, device=device, ydt=L.MOE_F32, odt=L.MOE_BF16, keep_logits=False)
        # the missed experts' FFN call has its own shape (no shared expert) and so its own
        # workspace layout: it gets its own zero-filled workspace
        self.ws_miss = torch.zeros(L.moe_workspace_size(self.shape_routed), dtype=torch.uint8, device=device)
        self.resid = torch.empty((shape.T, shape.d), dtype=torch.bfloat16, device=device)
        self.xn = torch.empty_like(self.resid)
        self.copy_stream = torch.cuda.Stream(device)
        self.ready = torch.cuda.Event()
        self.done = torch.cuda.Event()
        # torch creates an event on its first record; the library records `ready` by handle
        self.ready.record(self.copy_stream)
        self.done.record()
        cap = min(shape.E, shape.T * shape.k)
        # pinned lists in the library's active-list form: [count, ids...]
        self.h_active = torch.empty(1 + cap, dtype=torch.int32).pin_memory()
        self.h_hits = torch.zeros(1 + cap, dtype=torch.int32).pin_memory()
        self.h_misses = torch.zeros(1 + cap, dtype=torch.int32).pin_memory()
        self.d_hits = torch.zeros(1 + cap, dtype=torch.int32, device=device)
        self.d_misses = torch.zeros(1 + cap, dtype=torch.int32, device=device)
        self.stats = L.moe_slot_stats()
        self.layer_misses: list[int] = []
        # early routing: the next layer's predicted routing, its own workspace, and the events
        # recorded after each layer's prefetch copies
        self.pbuf = lay.alloc_buffers(shape, device=device, ydt=L.MOE_F32, odt=L.MOE_BF16, keep_logits=False)
        self.h_pred = torch.empty(1 + cap, dtype=torch.int32).pin_memory()
        self.h_pred_idx = torch.empty((shape.T, shape.k), dtype=torch.int32).pin_memory()
        self.h_pf = np.zeros(cap, dtype=np.int32)
        self.pf_ready = [torch.cuda.Event(), torch.cuda.Event()]
        for ev in self.pf_ready:
            ev.record(self.copy_stream)
        self.layer_prefetched: list[int] = []
        # bandwidth split: host copies of the layer input and the bucketing, host output rows
        self.h_records = list(h_records)
        self.h_xn = torch.empty((shape.T, shape.d), dtype=torch.bfloat16).pin_memory()
        self.h_offsets = torch.empty(shape.E + 1, dtype=torch.int32).pin_memory()
        self.h_sorted = torch.empty(max(1, shape.T * shape.k), dtype=torch.int32).pin_memory()
        self.h_y = torch.empty((shape.T * shape.k, shape.d), dtype=torch.float32).pin_memory()
        self.h_slot = np.zeros(cap, dtype=np.int32)
        self.h_upd = np.zeros(cap, dtype=np.int32)
        self.h_host = np.zeros(cap, dtype=np.int32)
        self.layer_host: list[int] = []
        # threads of the host expert FFN: a quarter of the cores stays free for the thread that
        # drives the GPU and the driver's own threads (with every core busy the host FFN ran ~4x slower)
        self.host_threads = max(1, (os.cpu_count() or 1) * 3 // 4)
        self.host_seconds = 0.0  # wall time spent in it, summed over calls
        if policy != L.MOE_SLOT_LRU:
            L.slot_table_set_policy(self.table, policy, half_life_steps * n_layers)
        self.n_warm = 0
        if profile is not None:
            w = np.ascontiguousarray(profile, dtype=np.float32)
            assert w.size == n_layers * shape.E
            self.n_warm = L.slot_table_warm(self.table, w.ctypes.data, self.copy_stream.cuda_stream,
                                            self.ready.cuda_event)
            self.ready.synchronize()
        self.native = None
        self._split = None
        if native:
            self.native = L.moe_tiered_create(shape, n_layers, routers, shared if shape.n_shared else None, self.table,
                                              self.pool, slot_bytes, n_slots, self.slot_of, self.h_records, fmt,
                                              RMS_EPS)
            self.h_layer_misses = np.zeros(n_layers, dtype=np.int32)
            self.h_layer_host = np.zeros(n_layers, dtype=np.int32)

    def status(self) -> int:
        """The device status words of the workspaces, OR-ed (waits for the current stream)."""
        st = L.moe_read_status(self.buf.ws) | L.moe_read_status(self.ws_miss) | L.moe_read_status(self.pbuf.ws)
        if self.native:
            st |= L.moe_tiered_status(self.native)
        return st

    def close(self):
        if getattr(self, "native", None):
            L.moe_tiered_destroy(self.native)
            self.native = None
        if self.table:
            L.slot_table_destroy(self.table)
            self.table = None

    def forward(self, x: torch.Tensor, keep: list | None = None, overlap: bool = True,
                prefetch: bool = False, prefetch_top: int | None = None, pcie_frac: float = 1.0) -> torch.Tensor:
        """prefetch_top: with prefetch, only the first prefetch_top of each token's predicted top-k
        experts (descending logit) are loaded early; all of them when None. pcie_frac: the share of
        each layer's missed experts copied to the device (the rest are computed on the host)."""
        split = pcie_frac < 1.0
        assert not split or overlap, "the bandwidth split runs with overlap"
        s, b = self.shape, self.buf
        stream = torch.cuda.current_stream()
        self.resid.copy_(x)
        if self.native:
            assert keep is None and not prefetch and overlap, "keep, prefetch and overlap=False need the Python loop"
            if self._split != (pcie_frac, self.host_threads):
                L.moe_tiered_set_split(self.native, pcie_frac, self.host_threads)
                self._split = (pcie_frac, self.host_threads)
            L.moe_tiered_forward(self.native, self.resid, stream, self.h_layer_misses.ctypes.data,
                                 self.h_layer_host.ctypes.data)
            self.layer_misses = self.h_layer_misses.tolist()
            self.layer_host = self.h_layer_host.tolist()
            self.layer_prefetched = []
            return self.resid
        self.layer_misses = []
        self.layer_prefetched = []
        self.layer_host = []
        for l in range(self.L):
            if keep is not None:
                keep.append(("in", self.resid.clone()))
            L.moe_rms_norm(s, self.resid, L.MOE_BF16, self.xn, L.MOE_BF16, RMS_EPS, stream)
            L.moe_route_permute(s, self.xn, L.MOE_BF16, self.routers[l], b.topk_idx, b.topk_w, None, b.counts,
                                b.offsets, b.sorted_pair, b.inv_pos, b.active, b.ws, b.ws_bytes, stream)
            early = prefetch and l + 1 < self.L
            if early:  # layer l+1's router on layer l's normalised input
                pb = self.pbuf
                L.moe_route_permute(s, self.xn, L.MOE_BF16, self.routers[l + 1], pb.topk_idx, pb.topk_w, None,
                                    pb.counts, pb.offsets, pb.sorted_pair, pb.inv_pos, pb.active, pb.ws, pb.ws_bytes,
                                    stream)
                if prefetch_top is None:
                    self.h_pred.copy_(pb.active, non_blocking=True)
                else:
                    self.h_pred_idx.copy_(pb.topk_idx, non_blocking=True)
            table = L.expert_table(self.pool, self.slot_bytes, self.n_slots, self.slot_of[l],
                                   self.shared[l] if s.n_shared else None, fmt=self.fmt)
            if overlap:
                if prefetch and l > 0:  # this layer's experts prefetched during the previous layer
                    stream.wait_event(self.pf_ready[l % 2])
                # the experts resident now: the ones the slot update below counts as hits
                L.moe_filter_resident(b.active, self.slot_of[l], s.E, self.d_hits, stream)
            self.h_active.copy_(b.active, non_blocking=True)
            if split:  # what the host needs to compute experts itself
                self.h_xn.copy_(self.xn, non_blocking=True)
                self.h_offsets.copy_(b.offsets, non_blocking=True)
                self.h_sorted.copy_(b.sorted_pair[:s.T * s.k], non_blocking=True)
            # the host needs the active list, and the previous layer's FFN must be done with the
            # slots before any of them is overwritten: one event wait per layer. With overlap, the
            # hit experts' FFN (and the shared expert's), enqueued after the event, runs meanwhile:
            # it reads only slots of this layer's resident experts, which the update never evicts
            self.done.record(stream)
            if overlap:
                L.moe_expert_ffn(s, L.MOE_MODE_AUTO, self.xn, L.MOE_BF16, table, b.offsets, b.sorted_pair,
                                 self.d_hits, b.y_perm, b.ydt, b.ws, b.ws_bytes, stream)
            self.done.synchronize()
            n = int(self.h_active[0])
            hp, mp = self.h_hits.data_ptr(), self.h_misses.data_ptr()
            upd_ptr, n_upd, n_host = self.h_active.data_ptr() + 4, n, 0
            if split and n:
                # the missed experts, in active-list order; the last (1 - pcie_frac) of them stay on the host
                L.slot_table_lookup(self.table, l, upd_ptr, n, self.h_slot.ctypes.data)
                act = self.h_active.numpy()[1:1 + n]
                miss = act[self.h_slot[:n] < 0]
                n_host = int(len(miss) * (1.0 - pcie_frac))
                host_ids = set(miss[len(miss) - n_host:].tolist()) if n_host else set()
                keep_ids = [e for e in act.tolist() if e not in host_ids]
                n_upd = len(keep_ids)
                self.h_upd[:n_upd] = keep_ids
                self.h_host[:n_host] = sorted(host_ids)
                upd_ptr = self.h_upd.ctypes.data
            self.layer_host.append(n_host)
            st = L.slot_table_update(self.table, l, upd_ptr, n_upd, self.copy_stream.cuda_stream,
                                     self.ready.cuda_event, hp + 4, hp, mp + 4, mp, self.stats)
            if st != L.MOE_OK:
                raise L.MoeError(st, "slot_table_update", L.moe_last_error_string())
            n_miss = int(self.h_misses[0])
            self.layer_misses.append(n_miss)
            if early:
                if prefetch_top is None:
                    pp, n_pf = self.h_pred.data_ptr() + 4, int(self.h_pred[0])
                else:  # each token's first prefetch_top predicted experts, in first-seen order
                    ids = dict.fromkeys(self.h_pred_idx.numpy()[:, :prefetch_top].reshape(-1).tolist())
                    n_pf = len(ids)
                    self.h_pf[:n_pf] = list(ids)
                    pp = self.h_pf.ctypes.data
                self.layer_prefetched.append(
                    L.slot_table_prefetch(self.table, l + 1, pp, n_pf, l, self.h_active.data_ptr() + 4, n,
                                          self.copy_stream.cuda_stream, self.pf_ready[(l + 1) % 2].cuda_event))
            # resid <- resid + MoE(n(resid)): the combine is fused into the expert-FFN call where the
            # layer makes only one
            comb = (b.inv_pos, b.topk_w, self.resid, self.resid, L.MOE_BF16)
            if overlap:
                if n_miss:
                    stream.wait_event(self.ready)
                    self.d_misses.copy_(self.h_misses, non_blocking=True)
                    routed = L.expert_table(self.pool, self.slot_bytes, self.n_slots, self.slot_of[l], None,
                                            fmt=self.fmt)
                    # the missed experts only (a shape without the shared expert, already done)
                    L.moe_expert_ffn(self.shape_routed, L.MOE_MODE_AUTO, self.xn, L.MOE_BF16, routed,
                                     b.offsets, b.sorted_pair, self.d_misses, b.y_perm, b.ydt, self.ws_miss,
                                     self.ws_miss.numel(), stream)
                if n_host:
                    # meanwhile the host computes the rest of the misses, then their rows go in
                    ids = self.h_host[:n_host]
                    recs = [self.h_records[l * s.E + int(e)] for e in ids]
                    t0 = time.perf_counter()
                    L.moe_host_expert_ffn(s, self.h_xn.data_ptr(), L.MOE_BF16, recs, ids.ctypes.data, n_host,
                                          self.h_offsets.data_ptr(), self.h_sorted.data_ptr(),
                                          self.h_y.data_ptr(), self.fmt, self.host_threads)
                    self.host_seconds += time.perf_counter() - t0
                    offs = self.h_offsets.numpy()
                    for e in ids:
                        r0, r1 = int(offs[e]), int(offs[e + 1])
                        b.y_perm[r0:r1].copy_(self.h_y[r0:r1], non_blocking=True)
                L.moe_combine(s, b.y_perm, b.ydt, *comb, stream)
            else:
                if prefetch and l > 0:
                    stream.wait_event(self.pf_ready[l % 2])
                stream.wait_event(self.ready)
                L.moe_expert_ffn_combine(s, L.MOE_MODE_AUTO, self.xn, L.MOE_BF16, table, b.offsets, b.sorted_pair,
                                         b.active, b.y_perm, b.ydt, *comb, b.ws, b.ws_bytes, stream)
            if keep is not None:
                keep.append(("idx", b.topk_idx.clone()))
                keep.append(("out", self.resid.clone()))
        return self.resid
