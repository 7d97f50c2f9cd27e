"""One MoE layer's forward pass through the C-ABI, with its buffers held in torch tensors.

torch provides device memory and streams only. The four calls (moe_route, moe_permute,
moe_expert_ffn, moe_combine) run the whole pass in the library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib as L


@dataclass
class LayerBuffers:
    """Outputs and scratch of one layer pass for a fixed shape."""
    shape: L.moe_shape
    topk_idx: torch.Tensor   # int32 [T][k]
    topk_w: torch.Tensor     # fp32 [T][k]
    logits: torch.Tensor     # fp32 [T][E]
    counts: torch.Tensor     # int32 [E]
    offsets: torch.Tensor    # int32 [E+1]
    sorted_pair: torch.Tensor  # int32 [P]
    inv_pos: torch.Tensor    # int32 [P]
    active: torch.Tensor     # int32 [1 + min(E, P)]
    y_perm: torch.Tensor     # [P + T*n_shared][d]
    out: torch.Tensor        # [T][d]
    ws: torch.Tensor         # uint8 workspace
    ydt: int
    odt: int

    @property
    def ws_bytes(self) -> int:
        return self.ws.numel()


def _dt(code: int) -> torch.dtype:
    return torch.float32 if code == L.MOE_F32 else torch.bfloat16


def alloc_buffers(shape: L.moe_shape, device="cuda", ydt: int = L.MOE_F32, odt: int = L.MOE_BF16,
                  keep_logits: bool = True) -> LayerBuffers:
    T, d, E, k, ns = shape.T, shape.d, shape.E, shape.k, shape.n_shared
    P = T * k
    i32 = dict(dtype=torch.int32, device=device)
    ws_bytes = L.moe_workspace_size(shape)
    return LayerBuffers(
        shape=shape,
        topk_idx=torch.empty((T, k), **i32),
        topk_w=torch.empty((T, k), dtype=torch.float32, device=device),
        logits=torch.empty((T, E) if keep_logits else (0,), dtype=torch.float32, device=device),
        counts=torch.empty(E, **i32),
        offsets=torch.empty(E + 1, **i32),
        sorted_pair=torch.empty(max(P, 1), **i32),
        inv_pos=torch.empty(max(P, 1), **i32),
        active=torch.empty(1 + min(E, max(P, 1)), **i32),
        y_perm=torch.empty((P + T * ns, d), dtype=_dt(ydt), device=device),
        out=torch.empty((T, d), dtype=_dt(odt), device=device),
        # zero-filled once: the decode expert FFN keeps counters here that each call leaves at zero
        ws=torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=device),
        ydt=ydt,
        odt=odt,
    )


def forward(buf: LayerBuffers, x: torch.Tensor, w_router: torch.Tensor, table: L.moe_expert_table,
            mode: int = L.MOE_MODE_AUTO, residual: torch.Tensor | None = None, stream=None,
            fused: bool = False) -> torch.Tensor:
    """Runs route -> permute -> expert FFN -> combine on `stream` as the four separate calls;
    returns buf.out. With fused, the whole pass is one call (moe_layer_forward)."""
    s = buf.shape
    xdt = L.MOE_F32 if x.dtype == torch.float32 else L.MOE_BF16
    logits = buf.logits if buf.logits.numel() else None
    if fused:
        L.moe_layer_forward(s, x, xdt, w_router, table, mode, buf.topk_idx, buf.topk_w, logits, buf.counts,
                            buf.offsets, buf.sorted_pair, buf.inv_pos, buf.active, buf.y_perm, buf.ydt, residual,
                            buf.out, buf.odt, buf.ws, buf.ws_bytes, stream)
        return buf.out
    L.moe_route(s, x, xdt, w_router, buf.topk_idx, buf.topk_w, logits, buf.ws, buf.ws_bytes, stream)
    L.moe_permute(s, buf.topk_idx, buf.counts, buf.offsets, buf.sorted_pair, buf.inv_pos, buf.active, buf.ws,
                  buf.ws_bytes, stream)
    L.moe_expert_ffn(s, mode, x, xdt, table, buf.offsets, buf.sorted_pair, buf.active, buf.y_perm, buf.ydt, buf.ws,
                     buf.ws_bytes, stream)
    L.moe_combine(s, buf.y_perm, buf.ydt, buf.inv_pos, buf.topk_w, residual, buf.out, buf.odt, stream)
    return buf.out
