"""ctypes binding of libmoe_b300.so (include/moe.h): argument marshalling only.

Every function here has the name of its C entry point and forwards to it. A pointer
argument may be a torch tensor (its data_ptr()), an int (a raw address) or None (NULL). A
stream may be a torch.cuda.Stream, a raw handle (int) or None (the current torch stream).
A negative moe_status raises MoeError with the library's message. Loading fails loudly
when the library has not been built: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK, MOE_EINVAL, MOE_EUNSUPPORTED, MOE_ECUDA, MOE_ENOSLOT, MOE_EDEVICE = 0, -1, -2, -3, -4, -5
MOE_DEV_NAN_LOGIT, MOE_DEV_BAD_EXPERT, MOE_DEV_MISSING_SLOT, MOE_DEV_TIMEOUT, MOE_DEV_BAD_SLOT = 0x1, 0x2, 0x4, 0x8, 0x10
MOE_BF16, MOE_F32 = 0, 1
MOE_MODE_AUTO, MOE_MODE_DECODE, MOE_MODE_PREFILL = 0, 1, 2
MOE_SLOT_LRU, MOE_SLOT_FREQ = 0, 1
MOE_FMT_INT8, MOE_FMT_Q2 = 0, 1

_STATUS_NAMES = {0: "MOE_OK", -1: "MOE_EINVAL", -2: "MOE_EUNSUPPORTED", -3: "MOE_ECUDA", -4: "MOE_ENOSLOT",
                 -5: "MOE_EDEVICE"}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class moe_shape(C.Structure):
    _fields_ = [("T", C.c_int32), ("d", C.c_int32), ("f", C.c_int32), ("E", C.c_int32), ("k", C.c_int32),
                ("n_shared", C.c_int32)]


class moe_expert_layout(C.Structure):
    _fields_ = [(n, C.c_uint64) for n in ("gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s", "record_bytes")]


class moe_expert_table(C.Structure):
    _fields_ = [("pool", C.c_void_p), ("slot_bytes", C.c_uint64), ("slot_of", C.c_void_p), ("shared", C.c_void_p),
                ("n_slots", C.c_uint64), ("format", C.c_uint32)]


class moe_slot_stats(C.Structure):
    _fields_ = [(n, C.c_uint64) for n in ("hits", "misses", "evictions", "bytes_h2d")]


MOE_COPY_FN = C.CFUNCTYPE(C.c_int, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p, C.c_void_p)

_P = C.c_void_p
_SIGS = {
    "moe_get_expert_layout": (C.c_int, [C.c_int32, C.c_int32, C.POINTER(moe_expert_layout)]),
    "moe_get_record_layout": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, C.POINTER(moe_expert_layout)]),
    "moe_workspace_size": (C.c_int, [C.POINTER(moe_shape), C.POINTER(C.c_size_t)]),
    "moe_route": (C.c_int, [C.POINTER(moe_shape), _P, C.c_int, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "moe_permute": (C.c_int, [C.POINTER(moe_shape), _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "moe_route_permute": (C.c_int, [C.POINTER(moe_shape), _P, C.c_int, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                    C.c_size_t, _P]),
    "moe_permute_static": (C.c_int, [C.POINTER(moe_shape), _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_expert_ffn": (C.c_int, [C.POINTER(moe_shape), C.c_int, _P, C.c_int, C.POINTER(moe_expert_table), _P, _P, _P,
                                 _P, C.c_int, _P, C.c_size_t, _P]),
    "moe_combine": (C.c_int, [C.POINTER(moe_shape), _P, C.c_int, _P, _P, _P, _P, C.c_int, _P]),
    "moe_layer_forward": (C.c_int, [C.POINTER(moe_shape), _P, C.c_int, _P, C.POINTER(moe_expert_table), C.c_int, _P, _P,
                                    _P, _P, _P, _P, _P, _P, _P, C.c_int, _P, _P, C.c_int, _P, C.c_size_t, _P]),
    "moe_expert_ffn_combine": (C.c_int, [C.POINTER(moe_shape), C.c_int, _P, C.c_int, C.POINTER(moe_expert_table), _P,
                                         _P, _P, _P, C.c_int, _P, _P, _P, _P, C.c_int, _P, C.c_size_t, _P]),
    "moe_rms_norm": (C.c_int, [C.POINTER(moe_shape), _P, C.c_int, _P, C.c_int, C.c_float, _P]),
    "moe_stack_forward": (C.c_int, [C.POINTER(moe_shape), C.c_int32, _P, C.POINTER(moe_expert_table), C.c_int, _P,
                                    C.c_int, C.c_float, _P, _P, _P, _P, _P, _P, _P, _P, _P, C.c_int, _P, C.c_size_t,
                                    _P]),
    "moe_read_status": (C.c_int, [_P, _P, C.POINTER(C.c_int32)]),
    "moe_set_wait_limit": (C.c_int, [C.c_uint64]),
    "moe_last_error_string": (C.c_char_p, []),
    "slot_table_create": (C.c_int, [C.POINTER(_P), C.c_int32, C.c_int32, C.c_int32, C.c_uint64, _P, _P, _P,
                                    MOE_COPY_FN, _P]),
    "slot_table_update": (C.c_int, [_P, C.c_int32, _P, C.c_int32, _P, _P, _P, _P, _P, _P,
                                    C.POINTER(moe_slot_stats)]),
    "slot_table_set_policy": (C.c_int, [_P, C.c_int32, C.c_double]),
    "slot_table_prefetch": (C.c_int, [_P, C.c_int32, _P, C.c_int32, C.c_int32, _P, C.c_int32, _P, _P, _P]),
    "slot_table_prefetch_stats": (C.c_int, [_P, C.POINTER(C.c_uint64), C.POINTER(C.c_uint64)]),
    "slot_table_warm": (C.c_int, [_P, _P, _P, _P, _P]),
    "slot_table_stats": (C.c_int, [_P, C.POINTER(moe_slot_stats)]),
    "slot_table_lookup": (C.c_int, [_P, C.c_int32, _P, C.c_int32, _P]),
    "moe_host_expert_ffn": (C.c_int, [C.POINTER(moe_shape), _P, C.c_int, _P, _P, C.c_int32, _P, _P, _P, C.c_int32,
                                      C.c_int32]),
    "slot_table_snapshot": (C.c_int, [_P, _P]),
    "slot_table_destroy": (C.c_int, [_P]),
    "moe_filter_resident": (C.c_int, [_P, _P, C.c_int32, _P, _P]),
    "moe_tiered_create": (C.c_int, [C.POINTER(moe_shape), C.c_int32, _P, _P, _P, _P, C.c_uint64, C.c_uint64, _P, _P,
                                    C.c_int32, C.c_float, C.POINTER(_P)]),
    "moe_tiered_set_split": (C.c_int, [_P, C.c_double, C.c_int32]),
    "moe_tiered_forward": (C.c_int, [_P, _P, _P, _P, _P]),
    "moe_tiered_status": (C.c_int, [_P, _P, C.POINTER(C.c_int32)]),
    "moe_tiered_destroy": (C.c_int, [_P]),
}

_lib = None


def lib() -> C.CDLL:
    """The loaded library (loaded on first use)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m routed_expert_ffn_bucketing_b300.build`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def stream_handle(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, where: str) -> int:
    if st < 0:
        raise MoeError(st, where, (lib().moe_last_error_string() or b"").decode())
    return st


def shape(T: int, d: int, f: int, E: int, k: int, n_shared: int = 0) -> moe_shape:
    return moe_shape(T, d, f, E, k, n_shared)


def moe_get_expert_layout(d: int, f: int) -> moe_expert_layout:
    out = moe_expert_layout()
    _check(lib().moe_get_expert_layout(d, f, C.byref(out)), "moe_get_expert_layout")
    return out


def moe_get_record_layout(d: int, f: int, fmt: int) -> moe_expert_layout:
    out = moe_expert_layout()
    _check(lib().moe_get_record_layout(d, f, fmt, C.byref(out)), "moe_get_record_layout")
    return out


def moe_workspace_size(s: moe_shape) -> int:
    n = C.c_size_t()
    _check(lib().moe_workspace_size(C.byref(s), C.byref(n)), "moe_workspace_size")
    return n.value


def moe_route(s, x, xdt, w_router, topk_idx, topk_w, logits_opt, ws, ws_bytes, stream=None) -> int:
    return _check(lib().moe_route(C.byref(s), ptr(x), xdt, ptr(w_router), ptr(topk_idx), ptr(topk_w),
                                  ptr(logits_opt), ptr(ws), ws_bytes, stream_handle(stream)), "moe_route")


def moe_permute(s, topk_idx, counts, offsets, sorted_pair, inv_pos, active, ws, ws_bytes, stream=None) -> int:
    return _check(lib().moe_permute(C.byref(s), ptr(topk_idx), ptr(counts), ptr(offsets), ptr(sorted_pair),
                                    ptr(inv_pos), ptr(active), ptr(ws), ws_bytes, stream_handle(stream)),
                  "moe_permute")


def moe_route_permute(s, x, xdt, w_router, topk_idx, topk_w, logits_opt, counts, offsets, sorted_pair, inv_pos,
                      active, ws, ws_bytes, stream=None) -> int:
    return _check(lib().moe_route_permute(C.byref(s), ptr(x), xdt, ptr(w_router), ptr(topk_idx), ptr(topk_w),
                                          ptr(logits_opt), ptr(counts), ptr(offsets), ptr(sorted_pair), ptr(inv_pos),
                                          ptr(active), ptr(ws), ws_bytes, stream_handle(stream)),
                  "moe_route_permute")


def moe_permute_static(s, topk_idx, counts, offsets, sorted_pair, inv_pos, active, status, stream=None) -> int:
    """moe_permute with the library's fixed scratch instead of a workspace; `status` is a
    device int32 that receives the MOE_DEV_* bits."""
    return _check(lib().moe_permute_static(C.byref(s), ptr(topk_idx), ptr(counts), ptr(offsets), ptr(sorted_pair),
                                           ptr(inv_pos), ptr(active), ptr(status), stream_handle(stream)),
                  "moe_permute_static")


def expert_table(pool, slot_bytes: int, n_slots: int, slot_of, shared=None, fmt: int = MOE_FMT_INT8) -> moe_expert_table:
    return moe_expert_table(ptr(pool), slot_bytes, ptr(slot_of), ptr(shared), n_slots, fmt)


def moe_expert_ffn(s, mode, x, xdt, table: moe_expert_table, offsets, sorted_pair, active, y_perm, ydt, ws,
                   ws_bytes, stream=None) -> int:
    return _check(lib().moe_expert_ffn(C.byref(s), mode, ptr(x), xdt, C.byref(table), ptr(offsets),
                                       ptr(sorted_pair), ptr(active), ptr(y_perm), ydt, ptr(ws), ws_bytes,
                                       stream_handle(stream)), "moe_expert_ffn")


def moe_expert_ffn_combine(s, mode, x, xdt, table: moe_expert_table, offsets, sorted_pair, active, y_perm, ydt,
                           inv_pos, topk_w, residual_opt, out, odt, ws, ws_bytes, stream=None) -> int:
    return _check(lib().moe_expert_ffn_combine(C.byref(s), mode, ptr(x), xdt, C.byref(table), ptr(offsets),
                                               ptr(sorted_pair), ptr(active), ptr(y_perm), ydt, ptr(inv_pos),
                                               ptr(topk_w), ptr(residual_opt), ptr(out), odt, ptr(ws), ws_bytes,
                                               stream_handle(stream)), "moe_expert_ffn_combine")


def moe_layer_forward(s, x, xdt, w_router, table: moe_expert_table, mode, topk_idx, topk_w, logits_opt, counts,
                      offsets, sorted_pair, inv_pos, active, y_perm, ydt, residual_opt, out, odt, ws, ws_bytes,
                      stream=None) -> int:
    return _check(lib().moe_layer_forward(C.byref(s), ptr(x), xdt, ptr(w_router), C.byref(table), mode, ptr(topk_idx),
                                          ptr(topk_w), ptr(logits_opt), ptr(counts), ptr(offsets), ptr(sorted_pair),
                                          ptr(inv_pos), ptr(active), ptr(y_perm), ydt, ptr(residual_opt), ptr(out),
                                          odt, ptr(ws), ws_bytes, stream_handle(stream)), "moe_layer_forward")


def moe_combine(s, y_perm, ydt, inv_pos, topk_w, residual_opt, out, odt, stream=None) -> int:
    return _check(lib().moe_combine(C.byref(s), ptr(y_perm), ydt, ptr(inv_pos), ptr(topk_w), ptr(residual_opt),
                                    ptr(out), odt, stream_handle(stream)), "moe_combine")


def moe_rms_norm(s, x, xdt, out, odt, eps: float, stream=None) -> int:
    return _check(lib().moe_rms_norm(C.byref(s), ptr(x), xdt, ptr(out), odt, C.c_float(eps), stream_handle(stream)),
                  "moe_rms_norm")


def moe_stack_forward(s, routers, tables, mode, resid, rdt, eps: float, xn, topk_idx, topk_w, counts, offsets,
                      sorted_pair, inv_pos, active, y_perm, ydt, ws, ws_bytes, stream=None) -> int:
    """routers: n_layers device tensors (or addresses); tables: n_layers moe_expert_table."""
    n = len(routers)
    if len(tables) != n:
        raise ValueError("moe_stack_forward: routers and tables differ in length")
    r = (C.c_void_p * max(1, n))(*[ptr(x) for x in routers])
    t = (moe_expert_table * max(1, n))(*tables)
    return _check(lib().moe_stack_forward(C.byref(s), n, r, t, mode, ptr(resid), rdt, C.c_float(eps), ptr(xn),
                                          ptr(topk_idx), ptr(topk_w), ptr(counts), ptr(offsets), ptr(sorted_pair),
                                          ptr(inv_pos), ptr(active), ptr(y_perm), ydt, ptr(ws), ws_bytes,
                                          stream_handle(stream)), "moe_stack_forward")


def moe_read_status(ws, stream=None) -> int:
    """Returns the device status word (0 when clean); raises only on MOE_ECUDA / MOE_EINVAL."""
    v = C.c_int32()
    st = lib().moe_read_status(ptr(ws), stream_handle(stream), C.byref(v))
    if st not in (MOE_OK, MOE_EDEVICE):
        _check(st, "moe_read_status")
    return v.value


def moe_set_wait_limit(ns: int) -> None:
    """Limit (ns) of the expert-FFN kernels' bounded waits for later calls; 0 = the 1 s default."""
    _check(lib().moe_set_wait_limit(ns), "moe_set_wait_limit")


def moe_last_error_string() -> str:
    return (lib().moe_last_error_string() or b"").decode()


# ------------------------------------------------------------------ slot table ------------

def slot_table_create(L, E, n_slots, slot_bytes, d_pool, d_slot_of, h_records, copy_fn=None, copy_user=None):
    """h_records: sequence of L*E host addresses (ints). copy_fn: a MOE_COPY_FN or None.
    Returns the opaque handle (int)."""
    arr = (C.c_void_p * (L * E))(*h_records)
    out = C.c_void_p()
    fn = copy_fn if copy_fn is not None else MOE_COPY_FN()
    st = lib().slot_table_create(C.byref(out), L, E, n_slots, slot_bytes, ptr(d_pool), ptr(d_slot_of), arr, fn,
                                 copy_user)
    if st < 0:
        raise MoeError(st, "slot_table_create", moe_last_error_string())
    return out.value


def slot_table_update(table, layer, h_active, n_active, copy_stream, ready, h_hits=None, n_hits=None,
                      h_misses=None, n_misses=None, stats=None) -> int:
    """Pointer arguments are raw host addresses (ints) or None; stats a moe_slot_stats or None."""
    st = lib().slot_table_update(table, layer, h_active, n_active, copy_stream, ready, h_hits, n_hits, h_misses,
                                 n_misses, C.byref(stats) if stats is not None else None)
    if st < 0 and st != MOE_ENOSLOT:
        raise MoeError(st, "slot_table_update", moe_last_error_string())
    return st


def slot_table_prefetch(table, layer: int, h_ids, n_ids: int, keep_layer: int, h_keep, n_keep: int, copy_stream=None,
                        ready=None) -> int:
    """h_ids, h_keep: host addresses (ints) of int32 arrays, or None. Returns the number of
    experts copied."""
    n = C.c_int32()
    _check(lib().slot_table_prefetch(table, layer, h_ids, n_ids, keep_layer, h_keep, n_keep, copy_stream, ready,
                                     C.byref(n)), "slot_table_prefetch")
    return n.value


def slot_table_prefetch_stats(table) -> tuple[int, int]:
    loads, used = C.c_uint64(), C.c_uint64()
    _check(lib().slot_table_prefetch_stats(table, C.byref(loads), C.byref(used)), "slot_table_prefetch_stats")
    return loads.value, used.value


def slot_table_set_policy(table, policy: int, half_life: float) -> None:
    """policy: MOE_SLOT_LRU or MOE_SLOT_FREQ; half_life in slot_table_update calls."""
    _check(lib().slot_table_set_policy(table, policy, half_life), "slot_table_set_policy")


def slot_table_warm(table, h_weight, copy_stream=None, ready=None) -> int:
    """h_weight: host address (int) of float32 [L*E] use weights. Returns the number of
    experts copied into empty slots."""
    n = C.c_int32()
    _check(lib().slot_table_warm(table, h_weight, copy_stream, ready, C.byref(n)), "slot_table_warm")
    return n.value


def slot_table_lookup(table, layer: int, h_ids: int, n: int, h_slot: int) -> None:
    """h_ids, h_slot: host addresses (ints) of int32 arrays of n entries."""
    _check(lib().slot_table_lookup(table, layer, h_ids, n, h_slot), "slot_table_lookup")


def moe_host_expert_ffn(s, h_x, xdt, h_records, h_experts, n_experts, h_offsets, h_sorted_pair, h_y, fmt=MOE_FMT_INT8,
                        n_threads=0) -> None:
    """All pointers are host addresses (ints); h_records: a sequence of n_experts addresses."""
    recs = (C.c_void_p * max(1, n_experts))(*h_records)
    _check(lib().moe_host_expert_ffn(C.byref(s), h_x, xdt, recs, h_experts, n_experts, h_offsets, h_sorted_pair, h_y,
                                     fmt, n_threads), "moe_host_expert_ffn")


def slot_table_stats(table) -> moe_slot_stats:
    out = moe_slot_stats()
    _check(lib().slot_table_stats(table, C.byref(out)), "slot_table_stats")
    return out


def slot_table_snapshot(table, h_out) -> None:
    _check(lib().slot_table_snapshot(table, h_out), "slot_table_snapshot")


def slot_table_destroy(table) -> None:
    _check(lib().slot_table_destroy(table), "slot_table_destroy")


def moe_tiered_create(s, n_layers, routers, shared, table, pool, slot_bytes, n_slots, slot_of, h_records,
                      fmt=MOE_FMT_INT8, eps=1e-6) -> int:
    """routers / shared: sequences of n_layers device tensors or addresses (shared may be None
    when s.n_shared == 0); h_records: n_layers * E host addresses. Returns the opaque handle."""
    r = (C.c_void_p * n_layers)(*[ptr(x) for x in routers])
    sh = (C.c_void_p * n_layers)(*[ptr(x) for x in shared]) if shared is not None else None
    rec = (C.c_void_p * len(h_records))(*h_records)
    out = C.c_void_p()
    _check(lib().moe_tiered_create(C.byref(s), n_layers, r, sh, table, ptr(pool), slot_bytes, n_slots, ptr(slot_of),
                                   rec, fmt, eps, C.byref(out)), "moe_tiered_create")
    return out.value


def moe_tiered_set_split(t, pcie_frac: float, host_threads: int = 0) -> int:
    return _check(lib().moe_tiered_set_split(t, pcie_frac, host_threads), "moe_tiered_set_split")


def moe_tiered_forward(t, resid, stream=None, h_layer_misses=None, h_layer_host=None) -> int:
    return _check(lib().moe_tiered_forward(t, ptr(resid), stream_handle(stream), h_layer_misses, h_layer_host),
                  "moe_tiered_forward")


def moe_tiered_status(t, stream=None) -> int:
    v = C.c_int32()
    st = lib().moe_tiered_status(t, stream_handle(stream), C.byref(v))
    if st not in (MOE_OK, MOE_EDEVICE):
        _check(st, "moe_tiered_status")
    return v.value


def moe_tiered_destroy(t) -> int:
    return _check(lib().moe_tiered_destroy(t), "moe_tiered_destroy")


def moe_filter_resident(active, slot_of_row, E: int, out, stream=None) -> int:
    return _check(lib().moe_filter_resident(ptr(active), ptr(slot_of_row), E, ptr(out), stream_handle(stream)),
                  "moe_filter_resident")
