"""GPU parity of the whole layer pass through the C-ABI against the CPU oracle, on the same
seeded inputs: routing (indices where the logit gap allows, weights), bucketing (bit-exact),
outputs (bf16: max |err| <= 2e-2 rms; fp32 debug mode: <= 1e-4 rms), and edge cases."""
import numpy as np
import pytest
import torch

import synth
from oracle import moe_oracle as O
from routed_expert_ffn_bucketing_b300 import _lib as L
from synth.device import DeviceLayer
from synth.workloads import WORKLOADS, custom

from gpu_util import GpuRun, check_bucketing, check_expert_rows, check_output, check_routing, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    return DeviceLayer(WORKLOADS["tiny"])


@pytest.fixture(scope="module")
def decode():
    return DeviceLayer(WORKLOADS["decode"])


def test_device_generator_matches_numpy():
    w = custom("decode", E=3, n_shared=1)
    dl = DeviceLayer(w, layer=5)
    for e in range(4):
        assert np.array_equal(dl.record_bytes_of(e), synth.pack_record(w.expert(5, e))), e
    w1 = WORKLOADS["tiny"]
    dl1 = DeviceLayer(w1)
    for e in (0, 7, 15):
        assert np.array_equal(dl1.record_bytes_of(e), synth.pack_record(w1.expert(0, e)))


def test_tiny_layer_bf16(tiny):
    for batch in range(3):
        run = run_layer(tiny, batch)
        assert run.status == 0
        check_routing(run, tiny.w)
        check_bucketing(run, tiny.w)
        check_output(run, tiny.w)


def test_tiny_layer_fp32_debug(tiny):
    run = run_layer(tiny, 1, f32=True)
    assert run.status == 0
    check_routing(run, tiny.w)
    check_bucketing(run, tiny.w)
    check_output(run, tiny.w, f32=True)


def test_tiny_layer_residual_and_bf16_y(tiny):
    run = run_layer(tiny, 2, residual=True, ydt=L.MOE_BF16)
    check_output(run, tiny.w, residual=True)


def test_decode_layer_full_size(decode):
    w = decode.w
    # the oracle sees the bytes the GPU holds, for every expert it uses
    for batch in range(2):
        run = run_layer(decode, batch)
        assert run.status == 0
        _, idx_g, n_checked = check_routing(run, w)
        assert n_checked == w.T
        check_bucketing(run, w)
        for e in list(np.unique(idx_g)[:3]) + [w.E]:
            assert np.array_equal(decode.record_bytes_of(int(e)), synth.pack_record(w.expert(0, int(e))))
        check_output(run, w)


def test_decode_layer_fp32_debug(decode):
    run = run_layer(decode, 3, f32=True)
    check_routing(run, decode.w)
    check_output(run, decode.w, f32=True)


@pytest.mark.parametrize("T,E,k,ns", [(1, 16, 2, 0), (3, 8, 8, 1), (16, 1, 1, 0), (7, 40, 5, 2), (16, 64, 32, 0)])
def test_small_shapes(T, E, k, ns):
    w = custom("tiny", T=T, E=E, k=k, n_shared=ns, d=96, f=64, router_sigma=1.0)
    dl = DeviceLayer(w, fill="host")
    run = run_layer(dl, 0)
    assert run.status == 0
    check_routing(run, w)
    check_bucketing(run, w)
    check_output(run, w)


@pytest.mark.parametrize("T", [17, 300])
def test_router_gemm_and_multichunk_bucketing(T):
    # T > 16 takes the tiled router GEMM; T*k > 1024 takes the multi-chunk bucketing
    w = custom("tiny", T=T, E=64, k=10, n_shared=1, router_sigma=1.0)
    dl = DeviceLayer(w)
    run = run_layer(dl, 0, mode=L.MOE_MODE_DECODE)
    assert run.status == 0
    check_routing(run, w)
    check_bucketing(run, w)
    check_output(run, w, tokens=np.arange(0, T, 7))


def test_empty_batch(tiny):
    w = custom("tiny", T=0)
    dl = DeviceLayer(w)
    run = run_layer(dl, 0)
    assert run.status == 0
    assert run.buf.active.cpu().numpy()[0] == 0
    assert np.all(run.buf.offsets.cpu().numpy() == 0)


def test_exact_ties_go_to_lowest_index():
    w = custom("tiny", T=8, E=32, k=4, router_sigma=1.0)
    dl = DeviceLayer(w)
    r = dl.router.clone()
    r[:, 20] = r[:, 3]     # experts 3 and 20 always tie exactly; so do 5, 6 and 30
    r[:, 6] = r[:, 5]
    r[:, 30] = r[:, 5]
    dl.router = r
    run = run_layer(dl, 0)
    idx = run.buf.topk_idx.cpu().numpy()
    for t in range(w.T):
        s = set(idx[t])
        assert not (20 in s and 3 not in s)
        assert not (6 in s and 5 not in s) and not (30 in s and 6 not in s)
    lg = run.buf.logits.cpu().numpy()
    assert np.all(lg[:, 3] == lg[:, 20]) and np.all(lg[:, 5] == lg[:, 30])
    # the GPU's selection equals the oracle's rule applied to the GPU's own (exactly tied) logits
    assert np.array_equal(idx, O.select_topk(lg, w.k))


def test_missing_slot_sets_status_and_skips(tiny):
    so = tiny.slot_of.clone()
    so[:] = -1
    run = run_layer(tiny, 0, slot_of=so)
    assert run.status & L.MOE_DEV_MISSING_SLOT


def test_bad_expert_index_sets_status(tiny):
    w = tiny.w
    s = L.shape(w.T, w.d, w.f, w.E, w.k, 0)
    from routed_expert_ffn_bucketing_b300 import layer as lay
    buf = lay.alloc_buffers(s)
    idx = torch.zeros((w.T, w.k), dtype=torch.int32, device="cuda")
    idx[:, 1] = 1
    idx[3, 0] = w.E + 5
    torch.cuda.synchronize()
    L.moe_route(s, tiny.x(0), L.MOE_BF16, tiny.router, buf.topk_idx, buf.topk_w, None, buf.ws, buf.ws_bytes)
    L.moe_permute(s, idx, buf.counts, buf.offsets, buf.sorted_pair, buf.inv_pos, buf.active, buf.ws, buf.ws_bytes)
    assert L.moe_read_status(buf.ws) & L.MOE_DEV_BAD_EXPERT


def test_nan_logit_sets_status(tiny):
    w = tiny.w
    s = L.shape(w.T, w.d, w.f, w.E, w.k, 0)
    from routed_expert_ffn_bucketing_b300 import layer as lay
    buf = lay.alloc_buffers(s)
    r = tiny.router.clone()
    r[0, 4] = float("nan")
    L.moe_route(s, tiny.x(0), L.MOE_BF16, r, buf.topk_idx, buf.topk_w, None, buf.ws, buf.ws_bytes)
    assert L.moe_read_status(buf.ws) & L.MOE_DEV_NAN_LOGIT
    assert not np.any(buf.topk_idx.cpu().numpy() == 4)


def test_deterministic(decode):
    a = run_layer(decode, 5)
    b = run_layer(decode, 5)
    assert torch.equal(a.buf.out, b.buf.out) and torch.equal(a.buf.topk_w, b.buf.topk_w)


@pytest.mark.parametrize("T,E,k,ns", [(300, 64, 10, 1), (200, 16, 2, 0), (97, 8, 8, 2)])
def test_prefill_gemm_small(T, E, k, ns):
    # the tensor-core grouped GEMM on shapes with partial 128-row tiles, several experts with
    # more than one tile and experts with one token
    w = custom("tiny", T=T, E=E, k=k, n_shared=ns, router_sigma=1.0)
    dl = DeviceLayer(w)
    run = run_layer(dl, 0, mode=L.MOE_MODE_PREFILL)
    assert run.status == 0
    check_routing(run, w)
    check_bucketing(run, w)
    check_output(run, w, tokens=np.arange(0, T, 3))


def test_prefill_gemm_matches_decode_kernels():
    # the same layer through the prefill GEMM and through the decode kernels: both within the
    # tolerance of the oracle, and within 2e-2 rms of each other everywhere
    w = custom("tiny", T=64, E=32, k=4, n_shared=1, router_sigma=1.0)
    dl = DeviceLayer(w)
    a = run_layer(dl, 0, mode=L.MOE_MODE_PREFILL)
    b = run_layer(dl, 0, mode=L.MOE_MODE_DECODE)
    assert torch.equal(a.buf.topk_idx, b.buf.topk_idx)
    oa, ob = a.buf.out.float(), b.buf.out.float()
    rms = float(torch.sqrt(torch.mean(ob * ob)))
    assert float(torch.max(torch.abs(oa - ob))) <= 2e-2 * rms
    check_output(a, w)


def test_prefill_layer_full_size():
    # the prefill chunk: T = 8192 tokens, Zipf(1.1) routing, tiles from one token to thousands;
    # routing and bucketing are checked for every token, outputs on a sample of tokens
    w = WORKLOADS["prefill"]
    dl = DeviceLayer(w)
    run = run_layer(dl, 0)  # AUTO takes the tensor-core GEMM for T > 16
    assert run.status == 0
    _, _, n_checked = check_routing(run, w)
    assert n_checked >= w.T - 8
    check_bucketing(run, w)
    check_output(run, w, tokens=np.array([0, 1, 77, 1023, 3333, 4096, 5000, 8191]))
    # whole experts' rows of y_perm, chosen to cover the GEMM's tile walk at full size (12
    # chunks of 64 columns of gate/up at f = 768, 16 of 128 rows of down at d = 2048): the
    # heaviest Zipf expert (every one of its 128-row token tiles, the partial last one
    # included), a mid-rank expert, the three experts with the fewest rows (one partial token
    # tile each, N of 16), the last three experts of the tile list, and the shared expert's
    # first and last token tiles
    counts = run.buf.counts.cpu().numpy()
    act = np.nonzero(counts)[0]
    heavy = int(act[np.argmax(counts[act])])
    assert counts[heavy] > 4 * 128 and counts[heavy] % 128, counts[heavy]
    by_count = act[np.argsort(counts[act], kind="stable")]
    mid = int(by_count[by_count.size // 2])
    fewest = [int(e) for e in by_count[:3]]
    last = [int(e) for e in act[-3:]]
    assert max(counts[fewest]) < 128
    shared = w.E
    got = check_expert_rows(run, w, sorted({heavy, mid, *fewest, *last}) + [shared],
                            rows={shared: (w.T - 128 - 64, w.T)})
    got.update(check_expert_rows(run, w, [shared], rows={shared: (0, 128)}))
    assert got[heavy][0] == counts[heavy]


@pytest.mark.parametrize("wl,mode,residual,odt,ydt", [
    ("decode", L.MOE_MODE_AUTO, False, L.MOE_BF16, L.MOE_F32),
    ("decode", L.MOE_MODE_AUTO, True, L.MOE_BF16, L.MOE_F32),
    ("decode", L.MOE_MODE_AUTO, True, L.MOE_F32, L.MOE_BF16),
    ("tiny", L.MOE_MODE_AUTO, True, L.MOE_BF16, L.MOE_F32),      # T = 16: separate launches
    ("tiny", L.MOE_MODE_PREFILL, False, L.MOE_BF16, L.MOE_BF16),
])
def test_fused_combine_is_bit_identical(wl, mode, residual, odt, ydt):
    # moe_expert_ffn_combine against moe_expert_ffn followed by moe_combine: the same bits
    from routed_expert_ffn_bucketing_b300 import layer as lay
    w = WORKLOADS[wl] if wl != "decode" else custom("decode", T=4)
    dl = DeviceLayer(w)
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    x = dl.x(3)
    table = L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of, dl.shared_ptr)
    outs = []
    for fused in (False, True):
        buf = lay.alloc_buffers(s, ydt=ydt, odt=odt, keep_logits=False)
        res = x.float().to(torch.float32 if odt == L.MOE_F32 else torch.bfloat16).contiguous() if residual else None
        L.moe_route(s, x, L.MOE_BF16, dl.router, buf.topk_idx, buf.topk_w, None, buf.ws, buf.ws_bytes)
        L.moe_permute(s, buf.topk_idx, buf.counts, buf.offsets, buf.sorted_pair, buf.inv_pos, buf.active, buf.ws,
                      buf.ws_bytes)
        if fused:
            L.moe_expert_ffn_combine(s, mode, x, L.MOE_BF16, table, buf.offsets, buf.sorted_pair, buf.active, buf.y_perm,
                                     buf.ydt, buf.inv_pos, buf.topk_w, res, buf.out, buf.odt, buf.ws, buf.ws_bytes)
        else:
            L.moe_expert_ffn(s, mode, x, L.MOE_BF16, table, buf.offsets, buf.sorted_pair, buf.active, buf.y_perm,
                             buf.ydt, buf.ws, buf.ws_bytes)
            L.moe_combine(s, buf.y_perm, buf.ydt, buf.inv_pos, buf.topk_w, res, buf.out, buf.odt)
        assert L.moe_read_status(buf.ws) == 0
        torch.cuda.synchronize()
        outs.append(buf.out.clone())
    assert torch.equal(outs[0], outs[1])
    # and in place (out aliases the residual), as the stacks use it
    if residual:
        buf = lay.alloc_buffers(s, ydt=ydt, odt=odt, keep_logits=False)
        r = x.float().to(torch.float32 if odt == L.MOE_F32 else torch.bfloat16).contiguous()
        L.moe_route(s, x, L.MOE_BF16, dl.router, buf.topk_idx, buf.topk_w, None, buf.ws, buf.ws_bytes)
        L.moe_permute(s, buf.topk_idx, buf.counts, buf.offsets, buf.sorted_pair, buf.inv_pos, buf.active, buf.ws,
                      buf.ws_bytes)
        L.moe_expert_ffn_combine(s, mode, x, L.MOE_BF16, table, buf.offsets, buf.sorted_pair, buf.active, buf.y_perm,
                                 buf.ydt, buf.inv_pos, buf.topk_w, r, r, buf.odt, buf.ws, buf.ws_bytes)
        torch.cuda.synchronize()
        assert torch.equal(r, outs[1])


@pytest.mark.parametrize("wl,T,E,k", [("decode", 4, 512, 10), ("decode", 1, 512, 10), ("decode", 16, 512, 10),
                                      ("tiny", 16, 16, 2), ("tiny", 7, 40, 5), ("decode", 16, 1024, 32),
                                      ("tiny", 300, 64, 10), ("decode", 8, 512, 32), ("tiny", 3, 36, 7)])
def test_route_permute_is_bit_identical(wl, T, E, k):
    # moe_route_permute against moe_route followed by moe_permute: the same bits in every output,
    # on shapes inside the one-kernel tail (T <= 8, T*k <= 256), at its edges and beyond it; the
    # tail's block-wide selection with its largest candidate table (16 warps x k = 32) and with a
    # warp holding fewer experts than k (E = 36)
    from routed_expert_ffn_bucketing_b300 import layer as lay
    w = custom(wl, T=T, E=E, k=k, n_shared=0, router_sigma=1.0)
    dl = DeviceLayer(w, fill="host" if w.d * w.f * (w.E + w.n_shared) < (1 << 26) else "device")
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    x = dl.x(1)
    outs = []
    for fused in (False, True):
        buf = lay.alloc_buffers(s)
        if fused:
            L.moe_route_permute(s, x, L.MOE_BF16, dl.router, buf.topk_idx, buf.topk_w, buf.logits, buf.counts,
                                buf.offsets, buf.sorted_pair, buf.inv_pos, buf.active, buf.ws, buf.ws_bytes)
        else:
            L.moe_route(s, x, L.MOE_BF16, dl.router, buf.topk_idx, buf.topk_w, buf.logits, buf.ws, buf.ws_bytes)
            L.moe_permute(s, buf.topk_idx, buf.counts, buf.offsets, buf.sorted_pair, buf.inv_pos, buf.active,
                          buf.ws, buf.ws_bytes)
        assert L.moe_read_status(buf.ws) == 0
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (buf.topk_idx, buf.topk_w, buf.logits, buf.counts, buf.offsets,
                                         buf.sorted_pair, buf.inv_pos)] + [buf.active[:1 + int(buf.active[0])].clone()])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    run = GpuRunLike(outs[1], dl)
    check_routing(run, w)
    check_bucketing(run, w)


class GpuRunLike:
    """The fields of a GpuRun that check_routing and check_bucketing read."""

    def __init__(self, o, dl):
        from types import SimpleNamespace
        self.buf = SimpleNamespace(topk_idx=o[0], topk_w=o[1], logits=o[2], counts=o[3], offsets=o[4],
                                   sorted_pair=o[5], inv_pos=o[6], active=o[7])
        self.x_np = dl.x(1).float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("wl,T", [("decode", 4), ("decode", 1), ("tiny", 16), ("tiny", 300)])
def test_layer_forward_is_bit_identical(wl, T):
    # moe_layer_forward (one call; the decode expert FFN a programmatic dependent of the
    # bucketing) against moe_route, moe_permute, moe_expert_ffn and moe_combine
    from routed_expert_ffn_bucketing_b300 import layer as lay
    w = custom(wl, T=T, router_sigma=1.0)
    dl = DeviceLayer(w)
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    table = L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of, dl.shared_ptr)
    outs = []
    for fused in (False, True):
        buf = lay.alloc_buffers(s, ydt=L.MOE_F32, odt=L.MOE_BF16)
        for batch in range(3):  # repeated calls on one workspace
            lay.forward(buf, dl.x(batch), dl.router, table, fused=fused)
        assert L.moe_read_status(buf.ws) == 0
        torch.cuda.synchronize()
        outs.append((buf.out.clone(), buf.topk_idx.clone(), buf.y_perm.clone()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_expert_ffn_on_a_sparse_subset_of_experts():
    # the active list may be any subset of the routed experts (a slot table's misses, say): their
    # rows lie scattered among the other experts' rows. Every other expert of the full decode layer,
    # then the complement, each into y_perm; together they equal one call on the whole list
    from routed_expert_ffn_bucketing_b300 import layer as lay
    w = custom("decode", T=4)
    dl = DeviceLayer(w)
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    s0 = L.shape(w.T, w.d, w.f, w.E, w.k, 0)
    table = L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of, dl.shared_ptr)
    routed = L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of, None)
    buf = lay.alloc_buffers(s)
    x = dl.x(5)
    L.moe_route_permute(s, x, L.MOE_BF16, dl.router, buf.topk_idx, buf.topk_w, None, buf.counts, buf.offsets,
                        buf.sorted_pair, buf.inv_pos, buf.active, buf.ws, buf.ws_bytes)
    L.moe_expert_ffn(s, L.MOE_MODE_AUTO, x, L.MOE_BF16, table, buf.offsets, buf.sorted_pair, buf.active, buf.y_perm,
                     buf.ydt, buf.ws, buf.ws_bytes)
    torch.cuda.synchronize()
    assert L.moe_read_status(buf.ws) == 0
    full = buf.y_perm.clone()
    act = buf.active.cpu().numpy()
    ids = act[1:1 + act[0]]
    ws2 = torch.zeros(L.moe_workspace_size(s0), dtype=torch.uint8, device="cuda")
    buf.y_perm.zero_()
    for part in (ids[::2], ids[1::2]):
        sub = torch.tensor(np.concatenate([[part.size], part]).astype(np.int32), device="cuda")
        L.moe_expert_ffn(s0, L.MOE_MODE_AUTO, x, L.MOE_BF16, routed, buf.offsets, buf.sorted_pair, sub, buf.y_perm,
                         buf.ydt, ws2, ws2.numel())
        torch.cuda.synchronize()
        assert L.moe_read_status(ws2) == 0
    P = w.P
    # the same rows as the full call up to the order of fp32 additions (stream-K cuts differ, which
    # can flip the f16 rounding of an h element: ~2^-11 of it)...
    assert float(torch.max(torch.abs(buf.y_perm[:P] - full[:P]))) <= 1e-4 * float(torch.max(torch.abs(full[:P])))
    # ...and every routed expert's rows against the oracle
    run = GpuRun(buf, 0, x.float().cpu().numpy().astype(np.float64))
    check_expert_rows(run, w, ids)



@pytest.mark.parametrize("n,E", [(0, 16), (5, 16), (40, 512), (77, 512), (300, 1024)])
def test_filter_resident_keeps_order_and_drops_missing(n, E):
    # moe_filter_resident against the plain filter on the host: the active experts whose slot is
    # >= 0, in active-list order, counted in element 0 (several 32-entry chunks for n > 32)
    rng = np.random.default_rng(n + E)
    ids = rng.choice(E, size=n, replace=False).astype(np.int32)
    slot = np.where(rng.random(E) < 0.6, rng.integers(0, 1000, E), -1).astype(np.int32)
    active = torch.tensor(np.concatenate([[n], ids]).astype(np.int32), device="cuda")
    d_slot = torch.tensor(slot, device="cuda")
    out = torch.full((1 + max(n, 1),), -7, dtype=torch.int32, device="cuda")
    L.moe_filter_resident(active, d_slot, E, out)
    torch.cuda.synchronize()
    want = [int(e) for e in ids if slot[e] >= 0]
    got = out.cpu().numpy()
    assert got[0] == len(want)
    assert got[1:1 + len(want)].tolist() == want
    with pytest.raises(L.MoeError):
        L.moe_filter_resident(active, d_slot, E, active)
