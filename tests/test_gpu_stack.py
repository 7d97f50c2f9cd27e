"""Multi-layer runs through the C-ABI: a decode stack with every expert resident (pre-norm
residual blocks, Zipf(1.1) routing), and a tiered stack whose experts are cached in a device
slot pool smaller than the set of experts, filled from pinned host memory. Every layer is
compared with the oracle given that layer's actual (bf16) input and the GPU's routing. The
RMS normalisation call is checked on its own against the oracle."""
import ctypes as C

import numpy as np
import pytest
import torch

import synth
from oracle import moe_oracle as O
from routed_expert_ffn_bucketing_b300 import _lib as L
from routed_expert_ffn_bucketing_b300.stack import DecodeStack, LayerWeights, TieredStack
from synth.device import DeviceLayer
from synth.workloads import custom

from gpu_util import TOL_BF16, cached_expert

pytestmark = pytest.mark.gpu


def check_layers(w, keep, layers):
    """keep: the ('in', x), ('idx', topk), ('out', y) records of a stack run. Each layer is
    x + MoE(bf16(n(x))) with n the oracle's RMS normalisation: the normalised input is a bf16
    activation tensor like every layer input, so the oracle rounds it once to bf16 (its own
    rounding, pinned on its own) before routing and the experts. Without that rounding the
    gate weights alone differ by about 2^-9 of a logit's size (logits of tens), which moves
    outputs by up to a few percent of their rms."""
    recs = [keep[i:i + 3] for i in range(0, len(keep), 3)]
    assert len(recs) == len(layers)
    for l, (a, b, c) in zip(layers, recs):
        assert a[0] == "in" and b[0] == "idx" and c[0] == "out"
        x_np = a[1].float().cpu().numpy().astype(np.float64)
        idx = b[1].cpu().numpy()
        shared = [cached_expert(w, l, w.E + s) for s in range(w.n_shared)]
        xn = O.round_to_bf16(O.rms_norm(x_np))
        moe = O.moe_layer(xn, w.router(l), w.k, lambda e: cached_expert(w, l, e), shared, forced_idx=idx)
        ref = x_np + moe.out
        out = c[1].float().cpu().numpy().astype(np.float64)
        err, r = np.max(np.abs(out - ref)), O.rms(ref)
        assert err <= TOL_BF16 * r, (l, err, r)


@pytest.mark.parametrize("T,d", [(1, 32), (5, 2080), (4, 2048), (3, 4096)])
@pytest.mark.parametrize("xdt,odt", [(L.MOE_BF16, L.MOE_BF16), (L.MOE_F32, L.MOE_F32), (L.MOE_BF16, L.MOE_F32)])
def test_rms_norm_matches_oracle(T, d, xdt, odt):
    g = torch.Generator().manual_seed(T * 7919 + d)
    x = torch.randn((T, d), generator=g) * torch.logspace(-3, 3, T)[:, None]
    x = x.to(torch.bfloat16 if xdt == L.MOE_BF16 else torch.float32)
    xd = x.cuda()
    out = torch.empty((T, d), dtype=torch.bfloat16 if odt == L.MOE_BF16 else torch.float32, device="cuda")
    s = L.shape(T, d, 32, 4, 1, 0)
    L.moe_rms_norm(s, xd, xdt, out, odt, 1e-6)
    got = out.float().cpu().numpy().astype(np.float64)
    ref = O.rms_norm(x.float().numpy().astype(np.float64), eps=1e-6)
    if odt == L.MOE_F32:
        assert np.max(np.abs(got - ref)) <= 1e-5 * np.max(np.abs(ref))
    else:
        # one bf16 rounding of an fp32 value within 1e-6 of the exact one: at most one bf16 step
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) * 1.001)
    # in place
    if xdt == odt:
        y = xd.clone()
        L.moe_rms_norm(s, y, xdt, y, odt, 1e-6)
        assert torch.equal(y, out)


def test_rms_norm_argument_errors():
    s = L.shape(2, 64, 32, 4, 1, 0)
    x = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.MoeError):
        L.moe_rms_norm(s, x, L.MOE_BF16, x, L.MOE_BF16, -1.0)
    with pytest.raises(L.MoeError):
        L.moe_rms_norm(s, x, L.MOE_BF16, x, L.MOE_F32, 1e-6)
    L.moe_rms_norm(L.shape(0, 64, 32, 4, 1, 0), None, L.MOE_BF16, None, L.MOE_BF16, 1e-6)  # T == 0: nothing to do
    z = torch.zeros((2, 64), dtype=torch.float32, device="cuda")
    L.moe_rms_norm(s, z, L.MOE_F32, z, L.MOE_F32, 1e-6)
    assert torch.equal(z, torch.zeros_like(z))


def test_decode_stack_layer_by_layer():
    w = custom("stack", d=256, f=128, E=32, k=4, layers=3)
    dls = [DeviceLayer(w, layer=l) for l in range(w.layers)]
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    layers = [LayerWeights(dl.router, L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of, dl.shared_ptr))
              for dl in dls]
    st = DecodeStack(s, layers)
    keep = []
    st.forward(dls[0].x(0), keep=keep)
    assert L.moe_read_status(st.buf.ws) == 0
    torch.cuda.synchronize()
    check_layers(w, keep, range(w.layers))


def test_decode_stack_full_shape_three_layers():
    # three consecutive layers of the 48-layer stack at its real shape (d = 2048, f = 768,
    # E = 512, top-10 + 1 shared, Zipf(1.1) routing), each against the oracle on its own input
    w = custom("stack", layers=3)
    dls = [DeviceLayer(w, layer=l) for l in range(w.layers)]
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    layers = [LayerWeights(dl.router, L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of, dl.shared_ptr))
              for dl in dls]
    st = DecodeStack(s, layers)
    for batch in (0, 1):
        keep = []
        st.forward(dls[0].x(batch), keep=keep)
        assert L.moe_read_status(st.buf.ws) == 0
        torch.cuda.synchronize()
        check_layers(w, keep, range(w.layers))


def _stack_layers(w):
    dls = [DeviceLayer(w, layer=l) for l in range(w.layers)]
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    layers = [LayerWeights(dl.router, L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of, dl.shared_ptr))
              for dl in dls]
    return dls, s, layers


@pytest.mark.parametrize("full", [False, True])
def test_stack_forward_is_bit_identical_to_layer_calls(full):
    # moe_stack_forward (one chain of programmatic dependents over all layers) against the
    # per-layer moe_rms_norm + moe_layer_forward calls, whose layers the oracle checks above: the
    # same residual stream, routing and bucketing, bit for bit
    w = custom("stack", layers=3) if full else custom("stack", d=256, f=128, E=32, k=4, layers=3)
    dls, s, layers = _stack_layers(w)
    per_layer = DecodeStack(s, layers, native=False)
    chain = DecodeStack(s, layers, native=True)
    for batch in (0, 1, 2):
        x = dls[0].x(batch)
        want = per_layer.forward(x).clone()
        got = chain.forward(x).clone()
        assert L.moe_read_status(chain.buf.ws) == 0
        torch.cuda.synchronize()
        assert torch.equal(got, want), batch
        for name in ("topk_idx", "topk_w", "counts", "offsets", "sorted_pair", "inv_pos"):
            assert torch.equal(getattr(chain.buf, name), getattr(per_layer.buf, name)), (batch, name)
        n = int(per_layer.buf.active[0])  # the list is [count, ids...]; the rest is not written
        assert torch.equal(chain.buf.active[:1 + n], per_layer.buf.active[:1 + n]), batch
        assert torch.equal(chain.xn, per_layer.xn)
        # x itself is left unchanged
        assert torch.equal(x, dls[0].x(batch))


def test_stack_forward_keeps_every_layers_status():
    # layer 0 has no resident slot for any routed expert (MOE_DEV_MISSING_SLOT; its routed rows
    # are not written), the later layers are clean: the flag survives their router kernels,
    # which clear the word in a single-layer call
    w = custom("stack", d=256, f=128, E=32, k=4, layers=3)
    dls, s, layers = _stack_layers(w)
    missing = torch.full_like(dls[0].slot_of, -1)
    d0 = dls[0]
    layers[0] = LayerWeights(d0.router, L.expert_table(d0.pool, d0.slot_bytes, d0.n_slots, missing, d0.shared_ptr))
    st = DecodeStack(s, layers, native=True)
    st.buf.y_perm.zero_()
    st.forward(dls[0].x(0))
    assert L.moe_read_status(st.buf.ws) == L.MOE_DEV_MISSING_SLOT
    # a clean stack clears it again at its first layer
    clean = DecodeStack(s, [LayerWeights(d.router, L.expert_table(d.pool, d.slot_bytes, d.n_slots, d.slot_of,
                                                                  d.shared_ptr)) for d in dls], native=True)
    clean.buf = st.buf
    clean.forward(dls[0].x(0))
    assert L.moe_read_status(st.buf.ws) == 0


def test_stack_forward_degenerate_and_bad_arguments():
    w = custom("stack", d=256, f=128, E=32, k=4, layers=2)
    dls, s, layers = _stack_layers(w)
    st = DecodeStack(s, layers, native=True)
    b = st.buf
    x = dls[0].x(0)
    st.resid.copy_(x)
    # no layers: nothing but the status word is touched
    L.moe_stack_forward(s, [], [], L.MOE_MODE_AUTO, st.resid, L.MOE_BF16, 1e-6, st.xn, b.topk_idx, b.topk_w,
                        b.counts, b.offsets, b.sorted_pair, b.inv_pos, b.active, b.y_perm, b.ydt, b.ws, b.ws_bytes)
    assert L.moe_read_status(b.ws) == 0
    assert torch.equal(st.resid, x)
    # T == 0
    s0 = L.shape(0, w.d, w.f, w.E, w.k, w.n_shared)
    L.moe_stack_forward(s0, [l.router for l in layers], [l.table for l in layers], L.MOE_MODE_AUTO, None,
                        L.MOE_BF16, 1e-6, None, None, None, b.counts, b.offsets, None, None, b.active, None, b.ydt,
                        b.ws, b.ws_bytes)
    bad = [
        dict(eps=-1.0),
        dict(xn=st.resid),   # xn aliases resid
        dict(rdt=7),
    ]
    for kw in bad:
        args = dict(eps=1e-6, xn=st.xn, rdt=L.MOE_BF16)
        args.update(kw)
        with pytest.raises(L.MoeError):
            L.moe_stack_forward(s, [l.router for l in layers], [l.table for l in layers], L.MOE_MODE_AUTO, st.resid,
                                args["rdt"], args["eps"], args["xn"], b.topk_idx, b.topk_w, b.counts, b.offsets,
                                b.sorted_pair, b.inv_pos, b.active, b.y_perm, b.ydt, b.ws, b.ws_bytes)
    torch.cuda.synchronize()
    assert torch.equal(st.resid, x)


def test_tiered_step_full_width():
    # the tiered path at the full layer width (d = 2048, f = 768, top-10 + 1 shared): 2 layers of
    # 64 experts in pinned host memory, 48 device slots, so a step's two layers (about 36
    # experts each) cannot both stay resident: misses, evictions and copies every step
    from synth.gpu import fill_expert_records
    w = custom("stack", E=64, layers=2)
    n_slots = 48
    rb = w.record_bytes
    n_all = w.layers * w.E
    host = torch.empty((n_all, rb), dtype=torch.uint8).pin_memory()
    tmp = torch.empty((w.E, rb), dtype=torch.uint8, device="cuda")
    for l in range(w.layers):
        fill_expert_records(w.seed, l, 0, w.E, w.d, w.f, tmp.data_ptr(), rb, w.expert_sigma)
        host[l * w.E:(l + 1) * w.E].copy_(tmp)
    torch.cuda.synchronize()
    dls = [DeviceLayer(w, layer=l) for l in range(w.layers)]
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    shared = [dl.pool[w.E * rb:(w.E + w.n_shared) * rb] for dl in dls]
    ts = TieredStack(s, w.layers, [dl.router for dl in dls], [host[i].data_ptr() for i in range(n_all)], n_slots,
                     rb, shared)
    try:
        for step in range(2):
            keep = []
            ts.forward(dls[0].x(step), keep=keep)
            assert ts.status() == 0
            torch.cuda.synchronize()
            check_layers(w, keep, range(w.layers))
        st = L.slot_table_stats(ts.table)
        assert st.misses > 0 and st.evictions > 0
    finally:
        ts.close()


@pytest.mark.parametrize("overlap,freq,prefetch,pcie_frac", [(True, False, False, 1.0), (False, False, False, 1.0),
                                                             (True, True, False, 1.0), (True, False, True, 1.0),
                                                             (True, True, True, 1.0), (True, False, False, 0.5),
                                                             (True, False, True, 0.0)])
def test_tiered_stack_misses_evictions_and_parity(overlap, freq, prefetch, pcie_frac):
    # 2 layers x 32 experts, but only 24 device slots: every step evicts and copies. With freq:
    # the decayed-use-count policy, and a usage profile that fills the pool before step 0
    w = custom("stack", d=256, f=128, E=32, k=6, layers=2, T=4)
    n_slots = 24
    rb = w.record_bytes
    host = torch.empty((w.layers * w.E, rb), dtype=torch.uint8).pin_memory()
    for l in range(w.layers):
        for e in range(w.E):
            host[l * w.E + e].copy_(torch.from_numpy(synth.pack_record(cached_expert(w, l, e))))
    h_records = [host[i].data_ptr() for i in range(w.layers * w.E)]
    dls = [DeviceLayer(w, layer=l) for l in range(w.layers)]  # routers and resident shared experts
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    shared = [dl.pool[w.E * rb:(w.E + w.n_shared) * rb] for dl in dls]
    profile = np.random.default_rng(5).random(w.layers * w.E).astype(np.float32) if freq else None
    ts = TieredStack(s, w.layers, [dl.router for dl in dls], h_records, n_slots, rb, shared,
                     policy=L.MOE_SLOT_FREQ if freq else L.MOE_SLOT_LRU, half_life_steps=2.0, profile=profile)
    assert ts.n_warm == (n_slots if freq else 0)
    lookups = 0
    n_host = 0
    try:
        for step in range(3):
            keep = []
            ts.forward(dls[0].x(step), keep=keep, overlap=overlap, prefetch=prefetch, pcie_frac=pcie_frac)
            n_host += sum(ts.layer_host)
            assert ts.status() == 0
            torch.cuda.synchronize()
            check_layers(w, keep, range(w.layers))
            lookups += sum(np.unique(rec[1].cpu().numpy()).size for rec in keep if rec[0] == "idx")
        lookups -= n_host  # experts computed on the host are neither hits nor misses of the table
        st = L.slot_table_stats(ts.table)
        assert (n_host > 0) == (pcie_frac < 1.0)
        assert st.hits + st.misses == lookups
        assert st.misses > 0 or pcie_frac == 0.0
        pf_loads, pf_used = L.slot_table_prefetch_stats(ts.table)
        assert st.bytes_h2d == (st.misses + ts.n_warm + pf_loads) * rb
        if prefetch:
            # layer 1 routed on layer 0's input: most of its experts are loaded before its turn
            assert pf_loads > 0 and pf_used > 0 and pf_used <= pf_loads
        else:
            assert pf_loads == 0
        # every resident expert's slot holds that expert's record
        snap = np.zeros(w.layers * w.E, dtype=np.int32)
        L.slot_table_snapshot(ts.table, snap.ctypes.data)
        assert np.array_equal(snap.reshape(w.layers, w.E), ts.slot_of.cpu().numpy())
        pool = ts.pool.cpu().numpy()
        for i in np.nonzero(snap >= 0)[0][:12]:
            slot = int(snap[i])
            assert np.array_equal(pool[slot * rb:(slot + 1) * rb], host[i].numpy())
    finally:
        ts.close()


@pytest.mark.parametrize("pcie_frac", [1.0, 0.5])
def test_tiered_stack_two_bit_records(pcie_frac):
    # the tiered path on 2-bit expert records (2.5 bits per weight): slots of the 2-bit record
    # size, misses copied and (pcie_frac < 1) computed on the host from 2-bit records; every
    # layer against the oracle on the same dequantised weights
    w = custom("stack", d=256, f=256, E=32, k=6, layers=2, T=4, fmt=synth.FMT_Q2)
    n_slots = 24
    rb = w.record_bytes
    host = torch.empty((w.layers * w.E, rb), dtype=torch.uint8).pin_memory()
    for l in range(w.layers):
        for e in range(w.E):
            host[l * w.E + e].copy_(torch.from_numpy(synth.pack_record(cached_expert(w, l, e))))
    h_records = [host[i].data_ptr() for i in range(w.layers * w.E)]
    dls = [DeviceLayer(w, layer=l) for l in range(w.layers)]
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    shared = [dl.pool[w.E * rb:(w.E + w.n_shared) * rb] for dl in dls]
    ts = TieredStack(s, w.layers, [dl.router for dl in dls], h_records, n_slots, rb, shared, fmt=L.MOE_FMT_Q2)
    n_host = 0
    try:
        for step in range(3):
            keep = []
            ts.forward(dls[0].x(step), keep=keep, pcie_frac=pcie_frac)
            n_host += sum(ts.layer_host)
            assert ts.status() == 0
            torch.cuda.synchronize()
            check_layers(w, keep, range(w.layers))
        st = L.slot_table_stats(ts.table)
        assert st.misses > 0 and st.evictions > 0
        assert (n_host > 0) == (pcie_frac < 1.0)
        snap = np.zeros(w.layers * w.E, dtype=np.int32)
        L.slot_table_snapshot(ts.table, snap.ctypes.data)
        pool = ts.pool.cpu().numpy()
        for i in np.nonzero(snap >= 0)[0][:8]:
            slot = int(snap[i])
            assert np.array_equal(pool[slot * rb:(slot + 1) * rb], host[i].numpy())
    finally:
        ts.close()


@pytest.mark.parametrize("fmt,pcie_frac,freq", [(0, 1.0, False), (0, 0.5, False), (1, 1.0, True), (1, 0.5, False)])
def test_tiered_native_executor_is_bit_identical(fmt, pcie_frac, freq):
    # moe_tiered_forward (the library's executor: the per-layer host work in C++) against the
    # Python loop of TieredStack, on two identical fresh stacks: the same outputs bit for bit, the
    # same misses and host-computed experts per layer, the same slot-table counters
    w = custom("stack", d=256, f=256, E=32, k=6, layers=3, T=4, fmt=fmt)
    n_slots = 24
    rb = w.record_bytes
    host = torch.empty((w.layers * w.E, rb), dtype=torch.uint8).pin_memory()
    for l in range(w.layers):
        for e in range(w.E):
            host[l * w.E + e].copy_(torch.from_numpy(synth.pack_record(cached_expert(w, l, e))))
    h_records = [host[i].data_ptr() for i in range(w.layers * w.E)]
    dls = [DeviceLayer(w, layer=l) for l in range(w.layers)]
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    shared = [dl.pool[w.E * rb:(w.E + w.n_shared) * rb] for dl in dls]
    profile = np.random.default_rng(3).random(w.layers * w.E).astype(np.float32) if freq else None
    runs = []
    for native in (False, True):
        ts = TieredStack(s, w.layers, [dl.router for dl in dls], h_records, n_slots, rb, shared, fmt=fmt,
                         policy=L.MOE_SLOT_FREQ if freq else L.MOE_SLOT_LRU, half_life_steps=2.0, profile=profile,
                         native=native)
        ts.host_threads = 2
        try:
            outs, misses, hosts = [], [], []
            for step in range(4):
                outs.append(ts.forward(dls[0].x(step % 2), pcie_frac=pcie_frac).clone())
                torch.cuda.synchronize()
                assert ts.status() == 0
                misses.append(list(ts.layer_misses))
                hosts.append(list(ts.layer_host))
            st = L.slot_table_stats(ts.table)
            runs.append((outs, misses, hosts, (st.hits, st.misses, st.evictions, st.bytes_h2d)))
        finally:
            ts.close()
    (o0, m0, h0, s0), (o1, m1, h1, s1) = runs
    for a, b in zip(o0, o1):
        assert torch.equal(a, b)
    assert m0 == m1 and h0 == h1 and s0 == s1
    assert sum(map(sum, m0)) > 0
    assert (sum(map(sum, h0)) > 0) == (pcie_frac < 1.0)
