"""The C-ABI library without a GPU: it loads, exports every symbol include/moe.h declares,
agrees with the generator on the record layout, rejects bad arguments on the host before
any CUDA call, and runs the slot table's LRU policy with an injected copier."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import synth
from routed_expert_ffn_bucketing_b300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:moe_status|const char\s*\*)\s*(\w+)\s*\(", text, flags=re.M)
    assert len(names) >= 12
    return names


def test_library_exports_every_declared_symbol():
    lib = L.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(L._SIGS), "binding misses a declared entry point"


def test_generator_library_exports_fill():
    lib = C.CDLL(os.path.join(ROOT, "synth", "libsynth_b300.so"))
    assert hasattr(lib, "synth_fill_expert_records")


@pytest.mark.parametrize("d,f", [(32, 32), (256, 128), (2048, 768), (96, 160), (4096, 1536)])
def test_expert_layout_matches_generator(d, f):
    a = L.moe_get_expert_layout(d, f)
    b = synth.record_layout(d, f)
    assert (a.gate_q, a.up_q, a.down_q, a.gate_s, a.up_s, a.down_s, a.record_bytes) == (
        b.gate_q, b.up_q, b.down_q, b.gate_s, b.up_s, b.down_s, b.record_bytes)
    assert a.record_bytes % 256 == 0


def test_layout_rejects_bad_sizes():
    for d, f in [(0, 32), (33, 32), (32, 48), (-32, 32)]:
        with pytest.raises(L.MoeError) as e:
            L.moe_get_expert_layout(d, f)
        assert e.value.status == L.MOE_EINVAL


def test_workspace_size_covers_activation_buffer():
    for T in (0, 1, 4, 16, 17, 8192):
        s = L.moe_workspace_size(L.shape(T, 2048, 768, 512, 10, 1))
        assert s % 256 == 0
        assert s >= 256 + 4 * (T * 10 + T) * 768   # status word + fp32 h rows


BAD_SHAPES = [
    (L.shape(4, 100, 768, 512, 10, 1), L.MOE_EINVAL),   # d % 32
    (L.shape(4, 2048, 770, 512, 10, 1), L.MOE_EINVAL),  # f % 32
    (L.shape(4, 2048, 768, 8, 10, 1), L.MOE_EINVAL),    # k > E
    (L.shape(-1, 2048, 768, 512, 10, 1), L.MOE_EINVAL),
    (L.shape(4, 2048, 768, 512, 0, 1), L.MOE_EINVAL),
    (L.shape(4, 2048, 768, 512, 33, 1), L.MOE_EUNSUPPORTED),
    (L.shape(4, 2048, 768, 2048, 10, 1), L.MOE_EUNSUPPORTED),
    (L.shape(70000, 2048, 768, 512, 10, 1), L.MOE_EUNSUPPORTED),
]


@pytest.mark.parametrize("s,code", BAD_SHAPES)
def test_bad_shapes_rejected_before_any_launch(s, code):
    # fake, never dereferenced addresses: the checks fail before any CUDA call
    fake = 0x10000
    with pytest.raises(L.MoeError) as e:
        L.moe_route(s, fake, L.MOE_BF16, fake, fake, fake, None, fake, 1 << 30, 0)
    assert e.value.status == code
    with pytest.raises(L.MoeError) as e:
        L.moe_workspace_size(s)
    assert e.value.status == code


def test_null_and_misaligned_arguments():
    s = L.shape(4, 256, 128, 16, 2, 0)
    need = L.moe_workspace_size(s)
    fake = 0x10000
    cases = [
        lambda: L.moe_route(s, None, L.MOE_BF16, fake, fake, fake, None, fake, need, 0),
        lambda: L.moe_route(s, fake, L.MOE_BF16, fake, fake, fake, None, fake + 16, need, 0),   # ws not 256-aligned
        lambda: L.moe_route(s, fake, L.MOE_BF16, fake, fake, fake, None, fake, need - 1, 0),    # ws too small
        lambda: L.moe_route(s, fake + 2, L.MOE_BF16, fake, fake, fake, None, fake, need, 0),    # x misaligned
        lambda: L.moe_route(s, fake, 7, fake, fake, fake, None, fake, need, 0),                 # bad dtype
        lambda: L.moe_permute(s, fake, None, fake, fake, fake, fake, fake, need, 0),
        lambda: L.moe_combine(s, fake, L.MOE_F32, fake, fake, None, fake + 4, L.MOE_BF16, 0),
        lambda: L.moe_expert_ffn(s, 9, fake, L.MOE_BF16, L.expert_table(fake, 104448, 16, fake), fake, fake, fake,
                                 fake, L.MOE_F32, fake, need, 0),
        lambda: L.moe_expert_ffn(s, 0, fake, L.MOE_BF16, L.expert_table(fake, 1000, 16, fake), fake, fake, fake,
                                 fake, L.MOE_F32, fake, need, 0),                              # slot_bytes too small
        lambda: L.moe_expert_ffn(s, 0, fake, L.MOE_BF16, L.expert_table(fake, 104448, 16, fake, fake), fake, fake,
                                 fake, fake, L.MOE_F32, fake, need, 0),                        # shared with n_shared 0
    ]
    for fn in cases:
        with pytest.raises(L.MoeError) as e:
            fn()
        assert e.value.status == L.MOE_EINVAL, L.moe_last_error_string()
        assert L.moe_last_error_string()


# ------------------------------------------------------------------ slot table ------------

class FakeCopier:
    """Records every copy the table asks for; optionally fails the n-th record copy."""

    def __init__(self, pool, table, slot_bytes, fail_at=None):
        self.pool, self.table, self.slot_bytes = pool, table, slot_bytes
        self.records, self.entries = [], {}
        self.fail_at, self.n_record_copies = fail_at, 0
        self.fn = L.MOE_COPY_FN(self._copy)

    def _copy(self, dst, src, nbytes, stream, user):
        dst = dst or 0
        if self.table <= dst < self.table + (1 << 20):
            vals = np.ctypeslib.as_array((C.c_int32 * (nbytes // 4)).from_address(src))
            for i, v in enumerate(vals):
                self.entries[(dst - self.table) // 4 + i] = int(v)
            return 0
        self.n_record_copies += 1
        if self.fail_at is not None and self.n_record_copies == self.fail_at:
            return 1
        assert (dst - self.pool) % self.slot_bytes == 0 and nbytes == self.slot_bytes
        self.records.append(((dst - self.pool) // self.slot_bytes, src))
        return 0


def _make_table(Lyr, E, n_slots, fail_at=None):
    pool, tab, sb = 0x100000, 0x40000000, 256
    hrec = [0x7000000 + 4096 * i for i in range(Lyr * E)]
    cp = FakeCopier(pool, tab, sb, fail_at)
    h = L.slot_table_create(Lyr, E, n_slots, sb, pool, tab, hrec, cp.fn, None)
    return h, cp, hrec


def _update(h, layer, ids):
    a = (C.c_int32 * max(1, len(ids)))(*ids)
    hits = (C.c_int32 * max(1, len(ids)))()
    miss = (C.c_int32 * max(1, len(ids)))()
    nh, nm = C.c_int32(), C.c_int32()
    st = L.slot_table_update(h, layer, C.addressof(a), len(ids), None, None, C.addressof(hits), C.addressof(nh),
                             C.addressof(miss), C.addressof(nm), None)
    return st, list(hits[:nh.value]), list(miss[:nm.value])


def _snapshot(h, Lyr, E):
    out = (C.c_int32 * (Lyr * E))()
    L.slot_table_snapshot(h, C.addressof(out))
    return np.array(out[:]).reshape(Lyr, E)


def test_slot_table_fills_empty_slots_then_evicts_lru():
    h, cp, hrec = _make_table(2, 8, 4)
    assert all(v == -1 for v in cp.entries.values()) and len(cp.entries) == 16
    st, hits, miss = _update(h, 0, [3, 5])
    assert st == 0 and hits == [] and miss == [3, 5]
    assert [s for s, _ in cp.records] == [0, 1] and [src for _, src in cp.records] == [hrec[3], hrec[5]]
    st, hits, miss = _update(h, 0, [5, 6])
    assert hits == [5] and miss == [6] and cp.records[-1] == (2, hrec[6])
    st, hits, miss = _update(h, 1, [0])        # last empty slot
    assert miss == [0] and cp.records[-1] == (3, hrec[8])
    # LRU now: slot 0 (layer0 e3), slot 1 (e5), slot 2 (e6), slot 3 (layer1 e0), with e5/e6 touched after e3
    st, hits, miss = _update(h, 1, [1])
    assert miss == [1] and cp.records[-1][0] == 0   # evicts layer 0 expert 3
    snap = _snapshot(h, 2, 8)
    assert snap[0, 3] == -1 and snap[1, 1] == 0 and snap[0, 5] == 1 and snap[0, 6] == 2 and snap[1, 0] == 3
    # the evicted entry of the other layer was written to the device table too
    assert cp.entries[0 * 8 + 3] == -1 and cp.entries[1 * 8 + 1] == 0
    s = L.slot_table_stats(h)
    assert (s.hits, s.misses, s.evictions, s.bytes_h2d) == (1, 5, 1, 5 * 256)
    L.slot_table_destroy(h)


def test_slot_table_never_evicts_current_experts():
    h, cp, _ = _make_table(1, 16, 3)
    _update(h, 0, [0, 1, 2])
    st, hits, miss = _update(h, 0, [2, 0, 9])   # 9 must evict expert 1 (not 0 or 2)
    assert hits == [2, 0] and miss == [9]
    snap = _snapshot(h, 1, 16)
    assert snap[0, 1] == -1 and snap[0, 9] >= 0 and snap[0, 0] >= 0 and snap[0, 2] >= 0
    L.slot_table_destroy(h)


def test_slot_table_reports_no_slot_and_leaves_table_unchanged():
    h, cp, _ = _make_table(1, 16, 3)
    _update(h, 0, [0, 1])
    before = _snapshot(h, 1, 16).copy()
    n_before = len(cp.records)
    st, _, _ = _update(h, 0, [0, 1, 2, 3])    # 2 misses, 1 evictable slot
    assert st == L.MOE_ENOSLOT
    assert np.array_equal(before, _snapshot(h, 1, 16)) and len(cp.records) == n_before
    L.slot_table_destroy(h)


def test_slot_table_rejects_bad_ids():
    h, cp, _ = _make_table(2, 8, 4)
    for layer, ids in [(0, [1, 1]), (0, [8]), (0, [-1]), (2, [0]), (-1, [0])]:
        a = (C.c_int32 * len(ids))(*ids)
        with pytest.raises(L.MoeError) as e:
            L.slot_table_update(h, layer, C.addressof(a), len(ids), None, None)
        assert e.value.status == L.MOE_EINVAL
    L.slot_table_destroy(h)


def test_slot_table_copy_failure_is_reported_and_not_resident():
    h, cp, _ = _make_table(1, 8, 4, fail_at=2)
    a = (C.c_int32 * 3)(4, 5, 6)
    with pytest.raises(L.MoeError) as e:
        L.slot_table_update(h, 0, C.addressof(a), 3, None, None)
    assert e.value.status == L.MOE_ECUDA
    snap = _snapshot(h, 1, 8)
    assert snap[0, 4] >= 0 and snap[0, 5] == -1 and snap[0, 6] == -1
    assert cp.entries[4] == snap[0, 4]
    # a retry succeeds once the copier works again
    cp.fail_at = None
    st, hits, miss = _update(h, 0, [4, 5, 6])
    assert st == 0 and hits == [4] and miss == [5, 6]
    L.slot_table_destroy(h)


# ---------------------------------------------------------------- decayed-frequency policy ----

def _freq_table(Lyr, E, n_slots, half_life, policy=None):
    h, cp, hrec = _make_table(Lyr, E, n_slots)
    L.slot_table_set_policy(h, L.MOE_SLOT_FREQ if policy is None else policy, half_life)
    return h, cp, hrec


def _resident(h, Lyr, E):
    snap = _snapshot(h, Lyr, E)
    return {(l, e) for l in range(Lyr) for e in range(E) if snap[l, e] >= 0}


def test_slot_table_freq_keeps_the_more_used_expert():
    # pool of 2; expert 0 used twice, expert 1 once, then expert 2 misses
    for policy, evicted in ((L.MOE_SLOT_FREQ, 1), (L.MOE_SLOT_LRU, 0)):
        h, cp, _ = _freq_table(1, 8, 2, 1e9, policy)
        for ids in ([0], [0], [1]):
            _update(h, 0, ids)
        st, hits, miss = _update(h, 0, [2])
        assert st == 0 and miss == [2]
        assert _resident(h, 1, 8) == {(0, 2), (0, 1 - evicted)}
        L.slot_table_destroy(h)


def test_slot_table_freq_counts_decay_with_the_half_life():
    # expert 0 used at calls 1..3, expert 1 at call 4; at call 5 a miss needs a slot.
    # half-life 1 call: 2^-4 + 2^-3 + 2^-2 = 0.4375 < 2^-1, so expert 0 goes;
    # no decay: 3 uses against 1, so expert 1 goes.
    for hl, keep in ((1.0, 1), (1e9, 0)):
        h, cp, _ = _freq_table(1, 8, 2, hl)
        for ids in ([0], [0], [0], [1]):
            _update(h, 0, ids)
        _update(h, 0, [5])
        assert _resident(h, 1, 8) == {(0, 5), (0, keep)}
        L.slot_table_destroy(h)


def test_slot_table_freq_never_evicts_current_experts():
    # expert 0 has the smallest count but is in the call, so the miss takes expert 1's slot
    h, cp, _ = _freq_table(1, 8, 2, 1e9)
    for ids in ([1], [1], [1], [0]):
        _update(h, 0, ids)
    st, hits, miss = _update(h, 0, [0, 2])
    assert hits == [0] and miss == [2]
    assert _resident(h, 1, 8) == {(0, 0), (0, 2)}
    L.slot_table_destroy(h)


class _FreqModel:
    """The decayed-frequency rule as stated in include/moe.h, by brute force: a use made now
    weighs inc (inc grows by 2^(1/half_life) per call, rescaled by 2^-600 past 2^600); a miss
    takes an empty slot (lowest index) or the unpinned slot whose owner has the smallest
    (count, last use), lowest slot index on ties."""

    def __init__(self, Lyr, E, n, hl):
        self.E, self.n, self.g, self.inc, self.calls = E, n, 2.0 ** (1.0 / hl), 1.0, 0
        self.score, self.last = [0.0] * (Lyr * E), [-1] * (Lyr * E)
        self.owner, self.slot_of = [-1] * n, {}

    def update(self, layer, ids):
        keys = [layer * self.E + e for e in ids]
        nh = sum(k in self.slot_of for k in keys)
        if len(keys) - nh > self.n - nh:
            return None
        self.calls += 1
        self.inc *= self.g
        if self.inc > 2.0 ** 600:
            self.score = [v * 2.0 ** -600 for v in self.score]
            self.inc *= 2.0 ** -600
        for k in keys:
            self.score[k] += self.inc
            self.last[k] = self.calls
        pinned = {self.slot_of[k] for k in keys if k in self.slot_of}
        hits = [e for e, k in zip(ids, keys) if k in self.slot_of]
        placed = []
        for e, k in zip(ids, keys):
            if k in self.slot_of:
                continue

            def order(s):
                o = self.owner[s]
                return (0, 0.0, 0, s) if o < 0 else (1, self.score[o], self.last[o], s)
            v = min((s for s in range(self.n) if s not in pinned), key=order)
            if self.owner[v] >= 0:
                del self.slot_of[self.owner[v]]
            self.owner[v], self.slot_of[k] = k, v
            pinned.add(v)
            placed.append((e, v))
        return hits, placed


@pytest.mark.parametrize("hl", [0.5, 2.5, 40.0])
def test_slot_table_freq_matches_brute_force_model(hl):
    # hl = 0.5 grows the use weight 4x per call: the 2^-600 rescale happens about every 300 calls
    Lyr, E, n = 3, 16, 10
    rng = np.random.default_rng(7)
    h, cp, hrec = _freq_table(Lyr, E, n, hl)
    model = _FreqModel(Lyr, E, n, hl)
    for call in range(700):
        layer = int(rng.integers(0, Lyr))
        # skewed ids so that counts differ; sometimes more misses than free slots
        size = int(rng.integers(1, 13 if call % 50 == 49 else 7))
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        ids = [int(e) for e in rng.choice(E, size=size, replace=False, p=p / p.sum())]
        n_rec = len(cp.records)
        st, hits, miss = _update(h, layer, ids)
        ref = model.update(layer, ids)
        if ref is None:
            assert st == L.MOE_ENOSLOT and len(cp.records) == n_rec
            continue
        assert st == 0 and hits == ref[0] and miss == [e for e, _ in ref[1]]
        assert [s for s, _ in cp.records[n_rec:]] == [v for _, v in ref[1]]
        assert [src for _, src in cp.records[n_rec:]] == [hrec[layer * E + e] for e, _ in ref[1]]
        snap = _snapshot(h, Lyr, E).reshape(-1)
        assert {k: int(snap[k]) for k in range(Lyr * E) if snap[k] >= 0} == model.slot_of
    L.slot_table_destroy(h)


def _zipf_trace(Lyr, E, k, n_calls, seed):
    rng = np.random.default_rng(seed)
    perms = [rng.permutation(E) for _ in range(Lyr)]
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    for c in range(n_calls):
        l = c % Lyr
        yield l, [int(perms[l][r]) for r in rng.choice(E, size=k, replace=False, p=p)]


def test_slot_table_freq_beats_lru_on_zipf_routing():
    # a stationary Zipf(1.1) popularity: counting uses keeps the hot experts that recency
    # alone lets go between two calls of their layer
    rates = {}
    for policy in (L.MOE_SLOT_LRU, L.MOE_SLOT_FREQ):
        h, cp, _ = _freq_table(4, 64, 48, 4000.0, policy)
        hits = total = 0
        for i, (l, ids) in enumerate(_zipf_trace(4, 64, 6, 4000, seed=3)):
            st, hh, mm = _update(h, l, ids)
            assert st == 0
            if i >= 400:
                hits, total = hits + len(hh), total + len(ids)
        rates[policy] = hits / total
        L.slot_table_destroy(h)
    assert rates[L.MOE_SLOT_FREQ] > rates[L.MOE_SLOT_LRU] + 0.03, rates


def test_slot_table_warm_fills_empty_slots_from_the_profile():
    Lyr, E, n = 2, 8, 5
    h, cp, hrec = _make_table(Lyr, E, n)
    _update(h, 1, [7])                       # one slot already taken
    w = np.zeros(Lyr * E, dtype=np.float32)
    w[[3, 9, 12, 0, 5]] = [5.0, 4.0, 3.0, 2.0, 2.0]   # keys l*E + e; 0 and 5 tie
    n_rec = len(cp.records)
    assert L.slot_table_warm(h, w.ctypes.data) == 4
    # empty slots 1..4 in order take keys 3, 9, 12, then 0 (the lower key of the tie)
    assert cp.records[n_rec:] == [(1, hrec[3]), (2, hrec[9]), (3, hrec[12]), (4, hrec[0])]
    assert _resident(h, Lyr, E) == {(1, 7), (0, 3), (1, 1), (1, 4), (0, 0)}
    for key, slot in ((3, 1), (9, 2), (12, 3), (0, 4)):
        assert cp.entries[key] == slot
    s = L.slot_table_stats(h)
    assert (s.hits, s.misses, s.bytes_h2d) == (0, 1, 5 * 256)
    st, hits, miss = _update(h, 0, [0, 3])
    assert hits == [0, 3] and miss == []
    # a full pool: nothing more is loaded and nothing is evicted
    assert L.slot_table_warm(h, w.ctypes.data) == 0
    L.slot_table_destroy(h)


def test_slot_table_warm_under_lru_evicts_the_lowest_weight_first():
    # 4 slots, 3 warm experts: the empty slot goes first, then warm experts from the lowest
    # weight up, the profile's best expert last
    h, cp, hrec = _make_table(1, 16, 4)
    w = np.zeros(16, dtype=np.float32)
    w[[2, 9, 5]] = [1.0, 7.0, 3.0]
    assert L.slot_table_warm(h, w.ctypes.data) == 3
    assert _resident(h, 1, 16) == {(0, 2), (0, 9), (0, 5)}
    _update(h, 0, [11])                      # takes the empty slot
    assert _resident(h, 1, 16) == {(0, 2), (0, 9), (0, 5), (0, 11)}
    _update(h, 0, [12])                      # evicts expert 2 (weight 1)
    assert _resident(h, 1, 16) == {(0, 9), (0, 5), (0, 11), (0, 12)}
    _update(h, 0, [13])                      # then expert 5 (weight 3)
    assert _resident(h, 1, 16) == {(0, 9), (0, 11), (0, 12), (0, 13)}
    _update(h, 0, [14])                      # then expert 9: warm loads are older than any use
    assert _resident(h, 1, 16) == {(0, 11), (0, 12), (0, 13), (0, 14)}
    L.slot_table_destroy(h)


def test_slot_table_warm_weights_seed_the_counts():
    # under FREQ a profile weight counts like uses: expert 1 (weight 10) outlives expert 0
    # (two real uses) when a miss needs a slot
    h, cp, _ = _freq_table(1, 8, 2, 1e9)
    w = np.zeros(8, dtype=np.float32)
    w[1] = 10.0
    assert L.slot_table_warm(h, w.ctypes.data) == 1
    _update(h, 0, [0])
    _update(h, 0, [0])
    _update(h, 0, [4])
    assert _resident(h, 1, 8) == {(0, 1), (0, 4)}
    L.slot_table_destroy(h)


def test_slot_table_policy_and_warm_reject_bad_arguments():
    h, cp, _ = _make_table(1, 8, 2)
    for policy, hl in ((2, 1.0), (-1, 1.0), (L.MOE_SLOT_FREQ, 0.0), (L.MOE_SLOT_FREQ, -3.0),
                       (L.MOE_SLOT_FREQ, float("inf")), (L.MOE_SLOT_FREQ, float("nan"))):
        with pytest.raises(L.MoeError) as e:
            L.slot_table_set_policy(h, policy, hl)
        assert e.value.status == L.MOE_EINVAL
    for bad in (-1.0, float("nan"), float("inf")):
        w = np.ones(8, dtype=np.float32)
        w[3] = bad
        with pytest.raises(L.MoeError) as e:
            L.slot_table_warm(h, w.ctypes.data)
        assert e.value.status == L.MOE_EINVAL
    assert len(cp.records) == 0 and _resident(h, 1, 8) == set()
    with pytest.raises(L.MoeError):
        L.slot_table_warm(h, None)
    L.slot_table_destroy(h)


def test_slot_table_errors_carry_a_message():
    h, cp, _ = _make_table(1, 16, 3)
    _update(h, 0, [0, 1])
    st, _, _ = _update(h, 0, [0, 1, 2, 3])
    assert st == L.MOE_ENOSLOT and "2 misses but 1 slots" in L.moe_last_error_string()
    a = (C.c_int32 * 2)(4, 4)
    with pytest.raises(L.MoeError, match="repeated"):
        L.slot_table_update(h, 0, C.addressof(a), 2, None, None)
    with pytest.raises(L.MoeError, match="layer 3 not in"):
        L.slot_table_update(h, 3, C.addressof(a), 1, None, None)
    with pytest.raises(L.MoeError, match="half-life"):
        L.slot_table_set_policy(h, L.MOE_SLOT_FREQ, 0.0)
    L.slot_table_destroy(h)
    with pytest.raises(L.MoeError, match="slot_table_create"):
        L.slot_table_create(1, 4, 0, 256, 0, 0, [1, 2, 3, 4], FakeCopier(0, 0, 256, None).fn, None)


def test_wait_limit_argument_check():
    # no CUDA call: the limit is host state that later launches copy into their arguments
    with pytest.raises(L.MoeError) as e:
        L.moe_set_wait_limit(11_000_000_000)
    assert e.value.status == L.MOE_EINVAL and "10 s" in L.moe_last_error_string()
    L.moe_set_wait_limit(5_000_000)
    L.moe_set_wait_limit(0)


@pytest.mark.parametrize("d,f", [(256, 256), (2048, 768), (512, 1024)])
def test_q2_record_layout_matches_generator(d, f):
    import synth
    lay = L.moe_get_record_layout(d, f, L.MOE_FMT_Q2)
    ref = synth.record_layout(d, f, synth.FMT_Q2)
    assert (lay.gate_q, lay.up_q, lay.down_q, lay.gate_s, lay.up_s, lay.down_s, lay.record_bytes) == \
        (ref.gate_q, ref.up_q, ref.down_q, ref.gate_s, ref.up_s, ref.down_s, ref.record_bytes)
    i8 = L.moe_get_record_layout(d, f, L.MOE_FMT_INT8)
    assert i8.record_bytes == L.moe_get_expert_layout(d, f).record_bytes
    assert lay.record_bytes < i8.record_bytes / 3


def test_q2_format_checks_before_any_launch():
    for d, f, fmt in ((288, 256, L.MOE_FMT_Q2), (256, 160, L.MOE_FMT_Q2), (256, 256, 7)):
        with pytest.raises(L.MoeError) as e:
            L.moe_get_record_layout(d, f, fmt)
        assert e.value.status == L.MOE_EINVAL
    fake = 1 << 20
    lay = L.moe_get_record_layout(256, 256, L.MOE_FMT_Q2)
    for T, fmt, want in ((16, L.MOE_FMT_Q2, L.MOE_EUNSUPPORTED), (4, 9, L.MOE_EINVAL)):
        s = L.shape(T, 256, 256, 16, 2, 0)
        ws = L.moe_workspace_size(s)
        table = L.expert_table(fake, lay.record_bytes, 16, fake, None, fmt=fmt)
        with pytest.raises(L.MoeError) as e:
            L.moe_expert_ffn(s, L.MOE_MODE_AUTO, fake, L.MOE_BF16, table, fake, fake, fake, fake, L.MOE_F32, fake,
                             ws, 1)
        assert e.value.status == want, L.moe_last_error_string()



def _prefetch(h, layer, ids, keep_layer=0, keep=()):
    a = (C.c_int32 * max(1, len(ids)))(*ids)
    k = (C.c_int32 * max(1, len(keep)))(*keep)
    return L.slot_table_prefetch(h, layer, C.addressof(a), len(ids), keep_layer, C.addressof(k), len(keep))


@pytest.mark.parametrize("policy", [L.MOE_SLOT_LRU, L.MOE_SLOT_FREQ])
def test_slot_table_prefetch_keeps_current_layer_and_turns_into_hits(policy):
    h, cp, hrec = _make_table(2, 8, 4)
    if policy == L.MOE_SLOT_FREQ:
        L.slot_table_set_policy(h, policy, 4.0)
    _update(h, 0, [0, 1, 2])                      # layer 0 uses 3 of the 4 slots
    n0 = len(cp.records)
    # layer 1 is expected to use 5, 6, 7: one empty slot, and nothing of layer 0's set may go
    assert _prefetch(h, 1, [5, 6, 7], keep_layer=0, keep=[0, 1, 2]) == 1
    assert _resident(h, 2, 8) == {(0, 0), (0, 1), (0, 2), (1, 5)}
    assert cp.records[n0:] == [(3, hrec[8 + 5])]
    s = L.slot_table_stats(h)
    assert (s.hits, s.misses) == (0, 3)          # a prefetch is neither a hit nor a miss
    # with layer 0 released, the next prefetch may evict its experts
    assert _prefetch(h, 1, [5, 6, 7]) == 2
    assert {(1, 5), (1, 6), (1, 7)} <= _resident(h, 2, 8)
    st, hits, miss = _update(h, 1, [5, 6, 7, 3])
    assert st == L.MOE_OK and hits == [5, 6, 7] and miss == [3]
    assert L.slot_table_prefetch_stats(h) == (3, 3)
    L.slot_table_destroy(h)


def test_slot_table_prefetch_stops_when_every_slot_is_kept():
    h, cp, hrec = _make_table(2, 8, 3)
    _update(h, 0, [0, 1, 2])
    n0 = len(cp.records)
    assert _prefetch(h, 1, [4, 5], keep_layer=0, keep=[0, 1, 2]) == 0
    assert len(cp.records) == n0 and _resident(h, 2, 8) == {(0, 0), (0, 1), (0, 2)}
    # already resident experts are left alone (no copy), ids of the call are never victims
    assert _prefetch(h, 0, [0, 1, 2]) == 0 and len(cp.records) == n0
    assert _prefetch(h, 1, [4, 5, 6, 7]) == 3
    assert _resident(h, 2, 8) == {(1, 4), (1, 5), (1, 6)}
    L.slot_table_destroy(h)


def test_slot_table_prefetch_rejects_bad_arguments():
    h, cp, _ = _make_table(2, 8, 3)
    for layer, ids, kl, keep in ((2, [1], 0, []), (0, [8], 0, []), (0, [-1], 0, []), (0, [1], 5, [0]),
                                 (0, [1], 0, [9])):
        with pytest.raises(L.MoeError) as e:
            _prefetch(h, layer, ids, kl, keep)
        assert e.value.status == L.MOE_EINVAL
    assert len(cp.records) == 0 and _resident(h, 2, 8) == set()
    L.slot_table_destroy(h)


@pytest.mark.parametrize("fmt,d,f", [(L.MOE_FMT_INT8, 256, 256), (L.MOE_FMT_Q2, 256, 256),
                                     (L.MOE_FMT_INT8, 288, 160)])
def test_host_expert_ffn_matches_oracle(fmt, d, f):
    # the host half of the bandwidth split: every row of the chosen experts against the oracle's
    # SwiGLU FFN of the same tokens, with records packed as the device reads them (288 and 160:
    # rows ending in a block without a partner, stored in order)
    import synth
    from oracle import moe_oracle as O
    from synth.workloads import custom
    w = custom("tiny", T=5, d=d, f=f, E=8, k=3, fmt=fmt)
    rng = np.random.default_rng(11)
    topk = np.stack([rng.choice(w.E, w.k, replace=False) for _ in range(w.T)]).astype(np.int32)
    flat = topk.reshape(-1)
    order = np.argsort(flat, kind="stable").astype(np.int32)          # pairs grouped by expert
    offsets = np.zeros(w.E + 1, np.int32)
    offsets[1:] = np.cumsum(np.bincount(flat, minlength=w.E))
    x_bits = w.x_bits(0)
    x = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
    experts = np.array([e for e in range(w.E) if offsets[e + 1] > offsets[e]][::2], np.int32)
    recs = [synth.pack_record(w.expert(0, int(e))) for e in experts]
    y = np.full((w.P, w.d), np.nan, np.float32)
    s = L.shape(w.T, w.d, w.f, w.E, w.k, 0)
    L.moe_host_expert_ffn(s, x_bits.ctypes.data, L.MOE_BF16, [r.ctypes.data for r in recs], experts.ctypes.data,
                          experts.size, offsets.ctypes.data, order.ctypes.data, y.ctypes.data, fmt, 3)
    for e in experts:
        r0, r1 = offsets[e], offsets[e + 1]
        ref = O.swiglu_ffn(x[order[r0:r1] // w.k], O.dense_expert(w.expert(0, int(e))))
        got = y[r0:r1].astype(np.float64)
        assert np.max(np.abs(got - ref)) <= 1e-5 * np.max(np.abs(ref)), e
    done = set()
    for e in experts:
        done |= set(range(offsets[e], offsets[e + 1]))
    untouched = [r for r in range(w.P) if r not in done]
    assert np.all(np.isnan(y[untouched]))                              # other rows are left alone


def test_host_expert_ffn_and_lookup_argument_checks():
    s = L.shape(2, 256, 256, 8, 2, 0)
    z = np.zeros(16, np.int32)
    with pytest.raises(L.MoeError) as e:
        L.moe_host_expert_ffn(s, None, L.MOE_BF16, [0], z.ctypes.data, 1, z.ctypes.data, z.ctypes.data, None)
    assert e.value.status == L.MOE_EINVAL
    with pytest.raises(L.MoeError):
        L.moe_host_expert_ffn(s, z.ctypes.data, L.MOE_BF16, [z.ctypes.data], z.ctypes.data, 1, z.ctypes.data,
                              z.ctypes.data, z.ctypes.data, fmt=5)
    h, cp, _ = _make_table(2, 8, 3)
    _update(h, 1, [2, 5])
    ids = np.array([2, 5, 6], np.int32)
    out = np.zeros(3, np.int32)
    L.slot_table_lookup(h, 1, ids.ctypes.data, 3, out.ctypes.data)
    assert out[0] >= 0 and out[1] >= 0 and out[2] == -1
    with pytest.raises(L.MoeError):
        L.slot_table_lookup(h, 2, ids.ctypes.data, 3, out.ctypes.data)
    L.slot_table_destroy(h)
