"""Pins of the CPU oracle against things other than itself: brute force, closed forms,
hand-computed examples, invariants and independent library routines. CPU only.

Each test names the mistake it is there to catch.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from synth import ExpertArrays

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand_expert(rng, d, f, zero=False, scale=0.02):
    if zero:
        return ExpertArrays(np.zeros((f, d), np.int8), np.ones((f, d // 32), np.float16),
                            np.zeros((f, d), np.int8), np.ones((f, d // 32), np.float16),
                            np.zeros((d, f), np.int8), np.ones((d, f // 32), np.float16))

    def q(r, c):
        return rng.integers(-127, 128, size=(r, c)).astype(np.int8)

    def s(r, c):
        return (rng.uniform(0.5, 1.5, size=(r, c // 32)) * scale / 127).astype(np.float16)
    return ExpertArrays(q(f, d), s(f, d), q(f, d), s(f, d), q(d, f), s(d, f))


# ------------------------------------------------------------------ top-k -----------------

def _brute_topk(l, k):
    """The k-subset whose keys (logit, -index), sorted descending, are lexicographically
    largest; returned in that descending order. Enumerates every subset."""
    E = len(l)
    best, best_keys = None, None
    for sub in itertools.combinations(range(E), k):
        keys = sorted(((float(l[e]) + 0.0, -e) for e in sub), reverse=True)
        if best_keys is None or keys > best_keys:
            best, best_keys = sub, keys
    return [-kk[1] for kk in best_keys]


@pytest.mark.parametrize("E", [1, 2, 3, 5, 8])
def test_topk_matches_brute_force_with_ties(E):
    # catches: wrong sort direction, tie going to the highest index, order of output
    rng = np.random.default_rng(E)
    for trial in range(30):
        # few distinct values, so exact ties are frequent
        l = rng.integers(-3, 4, size=(1, E)).astype(np.float32)
        if trial % 3 == 0:
            l = rng.standard_normal((1, E)).astype(np.float32)
        for k in range(1, E + 1):
            got = O.select_topk(l, k)[0].tolist()
            assert got == _brute_topk(l[0], k), (l, k, got)


def test_topk_negative_zero_ties_positive_zero():
    # catches: ordering -0.0 below +0.0 (then index 1 would lose to index 3)
    l = np.array([[-1.0, -0.0, -2.0, 0.0]], dtype=np.float32)
    assert O.select_topk(l, 1)[0].tolist() == [1]
    assert O.select_topk(l, 2)[0].tolist() == [1, 3]


def test_topk_nan_is_never_selected_before_finite():
    l = np.array([[np.nan, -5.0, 1.0]], dtype=np.float32)
    assert O.select_topk(l, 2)[0].tolist() == [2, 1]


# ------------------------------------------------------------------ gate ------------------

def test_gate_is_softmax_of_selected_logits():
    # catches: renormalising over the wrong set, forgetting the max shift, exp of the index
    rng = np.random.default_rng(1)
    l = (rng.standard_normal((6, 9)) * 3).astype(np.float32)
    for k in (1, 2, 4, 9):
        idx = O.select_topk(l, k)
        w = O.gate_weights(l, idx)
        for t in range(l.shape[0]):
            sel = [float(l[t, e]) for e in idx[t]]
            den = sum(math.exp(v) for v in sel)
            ref = [math.exp(v) / den for v in sel]
            assert np.allclose(w[t], ref, rtol=1e-13, atol=0)
            assert abs(sum(w[t]) - 1.0) < 1e-14


def test_gate_k_equals_E_is_plain_softmax():
    l = np.array([[0.5, -1.0, 2.0, 0.0]], dtype=np.float32)
    idx = O.select_topk(l, 4)
    w = O.gate_weights(l, idx)
    ex = [math.exp(v) for v in (2.0, 0.5, 0.0, -1.0)]
    assert idx[0].tolist() == [2, 0, 3, 1]
    assert np.allclose(w[0], [v / sum(ex) for v in ex], rtol=1e-14)


def test_gate_large_logits_do_not_overflow():
    l = np.array([[1000.0, 999.0, -1000.0]], dtype=np.float32)
    w = O.gate_weights(l, O.select_topk(l, 2))
    assert np.allclose(w[0], [1 / (1 + math.exp(-1)), math.exp(-1) / (1 + math.exp(-1))])


# ------------------------------------------------------------------ router ----------------

def test_router_logits_are_rounded_once():
    # 2^24 + 1 + 1 is exact in float64 and representable in fp32; summing in fp32 loses both 1s
    x = np.array([[2.0 ** 24, 1.0, 1.0]])
    w = np.ones((3, 1), dtype=np.float32)
    assert float(O.router_logits(x, w)[0, 0]) == 16777218.0


def test_router_logits_orientation():
    # catches: using w_router transposed ([E][d] instead of [d][E])
    x = np.array([[1.0, 2.0, 3.0]])
    w = np.array([[1, 0], [0, 1], [1, 1]], dtype=np.float32)   # [d=3][E=2]
    assert O.router_logits(x, w).tolist() == [[4.0, 5.0]]


# ------------------------------------------------------------------ dequant ---------------

def test_dequantize_block_index():
    # catches: scale indexed by i % 32 or by row-block instead of column-block
    q = np.zeros((2, 64), np.int8)
    q[0, 0], q[0, 31], q[0, 32], q[1, 63] = 3, -2, 5, 127
    s = np.array([[0.5, 0.25], [1.0, 2.0]], dtype=np.float16)
    W = O.dequantize(q, s)
    assert W[0, 0] == 1.5 and W[0, 31] == -1.0 and W[0, 32] == 1.25 and W[1, 63] == 254.0
    assert np.count_nonzero(W) == 4


def test_dequantize_exact_for_extreme_codes():
    q = np.full((1, 32), -127, np.int8)
    s = np.array([[np.float16(65504.0)]], dtype=np.float16)
    assert O.dequantize(q, s)[0, 0] == -127.0 * 65504.0


# ------------------------------------------------------------------ SwiGLU golden ---------

def _golden_expert(g):
    d, f = g["d"], g["f"]

    def mat(spec, r, c, dt, default):
        a = np.full((r, c), default, dtype=dt)
        for i, row in spec.items():
            for j, v in row.items():
                a[int(i), int(j)] = v
        return a
    sd = g["scale_default"]
    return ExpertArrays(mat(g["gate_q"], f, d, np.int8, 0), mat(g["gate_s"], f, d // 32, np.float16, sd),
                        mat(g["up_q"], f, d, np.int8, 0), mat(g["up_s"], f, d // 32, np.float16, sd),
                        mat(g["down_q"], d, f, np.int8, 0), mat(g["down_s"], d, f // 32, np.float16, sd))


def test_dense_swiglu_hand_example():
    # catches: gate and up swapped, silu applied to the wrong factor, down used transposed,
    # a scale applied to the wrong row, a gate weight other than 1 for E = k = 1
    g = json.load(open(os.path.join(HERE, "golden", "dense_swiglu_d32_f32.json")))
    ex = _golden_expert(g)
    x = np.zeros((g["T"], g["d"]))
    for t, row in g["x"].items():
        for i, v in row.items():
            x[int(t), int(i)] = v
    want = np.zeros((g["T"], g["d"]))
    for t, row in g["expected_out"].items():
        for i, v in row.items():
            want[int(t), int(i)] = v
    w_router = np.ones((g["d"], 1), dtype=np.float32)
    res = O.moe_layer(x, w_router, 1, lambda e: ex)
    assert np.max(np.abs(res.out - want)) <= g["tolerance_abs"]
    assert res.topk_w.tolist() == [[1.0], [1.0]]


# ------------------------------------------------------------------ layer invariants ------

def _small_layer(seed=0, T=12, d=64, f=32, E=6, k=3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d)).astype(np.float32).astype(np.float64)
    wr = (rng.standard_normal((d, E))).astype(np.float32)
    experts = [_rand_expert(rng, d, f) for _ in range(E)]
    shared = [_rand_expert(rng, d, f)]
    return x, wr, experts, shared, k


def test_token_permutation_invariance_bit_exact():
    x, wr, experts, shared, k = _small_layer()
    perm = np.random.default_rng(5).permutation(x.shape[0])
    a = O.moe_layer(x, wr, k, lambda e: experts[e], shared).out
    b = O.moe_layer(x[perm], wr, k, lambda e: experts[e], shared).out
    assert np.array_equal(a[perm], b)


def test_layer_matches_token_by_token_loop():
    x, wr, experts, shared, k = _small_layer(seed=3)
    a = O.moe_layer(x, wr, k, lambda e: experts[e], shared, residual=True).out
    b = O.moe_layer_reference_order(x, wr, k, lambda e: experts[e], shared, residual=True)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


def test_zero_weight_expert_contributes_exactly_zero():
    x, wr, experts, shared, k = _small_layer(seed=4)
    res = O.moe_layer(x, wr, k, lambda e: experts[e])
    z = int(res.topk_idx[0, 0])
    zeroed = list(experts)
    zeroed[z] = _rand_expert(None, x.shape[1], 32, zero=True)
    res0 = O.moe_layer(x, wr, k, lambda e: zeroed[e])
    # rebuild by hand: every term except expert z, with the same gate weights
    want = np.zeros_like(res.out)
    for t in range(x.shape[0]):
        for j in range(k):
            e = int(res.topk_idx[t, j])
            if e != z:
                want[t] += res.topk_w[t, j] * O.swiglu_ffn(x[t:t + 1], O.dense_expert(experts[e]))[0]
    assert np.allclose(res0.out, want, rtol=1e-12, atol=1e-15)
    all_zero = O.moe_layer(x, wr, k, lambda e: _rand_expert(None, x.shape[1], 32, zero=True))
    assert np.count_nonzero(all_zero.out) == 0


def test_shared_expert_added_with_weight_one():
    x, wr, experts, shared, k = _small_layer(seed=6)
    zero = _rand_expert(None, x.shape[1], 32, zero=True)
    res = O.moe_layer(x, wr, k, lambda e: zero, shared)
    want = O.swiglu_ffn(x, O.dense_expert(shared[0]))
    assert np.array_equal(res.out, want)


def test_residual_adds_input():
    x, wr, experts, shared, k = _small_layer(seed=7)
    a = O.moe_layer(x, wr, k, lambda e: experts[e], shared).out
    b = O.moe_layer(x, wr, k, lambda e: experts[e], shared, residual=True).out
    assert np.allclose(b - a, x, rtol=0, atol=1e-12)


def test_combine_is_linear_in_down_scales():
    # doubling every down scale (exact in fp16) doubles every routed contribution
    x, wr, experts, shared, k = _small_layer(seed=8)
    a = O.moe_layer(x, wr, k, lambda e: experts[e]).out
    doubled = [ExpertArrays(ex.gate_q, ex.gate_s, ex.up_q, ex.up_s, ex.down_q,
                            (ex.down_s.astype(np.float32) * 2).astype(np.float16)) for ex in experts]
    b = O.moe_layer(x, wr, k, lambda e: doubled[e]).out
    assert np.allclose(b, 2 * a, rtol=1e-12, atol=1e-15)


def test_forced_routing_uses_given_indices():
    x, wr, experts, shared, k = _small_layer(seed=9)
    res = O.moe_layer(x, wr, k, lambda e: experts[e])
    forced = res.topk_idx.copy()
    forced[:, [0, 1]] = forced[:, [1, 0]]
    res2 = O.moe_layer(x, wr, k, lambda e: experts[e], forced_idx=forced)
    assert np.array_equal(res2.topk_idx, forced)
    # the mixture is a sum over the selected set, so reordering the slots keeps the output
    assert np.allclose(res2.out, res.out, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ bucketing -------------

@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (5, 2, 4), (16, 2, 16), (33, 10, 512), (200, 4, 7)])
def test_bucketing_is_stable_sort_by_expert(T, k, E):
    # catches: unstable order inside a bucket, off-by-one offsets, wrong inverse
    rng = np.random.default_rng(T * 31 + E)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    b = O.bucketing(idx, E)
    flat = idx.reshape(-1)
    ref = sorted(range(T * k), key=lambda p: flat[p])      # Python's sort is stable
    assert b.sorted_pair.tolist() == ref
    assert int(b.counts.sum()) == T * k
    assert b.offsets[0] == 0 and b.offsets[-1] == T * k
    for e in range(E):
        assert b.offsets[e + 1] - b.offsets[e] == b.counts[e] == int(np.sum(flat == e))
    assert np.array_equal(b.sorted_pair[b.inv_pos], np.arange(T * k))
    assert b.active.tolist() == sorted(set(flat.tolist()))


# ------------------------------------------------------------------ bf16 rounding ---------

def test_round_to_bf16_matches_torch_on_fp32_inputs():
    # torch's own fp32 -> bf16 conversion is an independent implementation of the rounding
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.integers(-20, 20, 200000),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0, 3.0])])
    v32 = v.astype(np.float32)
    ours = O.round_to_bf16(v32.astype(np.float64))
    ref = torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_round_to_bf16_ties_to_even_by_hand():
    assert O.round_to_bf16(np.array([1.0 + 2 ** -8]))[0] == 1.0              # tie, even is 1.0
    assert O.round_to_bf16(np.array([1.0 + 3 * 2 ** -8]))[0] == 1.0 + 2 ** -6  # tie, even is up
    assert O.round_to_bf16(np.array([1.0 + 2 ** -8 + 2 ** -30]))[0] == 1.0 + 2 ** -7


def test_logit_gap():
    l = np.array([[5.0, 1.0, 3.0, 2.5]], dtype=np.float32)
    assert O.logit_gap(l, 2)[0] == 0.5
    assert O.logit_gap(l, 4)[0] == np.inf


# ---------------------------------------------------------------------------------------
# RMS normalisation (pre-norm residual block of a layer stack)
# ---------------------------------------------------------------------------------------

def test_rms_norm_hand_example():
    # [3, 4]: mean of squares 12.5, so the row is divided by sqrt(12.5 + eps)
    out = O.rms_norm(np.array([[3.0, 4.0]]), eps=0.0)
    assert np.allclose(out, [[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]], rtol=0, atol=1e-15)
    assert abs(out[0, 0] - 0.848528137423857) < 1e-14


def test_rms_norm_eps_sits_under_the_root():
    # a constant row c with c^2 == eps: c / sqrt(2 eps) = 1/sqrt(2); a zero row stays zero
    c = 1e-3
    out = O.rms_norm(np.full((1, 64), c), eps=1e-6)
    assert np.allclose(out, 1 / math.sqrt(2), rtol=1e-12)
    assert np.array_equal(O.rms_norm(np.zeros((1, 32))), np.zeros((1, 32)))


def test_rms_norm_is_per_row_and_scale_free():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(3, 256)) * np.array([[0.5], [7.0], [300.0]])
    out = O.rms_norm(x, eps=0.0)
    assert np.allclose(np.sqrt(np.mean(out * out, axis=1)), 1.0, rtol=1e-12)
    assert np.allclose(O.rms_norm(x * 19.0, eps=0.0), out, rtol=1e-12)
    assert np.all(np.sign(out) == np.sign(x))

# ------------------------------------------------------------------ 2-bit format ----------

def test_dequantize_q2_levels_and_block_scales():
    # catches: a level offset other than 1.5, codes read as signed, a block scale applied to the
    # wrong block, a factor of 2 in the levels
    c = np.zeros((2, 64), np.uint8)
    c[0, :4] = [0, 1, 2, 3]
    c[0, 32:36] = [3, 2, 1, 0]
    c[1, 40] = 3
    s = np.array([[2.0, 0.5], [1.0, 4.0]], dtype=np.float16)
    w = O.dequantize_q2(c, s)
    assert w[0, :4].tolist() == [-3.0, -1.0, 1.0, 3.0]
    assert w[0, 32:36].tolist() == [0.75, 0.25, -0.25, -0.75]
    assert w[0, 4] == -3.0 and w[0, 36] == -0.75  # code 0 is the lowest level, not zero
    assert w[1, 40] == 6.0 and w[1, 0] == -1.5


def test_q2_levels_are_symmetric_and_exact():
    # catches: asymmetric levels (c - 2 or c - 1), rounding of the level times the scale
    c = np.tile(np.arange(4, dtype=np.uint8), 8)[None, :]
    for sv in (1.0, 0.000061035156, 65504.0, 0.1):
        s = np.array([[sv]], dtype=np.float16)
        w = O.dequantize_q2(c, s)[0, :4]
        assert np.array_equal(w, -w[::-1])
        assert np.array_equal(w, float(s[0, 0]) * np.array([-1.5, -0.5, 0.5, 1.5]))


def test_q2_dense_swiglu_hand_example():
    # catches, in the 2-bit path: the level offset, gate and up swapped, down used transposed,
    # a scale on the wrong row
    g = json.load(open(os.path.join(HERE, "golden", "dense_swiglu_q2_d32_f32.json")))
    d, f = g["d"], g["f"]

    def mat(spec, r, c, dt, default):
        a = np.full((r, c), default, dtype=dt)
        for i, row in spec.items():
            for j, v in row.items():
                a[int(i), int(j)] = v
        return a
    cd, sd = g["code_default"], g["scale_default"]
    ex = ExpertArrays(mat(g["gate_c"], f, d, np.uint8, cd), mat(g["gate_s"], f, d // 32, np.float16, sd),
                      mat(g["up_c"], f, d, np.uint8, cd), mat(g["up_s"], f, d // 32, np.float16, sd),
                      mat(g["down_c"], d, f, np.uint8, cd), mat(g["down_s"], d, f // 32, np.float16, sd), fmt="q2")
    x = np.zeros((g["T"], d))
    for t, row in g["x"].items():
        for i, v in row.items():
            x[int(t), int(i)] = v
    want = np.zeros((g["T"], d))
    for t, row in g["expected_out"].items():
        for i, v in row.items():
            want[int(t), int(i)] = v
    res = O.moe_layer(x, np.ones((d, 1), dtype=np.float32), 1, lambda e: ex)
    assert np.max(np.abs(res.out - want)) <= g["tolerance_abs"]

