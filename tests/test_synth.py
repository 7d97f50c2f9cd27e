"""The seeded input generator: determinism, distribution, the block-32 quantiser's
invariants and the record packing. CPU only."""
import numpy as np
import torch

import synth


def test_splitmix64_reference_values():
    # SplitMix64 seeded with 0: published first outputs of the generator
    r = synth.draws_u64(0, 0, 3)
    assert [int(v) for v in r] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_draws_are_counter_based():
    k = synth.stream_key(7, synth.TAG_GATE, 3, 4)
    a = synth.draws_u64(k, 0, 1000)
    b = synth.draws_u64(k, 600, 400)
    assert np.array_equal(a[600:], b)
    assert synth.stream_key(7, synth.TAG_GATE, 3, 4) != synth.stream_key(7, synth.TAG_GATE, 4, 3)


def test_normal_moments():
    z = synth.normal_f32(synth.stream_key(1, 99), 0, 2_000_000, 1.0).astype(np.float64)
    assert abs(z.mean()) < 3e-3
    assert abs(z.var() - 1.0) < 5e-3
    assert np.max(np.abs(z)) <= 2 * np.sqrt(3.0) + 1e-6   # Irwin-Hall(4) support


def test_quantizer_invariants():
    w = synth.normal_f32(synth.stream_key(2, 98), 0, 64 * 256, 0.02).reshape(64, 256)
    w[3, :32] = 0.0                                      # an all-zero block
    q, s = synth.quantize_block32(w)
    assert q.dtype == np.int8 and s.dtype == np.float16 and s.shape == (64, 8)
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    sf = np.repeat(s.astype(np.float64), 32, axis=1)
    err = np.abs(q * sf - w.astype(np.float64))
    assert np.all(err <= sf / 2 + 1e-12)
    blocks = np.abs(q.astype(np.int32)).reshape(64, 8, 32).max(axis=2)
    nz = s.astype(np.float32) > 0
    assert np.all(blocks[nz] == 127)                     # the block maximum maps to +-127
    assert np.all(q[3, :32] == 0) and s[3, 0] == 0


def test_quantizer_scale_rounding_matches_torch():
    w = synth.normal_f32(synth.stream_key(3, 97), 0, 32 * 4096, 0.02).reshape(4096, 32)
    _, s = synth.quantize_block32(w)
    amax = np.abs(w).max(axis=1)
    ref = torch.from_numpy((amax / np.float32(127)).astype(np.float32)).to(torch.float16).numpy()
    assert np.array_equal(s[:, 0].view(np.uint16), ref.view(np.uint16))


def test_bf16_bits_match_torch():
    v = synth.normal_f32(synth.stream_key(4, 96), 0, 100000, 3.0)
    ours = synth.fp32_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_record_pack_roundtrip_and_layout():
    L = synth.record_layout(2048, 768)
    assert L.record_bytes == 5013504
    assert (L.gate_q, L.up_q, L.down_q, L.gate_s, L.up_s, L.down_s) == (
        0, 1572864, 3145728, 4718592, 4816896, 4915200)
    assert synth.record_layout(256, 128).record_bytes == 104448
    a = synth.expert_arrays(0, 1, 2, 64, 32)
    rec = synth.pack_record(a)
    b = synth.unpack_record(rec, 64, 32)
    for name in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        assert np.array_equal(getattr(a, name).view(np.uint8), getattr(b, name).view(np.uint8))


def test_expert_streams_are_distinct():
    a = synth.expert_arrays(0, 0, 0, 64, 32)
    b = synth.expert_arrays(0, 0, 1, 64, 32)
    c = synth.expert_arrays(0, 1, 0, 64, 32)
    assert not np.array_equal(a.gate_q, b.gate_q) and not np.array_equal(a.gate_q, c.gate_q)
    assert not np.array_equal(a.gate_q, a.up_q)


def test_zipf_scales_give_skewed_popularity():
    c, freq = synth.zipf_column_scales(512, 10, 1.1, 0)
    assert abs(freq.sum() - 10.0) < 1e-9
    assert np.all(np.diff(c) <= 0)
    r = np.arange(1, 513)
    slope = np.polyfit(np.log(r[4:]), np.log(np.maximum(freq[4:], 1e-4)), 1)[0]
    assert -1.6 < slope < -0.8
    assert freq[0] > 0.3 and freq[-1] < 0.01


def test_router_zipf_columns_follow_permutation():
    w = synth.router_weights(0, 5, 64, 32, 1.0, zipf_s=1.1, k=4)
    base = synth.router_weights(0, 5, 64, 32, 1.0)
    c, _ = synth.zipf_column_scales(32, 4, 1.1, 0)
    perm = synth.expert_rank_permutation(0, 5, 32)
    assert np.array_equal(w[:, perm[0]], (base[:, perm[0]] * c[0]).astype(np.float32))


def test_interleaved_code_order():
    # in each 64-code span, 16-byte chunk c holds codes 8c..8c+7 of the first block, then
    # 8c..8c+7 of the second; a trailing unpaired block stays in place
    K = 160  # two pairs and one unpaired block
    q = np.arange(K, dtype=np.int64).reshape(1, K)
    st = synth.interleave_codes(q)[0]
    assert list(st[:16]) == list(range(0, 8)) + list(range(32, 40))
    assert list(st[16:32]) == list(range(8, 16)) + list(range(40, 48))
    assert list(st[48:64]) == list(range(24, 32)) + list(range(56, 64))
    assert list(st[64:80]) == list(range(64, 72)) + list(range(96, 104))
    assert list(st[128:]) == list(range(128, 160))
    assert np.array_equal(synth.deinterleave_codes(synth.interleave_codes(q)), q)
    # the device generator's position rule, written out here independently
    def pos(k):
        if k >= K // 64 * 64:
            return k
        p, h, c, i = k // 64, (k // 32) % 2, (k // 8) % 4, k % 8
        return 64 * p + 16 * c + 8 * h + i
    assert all(st[pos(k)] == k for k in range(K))
