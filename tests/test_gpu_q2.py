"""The sub-4-bit expert format (2-bit codes, one fp16 scale per 32 weights, W = s (c - 1.5)) in
the decode expert FFN, through the C-ABI, against the CPU oracle on the same seeded inputs."""
import numpy as np
import pytest

import synth
from routed_expert_ffn_bucketing_b300 import _lib as L
from synth.device import DeviceLayer
from synth.workloads import WORKLOADS, custom

from gpu_util import check_bucketing, check_output, check_routing, run_layer

pytestmark = pytest.mark.gpu


def test_device_generator_matches_numpy_q2():
    w = custom("decode_q2", E=3, n_shared=1)
    dl = DeviceLayer(w, layer=2)
    for e in range(4):
        assert np.array_equal(dl.record_bytes_of(e), synth.pack_record(w.expert(2, e))), e
    a = synth.unpack_record(dl.record_bytes_of(1), w.d, w.f, synth.FMT_Q2)
    assert a.fmt == "q2" and a.gate_q.max() <= 3


@pytest.mark.parametrize("T,E,k,ns", [(4, 32, 4, 1), (1, 16, 2, 0), (8, 64, 8, 2), (3, 8, 8, 1)])
def test_q2_decode_small(T, E, k, ns):
    w = custom("tiny", T=T, E=E, k=k, n_shared=ns, d=256, f=256, router_sigma=1.0, fmt=synth.FMT_Q2)
    dl = DeviceLayer(w)
    for batch in range(2):
        run = run_layer(dl, batch)
        assert run.status == 0
        check_routing(run, w)
        check_bucketing(run, w)
        check_output(run, w)


def test_q2_decode_full_size():
    # T = 4, d = 2048, f = 768, E = 512, top-10 + 1 shared: every output element against the oracle
    w = WORKLOADS["decode_q2"]
    dl = DeviceLayer(w)
    for batch in range(2):
        run = run_layer(dl, batch)
        assert run.status == 0
        _, _, n = check_routing(run, w)
        assert n == w.T
        check_bucketing(run, w)
        check_output(run, w)


def test_q2_bf16_y_and_residual():
    w = custom("decode_q2", T=4)
    dl = DeviceLayer(w)
    run = run_layer(dl, 3, residual=True, ydt=L.MOE_BF16)
    assert run.status == 0
    check_output(run, w, residual=True)
