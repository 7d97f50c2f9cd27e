"""Failure paths of the expert-FFN kernels on the GPU, made on purpose with no fault: a short
limit on the kernels' bounded waits makes them run out (the kernel sets MOE_DEV_TIMEOUT,
abandons its work, drains its copies and tensor-core operations and exits), after which the
context still works and the same call gives correct results again. And AUTO refuses, on the
host, a many-token shape that only the slow SIMT kernels could run."""
import numpy as np
import pytest

from routed_expert_ffn_bucketing_b300 import _lib as L
from synth.device import DeviceLayer
from synth.workloads import custom

from gpu_util import check_output, check_routing, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture
def restore_wait_limit():
    yield
    L.moe_set_wait_limit(0)


@pytest.mark.parametrize("mode,T", [(L.MOE_MODE_PREFILL, 300), (L.MOE_MODE_DECODE, 4)])
def test_short_wait_limit_times_out_and_context_survives(restore_wait_limit, mode, T):
    w = custom("tiny", T=T, E=64, k=10, n_shared=1, d=2048, f=768, router_sigma=1.0)
    dl = DeviceLayer(w)
    L.moe_set_wait_limit(1)  # 1 ns: every wait that does not succeed at once runs out
    run = run_layer(dl, 0, mode=mode)
    if mode == L.MOE_MODE_PREFILL:
        # the MMA thread's first wait for a TMA tile cannot succeed within 16 polls
        assert run.status == L.MOE_DEV_TIMEOUT, hex(run.status)
    else:
        # the persistent kernel's waits for other CTAs' gate/up work: timed out or not, no
        # other error bit
        assert run.status in (0, L.MOE_DEV_TIMEOUT), hex(run.status)
    L.moe_set_wait_limit(0)
    run = run_layer(dl, 0, mode=mode)
    assert run.status == 0
    check_output(run, w, tokens=np.arange(0, T, 7))


def test_auto_refuses_many_tokens_on_a_shape_without_the_gemm():
    # d = 96 is not a multiple of 256: the tensor-core GEMM cannot take it
    w = custom("tiny", T=40, E=16, k=2, n_shared=0, d=96, f=64, router_sigma=1.0)
    dl = DeviceLayer(w, fill="host")
    with pytest.raises(L.MoeError) as e:
        run_layer(dl, 0, mode=L.MOE_MODE_AUTO)
    assert e.value.status == L.MOE_EUNSUPPORTED and "MOE_MODE_DECODE" in str(e.value)
    run = run_layer(dl, 0, mode=L.MOE_MODE_DECODE)  # the explicit request runs the SIMT kernels
    assert run.status == 0
    check_routing(run, w)  # d % 256 != 0: the router is the fp32 SIMT GEMM, not the tensor-core one
    check_output(run, w)


def test_counters_left_at_zero_for_the_next_call(restore_wait_limit):
    # the decode expert FFN keeps counters in the workspace that must read zero at every launch:
    # three FFN calls on one routing with no moe_route between them (which would clear them), the
    # middle one with a wait limit that runs out; the first and last give the same bits
    import torch
    from routed_expert_ffn_bucketing_b300 import layer as lay
    w = custom("decode", T=4)
    dl = DeviceLayer(w)
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    buf = lay.alloc_buffers(s)
    x = dl.x(2)
    table = L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of, dl.shared_ptr)
    L.moe_route(s, x, L.MOE_BF16, dl.router, buf.topk_idx, buf.topk_w, None, buf.ws, buf.ws_bytes)
    L.moe_permute(s, buf.topk_idx, buf.counts, buf.offsets, buf.sorted_pair, buf.inv_pos, buf.active, buf.ws,
                  buf.ws_bytes)

    def ffn():
        L.moe_expert_ffn(s, L.MOE_MODE_DECODE, x, L.MOE_BF16, table, buf.offsets, buf.sorted_pair, buf.active,
                         buf.y_perm, buf.ydt, buf.ws, buf.ws_bytes)
        torch.cuda.synchronize()
        return buf.y_perm.clone()

    y1 = ffn()
    assert L.moe_read_status(buf.ws) == 0
    y2 = ffn()
    assert torch.equal(y1, y2)
    L.moe_set_wait_limit(1)
    ffn()
    assert L.moe_read_status(buf.ws) in (0, L.MOE_DEV_TIMEOUT)
    L.moe_set_wait_limit(0)
    y4 = ffn()
    assert torch.equal(y1, y4)
