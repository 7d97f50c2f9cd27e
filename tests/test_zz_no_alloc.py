"""moe_permute_static, the bucketing entry point for callers that cannot allocate device
memory (for instance an engine that sizes all device memory once and lets no library add to
it). It must give exactly what moe_permute gives with a workspace, call after call, on the
same inputs; bucketing is integer work, so the comparison is bit for bit.

This file is collected last so that a run stopping at its first failure has already run
every other test."""
import numpy as np
import pytest
import torch

from routed_expert_ffn_bucketing_b300 import _lib as L

pytestmark = pytest.mark.gpu


def _topk(T, E, k, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    idx = torch.rand((T, E), generator=g).argsort(dim=1)[:, :k].to(torch.int32)
    return idx.cuda()


def _outputs(s):
    P = max(s.T * s.k, 1)
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(counts=torch.full((s.E,), -7, **i32), offsets=torch.full((s.E + 1,), -7, **i32),
                sorted_pair=torch.full((P,), -7, **i32), inv_pos=torch.full((P,), -7, **i32),
                active=torch.full((1 + min(s.E, P),), -7, **i32))


def _with_workspace(s, idx):
    o = _outputs(s)
    ws = torch.zeros(L.moe_workspace_size(s), dtype=torch.uint8, device="cuda")  # status word starts at 0
    L.moe_permute(s, idx, o["counts"], o["offsets"], o["sorted_pair"], o["inv_pos"], o["active"], ws, ws.numel())
    return o, ws


def _static(s, idx):
    o = _outputs(s)
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    L.moe_permute_static(s, idx, o["counts"], o["offsets"], o["sorted_pair"], o["inv_pos"], o["active"], status)
    return o, status


def _same(a, b, s):
    P = s.T * s.k
    for name in ("counts", "offsets", "active"):
        assert torch.equal(a[name], b[name]), name
    for name in ("sorted_pair", "inv_pos"):
        assert torch.equal(a[name][:P], b[name][:P]), name


# Two shapes per case, run back to back: the second call must not see anything the first
# left in the shared scratch.
CASES = [
    [(300, 64, 10), (200, 512, 8)],   # multi-chunk (3000 pairs), then 1600 pairs over 512 experts
    [(40, 16, 2), (3000, 128, 10)],   # one chunk (80 pairs), then 30000 pairs
    [(4, 512, 10), (4, 512, 10)],     # the decode shape twice, different routing
]


@pytest.mark.parametrize("case", CASES)
def test_static_matches_workspace_on_consecutive_calls(case):
    for n, (T, E, k) in enumerate(case):
        s = L.shape(T, 2048, 768, E, k, 1)
        idx = _topk(T, E, k, seed=1000 * n + T)
        ref, ws = _with_workspace(s, idx)
        got, status = _static(s, idx)
        torch.cuda.synchronize()
        _same(ref, got, s)
        assert int(status.item()) == 0
        # and the pair permutation is a real permutation
        P = T * k
        sp = got["sorted_pair"][:P].cpu().numpy()
        assert np.array_equal(np.sort(sp), np.arange(P))


def test_static_reports_bad_expert_in_callers_status_word():
    s = L.shape(64, 256, 128, 32, 4, 0)
    idx = _topk(64, 32, 4, seed=7)
    idx[5, 1] = 99
    got, status = _static(s, idx)
    torch.cuda.synchronize()
    assert int(status.item()) & L.MOE_DEV_BAD_EXPERT
    good = _topk(64, 32, 4, seed=8)
    got, status = _static(s, good)          # the next call starts from a clear status word
    ref, _ = _with_workspace(s, good)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _same(ref, got, s)


def test_static_rejects_sizes_beyond_its_scratch():
    s = L.shape(8192, 2048, 768, 512, 10, 1)     # 81920 pairs > 65536
    idx = torch.zeros((1,), dtype=torch.int32, device="cuda")
    o = _outputs(L.shape(1, 2048, 768, 512, 10, 1))
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    with pytest.raises(L.MoeError) as e:
        L.moe_permute_static(s, idx, o["counts"], o["offsets"], o["sorted_pair"], o["inv_pos"], o["active"], status)
    assert e.value.status == L.MOE_EUNSUPPORTED
    assert "65536" in L.moe_last_error_string()
