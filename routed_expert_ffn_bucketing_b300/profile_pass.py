"""A few passes of one MoE layer of a named synthetic workload, for an external profiler.

    python -m routed_expert_ffn_bucketing_b300.profile_pass decode --passes 4

One layer's experts are resident (the decode and prefill layers hold about 2.6 GB of records),
each pass is one moe_layer_forward call on the next seeded input batch, launched eagerly on the
current stream, and the program checks the device status word at the end. Every kernel of a
pass is the library's; the launches are those a profiler such as ncu lists or captures (one
pass launches the router, the routing tail, the expert FFN kernels and the combine).
"""
from __future__ import annotations

import argparse

import torch

from . import _lib as L
from . import layer as lay


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("workload", help="tiny, decode, decode_q2 or prefill")
    ap.add_argument("--passes", type=int, default=4)
    args = ap.parse_args()
    if not torch.cuda.is_available():
        raise SystemExit("profile_pass needs a CUDA device")
    from synth.device import DeviceLayer
    from synth.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if w.layers > 1:
        raise SystemExit(f"{args.workload} is a multi-layer workload; profile one of its layers as 'decode'")
    dl = DeviceLayer(w)
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    # y_perm as bench.py runs each workload: fp32 for decode, bf16 for prefill
    buf = lay.alloc_buffers(s, ydt=L.MOE_BF16 if w.T > 16 else L.MOE_F32, odt=L.MOE_BF16, keep_logits=False)
    table = L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of, dl.shared_ptr, fmt=w.fmt)
    xs = [dl.x(b) for b in range(min(args.passes, 4))]
    for i in range(args.passes):
        lay.forward(buf, xs[i % len(xs)], dl.router, table, fused=True)
    torch.cuda.synchronize()
    st = L.moe_read_status(buf.ws)
    if st:
        raise SystemExit(f"device status {st:#x} after {args.passes} passes")
    print(f"{args.workload}: {args.passes} passes, status 0")


if __name__ == "__main__":
    main()
