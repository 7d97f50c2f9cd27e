"""Benchmark of one sparse MoE layer's forward pass on B300 (the decode workload by default).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload decode]

A step is one whole pass (router + top-k, bucketing, slot-table lookup inside the expert
FFN, SwiGLU experts, combine) over one batch of T tokens. Batches rotate over 16 seeded
inputs, so each step routes to its own experts. A 512 MiB buffer (larger than the 126 MB
L2) is written between timed steps, outside the timed events. Times are CUDA events on
the launching stream, and the maximum is taken over ranks. One JSON line is printed by rank 0.

--impl reference times the CPU oracle on this host's cores instead, over the same
workload and metric (one oracle layer pass per step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

# the CPU oracle is timed on one core: fix the BLAS thread count before numpy loads
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; decode HBM GB/s & prefill int8 TOPS as % of B300 peak"
N_BATCHES = 16
FLUSH_BYTES = 512 << 20

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the dominant kernel(s),
# from one ncu capture of the current kernels (the summaries in profiles/ give the command). A
# capture is of one launch, i.e. one batch: the decode FFN's algorithmic bytes vary by batch.
TRAFFIC = {
    "decode": {"bytes": 186_220_288 + 3_603_200, "kernel": "ffn_persist_kernel<8, 8>",
               "capture": "profiles/ffn_persist_decode_T4.md (one launch)"},
    "prefill": {"bytes": 2_721_439_000 + 241_189_888 + 1_198_355_000 + 314_232_576,
                "kernel": "prefill_gemm_kernel<0> + prefill_gemm_kernel<1>",
                "capture": "profiles/prefill_gemm_T8192.md (one launch each; gather and h conversion not included)"},
}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6400.0, 1800.0, "fallback"


# ------------------------------------------------------------------ clocks ----------------

class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.path = index, None, None

    def start(self):
        try:
            self.path = f"/tmp/moe_bench_clocks_{os.getpid()}.csv"
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [c.strip() for c in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx = float(f[2])
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
            os.unlink(self.path)
        except Exception:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle ------------

def _gen_expert(args):
    import synth
    seed, layer, e, d, f, sigma = args
    return e, synth.expert_arrays(seed, layer, e, d, f, sigma)


def oracle_experts(w, layer: int, ids, workers: int):
    """Expert arrays for the oracle, made by the numpy generator in a spawn process pool."""
    import concurrent.futures as cf
    import multiprocessing as mp
    ids = sorted(set(int(e) for e in ids))
    jobs = [(w.seed, layer, e, w.d, w.f, w.expert_sigma) for e in ids]
    with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
        return dict(ex.map(_gen_expert, jobs))


ORACLE_MAX_TOKENS = 64  # tokens per oracle pass: large batches are timed on their first rows


def prepare_oracle(w, batches):
    """Inputs of the timed oracle passes: activations (at most ORACLE_MAX_TOKENS rows of each
    batch), router and every expert those rows route to (made before, and outside, the timing)."""
    from oracle import moe_oracle as O
    router = w.router(0)
    xs = [w.x_f64(b)[:ORACLE_MAX_TOKENS] for b in batches]
    need = set()
    for x in xs:
        need |= set(O.select_topk(O.router_logits(x, router), w.k).reshape(-1).tolist())
    need |= {w.E + s for s in range(w.n_shared)}
    ex = oracle_experts(w, 0, need, workers=max(1, min(16, os.cpu_count() or 1)))
    return xs, router, ex


def time_oracle(w, prep, budget_s: float, max_steps: int | None = None):
    """Times the oracle's layer pass over the prepared batches, one batch per step, on one
    thread. Returns (tokens/s, steps, seconds, threads)."""
    from oracle import moe_oracle as O
    xs, router, ex = prep
    shared = [ex[w.E + s] for s in range(w.n_shared)]
    steps, t0 = 0, time.perf_counter()
    while True:
        O.moe_layer(xs[steps % len(xs)], router, w.k, lambda e: ex[e], shared)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps is not None and steps >= max_steps):
            break
    return xs[0].shape[0] * steps / el, steps, el, int(os.environ.get("OPENBLAS_NUM_THREADS", "1"))


# ------------------------------------------------------------------ distributed -----------

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("MOE_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
    return ws, rank, local


def dist_max(v: float, ws: int, device) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ reference arm ---------

def run_reference(args, ws, rank):
    if rank != 0:
        return
    from synth.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    K, W = args.steps, args.warmup
    batches = list(range(4))
    prep = prepare_oracle(w, batches)
    # W untimed oracle passes, then K timed ones (one batch of T tokens per step), stopping
    # early once 150 s have passed so that the run stays within a few minutes
    time_oracle(w, prep, budget_s=1e9, max_steps=max(W, 1))
    tps, steps, el, cores = time_oracle(w, prep, budget_s=150.0, max_steps=K)
    sample = (f"{steps} oracle layer passes over {len(batches)} rotating batches of "
              f"{min(w.T, ORACLE_MAX_TOKENS)} tokens of T={w.T}")
    if w.layers > 1:
        tps /= w.layers
        sample += f" (layer 0); tokens/s divided by the {w.layers} layers of a step"
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps,
        "warmup": W, "ms_per_step": 1e3 * el / steps * w.layers, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": w.describe(), "tokens_per_step": w.T},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm ---------------

def run_ours(args, ws, rank, local):
    import torch
    from routed_expert_ffn_bucketing_b300 import _lib as L
    from routed_expert_ffn_bucketing_b300 import layer as lay
    from synth.device import DeviceLayer
    from synth.workloads import WORKLOADS

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    K, W = args.steps, args.warmup
    hbm_peak, bf16_peak, peak_kind = peaks()

    prefill = w.T > 16
    n_batches = 4 if prefill else N_BATCHES
    dl = DeviceLayer(w, device=str(dev))
    xs = [dl.x(b) for b in range(n_batches)]
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    # prefill writes y_perm in bf16 (half the combine's reads); decode keeps fp32
    buf = lay.alloc_buffers(s, device=dev, ydt=L.MOE_BF16 if prefill else L.MOE_F32, odt=L.MOE_BF16,
                            keep_logits=False)
    table = L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of, dl.shared_ptr)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    xdt = L.MOE_BF16

    def step(x):
        lay.forward(buf, x, dl.router, table, L.MOE_MODE_AUTO, stream=stream, fused=True)

    # active experts per batch (for the algorithmic byte count), from untimed passes
    n_active = []
    for b in range(n_batches):
        step(xs[b])
        torch.cuda.synchronize(dev)
        n_active.append(int(buf.active[0].item()))
        assert L.moe_read_status(buf.ws) == 0
    for i in range(W):
        flush.fill_(i & 0xFF)
        step(xs[i % n_batches])
    torch.cuda.synchronize(dev)

    # The timed steps replay CUDA graphs of the C-ABI calls, one graph per stage and batch:
    # (route + permute), expert FFN with the combine (moe_expert_ffn_combine). The kernels
    # and their arguments are those of the eager calls; the graphs only take the host's launch
    # cost out of the device time.
    def seg_route(x):
        L.moe_route(s, x, xdt, dl.router, buf.topk_idx, buf.topk_w, None, buf.ws, buf.ws_bytes, None)
        L.moe_permute(s, buf.topk_idx, buf.counts, buf.offsets, buf.sorted_pair, buf.inv_pos, buf.active, buf.ws,
                      buf.ws_bytes, None)

    def seg_ffn_combine(x):
        L.moe_expert_ffn_combine(s, L.MOE_MODE_AUTO, x, xdt, table, buf.offsets, buf.sorted_pair, buf.active,
                                 buf.y_perm, buf.ydt, buf.inv_pos, buf.topk_w, None, buf.out, buf.odt, buf.ws,
                                 buf.ws_bytes, None)

    # for the breakdown: the same kernels as two calls
    def seg_ffn(x):
        L.moe_expert_ffn(s, L.MOE_MODE_AUTO, x, xdt, table, buf.offsets, buf.sorted_pair, buf.active, buf.y_perm,
                         buf.ydt, buf.ws, buf.ws_bytes, None)

    def seg_comb(x):
        L.moe_combine(s, buf.y_perm, buf.ydt, buf.inv_pos, buf.topk_w, None, buf.out, buf.odt, None)

    cap = torch.cuda.Stream(dev)
    graphs, layer_graphs = [], []
    for b in range(n_batches):
        gs = []
        for seg in (seg_route, seg_ffn, seg_comb):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                seg(xs[b])
            gs.append(g)
        graphs.append(gs)
        g = torch.cuda.CUDAGraph()  # the whole layer: the four calls in one graph
        with torch.cuda.graph(g, stream=cap):
            seg_route(xs[b])
            seg_ffn_combine(xs[b])
        layer_graphs.append(g)
    for i in range(W):
        flush.fill_(i & 0xFF)
        for g in graphs[i % n_batches]:
            g.replay()
        layer_graphs[i % n_batches].replay()
    torch.cuda.synchronize(dev)

    # timed region 1 (the headline): one whole-layer graph per step
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize(dev)
    clocks.start()
    t_wall = time.perf_counter()
    for i in range(K):
        flush.fill_(i & 0xFF)
        a, b = ev_step[i]
        a.record(stream)
        layer_graphs[i % n_batches].replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev_step]

    # timed region 2 (the breakdown and the expert-FFN roofline): one graph per stage, events between
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize(dev)
    for i in range(K):
        flush.fill_(i & 0xFF)
        g_route, g_ffn, g_comb = graphs[i % n_batches]
        e0, e1, e2, e3 = ev[i]
        e0.record(stream)
        g_route.replay()
        e1.record(stream)
        g_ffn.replay()
        e2.record(stream)
        g_comb.replay()
        e3.record(stream)
    torch.cuda.synchronize(dev)
    assert L.moe_read_status(buf.ws) == 0, "a kernel reported an error during the timed steps"
    staged_ms = [a.elapsed_time(d) for a, _, _, d in ev]
    ffn_ms = [b.elapsed_time(c) for _, b, c, _ in ev]
    route_ms = [a.elapsed_time(b) for a, b, _, _ in ev]
    comb_ms = [c.elapsed_time(d) for _, _, c, d in ev]
    total_s = dist_max(sum(step_ms) / 1e3, ws, dev)
    value = ws * w.T * K / total_s

    # algorithmic bytes of the expert-FFN call: each selected expert's record once, the T
    # activation rows read, the y_perm rows written (fp32); scratch (h) is not counted
    rows = w.P + w.T * w.n_shared
    small = w.T * w.d * 2 + rows * w.d * 4
    ffn_bytes = [(n_active[i % n_batches] + w.n_shared) * w.record_bytes + small for i in range(K)]
    achieved = sum(ffn_bytes) / (sum(ffn_ms) / 1e3) / 1e9
    if prefill:
        # tensor-bound: algorithmic FLOPs of the expert FFN (gate, up and down over every row)
        ffn_flops = 2.0 * rows * 3 * w.d * w.f
        tflops = ffn_flops / (sum(ffn_ms) / 1e3 / K) / 1e12
        roofline = {"kernel": "moe_expert_ffn (grouped GEMM: gate/up + SwiGLU, down)", "bound": "tensor",
                    "achieved": tflops, "peak": bf16_peak, "unit": "TFLOP/s", "frac": tflops / bf16_peak,
                    "peak_kind": f"{peak_kind} dense bf16 (the f16 dense rate is the same)",
                    "traffic": TRAFFIC["prefill"]["bytes"], "traffic_source": TRAFFIC["prefill"],
                    "flops_per_launch": ffn_flops, "ms_per_launch": sum(ffn_ms) / K}
    else:
        roofline = {"kernel": "moe_expert_ffn (persistent kernel: gate/up + SwiGLU, down)", "bound": "hbm",
                    "achieved": achieved,
                    "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                    "peak_kind": f"{peak_kind} copy bandwidth",
                    "traffic": TRAFFIC["decode"]["bytes"], "traffic_source": TRAFFIC["decode"],
                    "bytes_per_launch": float(np.mean(ffn_bytes)), "ms_per_launch": sum(ffn_ms) / K}
    router_bytes = w.d * w.E * 4
    step_bytes = [b + router_bytes for b in ffn_bytes]
    step_gbs = sum(step_bytes) / (sum(step_ms) / 1e3) / 1e9

    # end to end through the public API with host buffers: pinned x in, bf16 out back, per step
    x_host = [x.cpu().pin_memory() for x in xs]
    out_host = torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(xs[0])
    e2e_s = 0.0
    for i in range(W + K):
        flush.fill_(i & 0xFF)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        x_dev.copy_(x_host[i % n_batches], non_blocking=True)
        step(x_dev)
        out_host.copy_(buf.out, non_blocking=True)
        torch.cuda.synchronize(dev)
        if i >= W:
            e2e_s += time.perf_counter() - t0
    e2e_s = dist_max(e2e_s, ws, dev)
    e2e = {"value": ws * w.T * K / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": w.T * w.d * 2,
           "d2h_bytes_per_step": w.T * w.d * 2}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tps, steps, el, cores = time_oracle(w, prepare_oracle(w, list(range(4))), budget_s=args.cpu_seconds)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{steps} oracle layer passes ({el:.1f} s) over 4 rotating batches of "
                         f"{min(w.T, ORACLE_MAX_TOKENS)} tokens of T={w.T}"}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": sum(step_ms) / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded)",
        "config": {"workload": w.describe(), "tokens_per_step": w.T, "weights": "int8 block-32 + fp16 scales",
                   "activations": "bf16", "l2": "512 MiB buffer written between timed steps (outside events)",
                   "batches": n_batches, "mean_active_experts": float(np.mean(n_active)),
                   "launch": "one CUDA graph of the three C-ABI calls per step: moe_route, moe_permute, "
                             "moe_expert_ffn_combine (stages_ms: the same kernels as moe_expert_ffn and "
                             "moe_combine, one graph per stage, events between)",
                   "parallelism": f"replicas x{ws}"},
        "roofline": roofline,
        "stages_ms": {"route_permute": sum(route_ms) / K, "expert_ffn": sum(ffn_ms) / K,
                      "combine": sum(comb_ms) / K, "step_as_three_graphs": sum(staged_ms) / K},
        "step_hbm_gbs": step_gbs,
        "wall_s": wall,
        "e2e": e2e,
        "cpu_baseline": cpu,
        # kernels per step: decode 4 (router GEMV, top-k, bucketing, persistent expert FFN with
        # the combine); prefill 11 (router GEMM, top-k, 3 bucketing, 5 expert FFN, combine)
        "gpu_launches": (11 if prefill else 4) * K,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ multi-layer workloads ---

def stack_cpu_baseline(w, rank, args):
    """The oracle on one layer (layer 0's router and experts) at T tokens, extrapolated to the
    L-layer step by dividing its tokens/s by L."""
    if rank != 0 or args.no_cpu_baseline:
        return None
    tps, steps, el, cores = time_oracle(w, prepare_oracle(w, list(range(4))), budget_s=args.cpu_seconds)
    return {"value": tps / w.layers, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{steps} oracle passes ({el:.1f} s) of one layer (layer 0) over 4 rotating batches of "
                      f"T={w.T}; tokens/s divided by the {w.layers} layers of a step"}


def run_stack(args, ws, rank, local, w):
    """L resident layers on a residual stream; one CUDA graph of the whole L-layer step."""
    import torch
    from routed_expert_ffn_bucketing_b300 import _lib as L
    from routed_expert_ffn_bucketing_b300.stack import DecodeStack, LayerWeights
    from synth.device import DeviceLayer

    dev = torch.device("cuda", local)
    K, W = args.steps, args.warmup
    hbm_peak, _, peak_kind = peaks()
    need = w.layers * (w.E + w.n_shared) * w.record_bytes
    free, _ = torch.cuda.mem_get_info(dev)
    if need > free - (4 << 30):
        raise SystemExit(f"stack workload needs {need / 1e9:.1f} GB of device memory, {free / 1e9:.1f} GB free")
    dls = [DeviceLayer(w, layer=l, device=str(dev)) for l in range(w.layers)]
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    st = DecodeStack(s, [LayerWeights(dl.router, L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of,
                                                                dl.shared_ptr)) for dl in dls], device=dev)
    n_batches = 4
    xs = [dls[0].x(b) for b in range(n_batches)]
    stream = torch.cuda.current_stream(dev)
    # experts per layer and batch (for the algorithmic bytes), from untimed eager passes
    n_active = []
    for b in range(n_batches):
        keep = []
        st.forward(xs[b], keep=keep)
        torch.cuda.synchronize(dev)
        assert L.moe_read_status(st.buf.ws) == 0
        n_active.append([int(np.unique(r[1].cpu().numpy()).size) for r in keep if r[0] == "idx"])
    cap = torch.cuda.Stream(dev)
    graphs = []
    for b in range(n_batches):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            st.forward(xs[b])
        graphs.append(g)
    for i in range(W):
        graphs[i % n_batches].replay()
    torch.cuda.synchronize(dev)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize(dev)
    clocks.start()
    for i in range(K):
        a, b = ev[i]
        a.record(stream)
        graphs[i % n_batches].replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clk = clocks.stop()
    assert L.moe_read_status(st.buf.ws) == 0, "a kernel reported an error during the timed steps"
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_s = dist_max(sum(step_ms) / 1e3, ws, dev)
    value = ws * w.T * K / total_s
    small = w.T * w.d * 2 + (w.P + w.T * w.n_shared) * w.d * 4
    layer_bytes = [[(n + w.n_shared) * w.record_bytes + w.d * w.E * 4 + small for n in na] for na in n_active]
    step_bytes = [sum(layer_bytes[i % n_batches]) for i in range(K)]
    achieved = sum(step_bytes) / (sum(step_ms) / 1e3) / 1e9

    # end to end: pinned x in, the eager stack through the public API, bf16 out back
    x_host = [x.cpu().pin_memory() for x in xs]
    out_host = torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(xs[0])
    K_e2e = min(K, 50)
    e2e_s = 0.0
    for i in range(W + K_e2e):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        x_dev.copy_(x_host[i % n_batches], non_blocking=True)
        out_host.copy_(st.forward(x_dev), non_blocking=True)
        torch.cuda.synchronize(dev)
        if i >= W:
            e2e_s += time.perf_counter() - t0
    e2e_s = dist_max(e2e_s, ws, dev)
    cpu = stack_cpu_baseline(w, rank, args)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": sum(step_ms) / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded)",
        "config": {"workload": w.describe(), "tokens_per_step": w.T, "weights": "int8 block-32 + fp16 scales",
                   "resident_gb": need / 1e9, "activations": "bf16 residual stream",
                   "l2": "inputs larger than L2 (each step reads every layer's selected experts, ~10 GB)",
                   "batches": n_batches, "mean_active_experts_per_layer": float(np.mean(n_active)),
                   "launch": f"one CUDA graph of the {4 * w.layers} C-ABI calls of a step (norm, route, permute, "
                             "expert FFN with the combine, per layer)",
                   "block": "pre-norm residual: x + MoE(rms_norm(x)), eps 1e-6, no gain",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"kernel": f"whole {w.layers}-layer step (route, permute, expert FFN, combine per layer)",
                     "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_kind": f"{peak_kind} copy bandwidth", "traffic": None,
                     "bytes_per_step": float(np.mean(step_bytes)), "ms_per_step": sum(step_ms) / K},
        "e2e": {"value": ws * w.T * K_e2e / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": w.T * w.d * 2,
                "d2h_bytes_per_step": w.T * w.d * 2, "steps": K_e2e, "launch": "eager C-ABI calls"},
        "cpu_baseline": cpu,
        "gpu_launches": 5 * w.layers * K,  # per layer: norm, router GEMV, top-k, bucketing, expert FFN + combine
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def _host_images(w, n_img: int, dev):
    """Pinned host records of the first n_img experts in (layer, expert) order, made on the
    device by the seeded generator and copied back in chunks."""
    import torch
    from synth.gpu import fill_expert_records
    rb = w.record_bytes
    host = torch.empty((n_img, rb), dtype=torch.uint8, pin_memory=True)
    chunk = 256
    tmp = torch.empty((chunk, rb), dtype=torch.uint8, device=dev)
    i = 0
    while i < n_img:
        l, e = divmod(i, w.E)
        n = min(chunk, n_img - i, w.E - e)
        fill_expert_records(w.seed, l, e, n, w.d, w.f, tmp.data_ptr(), rb, w.expert_sigma)
        host[i:i + n].copy_(tmp[:n])
        i += n
    torch.cuda.synchronize(dev)
    return host


def run_tiered(args, ws, rank, local, w):
    """L layers, experts in pinned host memory, a device pool of w.slots slots; Zipf routing
    whose hot set drifts every few steps. Wall-clock tokens/s, hit rate and H2D GB/s."""
    import torch
    import synth
    from routed_expert_ffn_bucketing_b300 import _lib as L
    from routed_expert_ffn_bucketing_b300.stack import TieredStack
    from synth.gpu import fill_expert_records

    dev = torch.device("cuda", local)
    K, W = args.steps, args.warmup
    rb = w.record_bytes
    n_all = w.layers * w.E
    with open("/proc/meminfo") as f:
        avail = next(int(l.split()[1]) * 1024 for l in f if l.startswith("MemAvailable"))
    n_img = int(min(n_all, args.host_gb * 1e9 // rb, 0.5 * avail // rb))
    host = _host_images(w, n_img, dev)
    h_records = [host[i % n_img].data_ptr() for i in range(n_all)]
    shared = []
    for l in range(w.layers):
        t = torch.empty(max(w.n_shared, 1) * rb, dtype=torch.uint8, device=dev)
        if w.n_shared:
            fill_expert_records(w.seed, l, w.E, w.n_shared, w.d, w.f, t.data_ptr(), rb, w.expert_sigma)
        shared.append(t)
    base = [torch.from_numpy(synth.router_weights_unscaled(w.seed, l, w.d, w.E, w.router_sigma)).to(dev)
            for l in range(w.layers)]
    perms = [synth.expert_rank_permutation(w.seed, l, w.E) for l in range(w.layers)]
    routers = [torch.empty_like(b) for b in base]

    def set_routers():
        for l in range(w.layers):
            col = synth.router_column_scales(perms[l], w.E, w.k, w.zipf_s, w.seed)
            torch.mul(base[l], torch.from_numpy(col).to(dev)[None, :], out=routers[l])

    set_routers()
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    policy = L.MOE_SLOT_FREQ if args.slot_policy == "freq" else L.MOE_SLOT_LRU
    profile = None
    if args.warm_profile:
        # the usage profile a deployment would ship: each expert's inclusion frequency under the
        # routing at step 0 (before any drift)
        _, freq = synth.zipf_column_scales(w.E, w.k, w.zipf_s, w.seed)
        profile = np.zeros(n_all, dtype=np.float32)
        for l in range(w.layers):
            profile[l * w.E + perms[l]] = freq
    ts = TieredStack(s, w.layers, routers, h_records, w.slots, rb, shared, device=dev, policy=policy,
                     half_life_steps=args.half_life_steps, profile=profile)
    n_batches = 16
    x_host = [torch.from_numpy(w.x_bits(b).astype(np.int16)).view(torch.bfloat16).pin_memory()
              for b in range(n_batches)]
    x_dev = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=dev)
    out_host = torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory()

    # H2D copy rate of this host's pinned memory: one 2 GB copy after a warm one
    probe = host[:max(1, min(n_img, (2 << 30) // rb))]
    pd = torch.empty_like(probe, device=dev)
    pcie = 0.0
    for _ in range(2):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        pd.copy_(probe, non_blocking=True)
        b.record()
        torch.cuda.synchronize(dev)
        pcie = probe.numel() / (a.elapsed_time(b) / 1e3) / 1e9
    del pd

    launches = [0]

    def run(step0, n, e2e):
        wall = 0.0
        for i in range(step0, step0 + n):
            if i and i % synth.DRIFT_EVERY == 0:
                for l in range(w.layers):
                    perms[l] = synth.drift_rank_permutation(perms[l], w.seed, l, i // synth.DRIFT_EVERY)
                set_routers()
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            x_dev.copy_(x_host[i % n_batches], non_blocking=True)
            y = ts.forward(x_dev)
            if e2e:
                out_host.copy_(y, non_blocking=True)
            torch.cuda.synchronize(dev)
            wall += time.perf_counter() - t0
            # per layer: norm, router GEMV, top-k, bucketing, expert FFN with the combine; with misses
            # one more FFN call and a separate combine
            launches[0] += sum(5 + 2 * (m > 0) for m in ts.layer_misses)
        return wall

    try:
        run(0, W, False)
        launches[0] = 0
        s0 = L.slot_table_stats(ts.table)
        clocks = ClockSampler(local)
        barrier(ws)
        clocks.start()
        wall = run(W, K, True)
        barrier(ws)
        clk = clocks.stop()
        s1 = L.slot_table_stats(ts.table)
        assert L.moe_read_status(ts.buf.ws) == 0, "a kernel reported an error during the timed steps"
    finally:
        ts.close()
    wall = dist_max(wall, ws, dev)
    hits, misses = s1.hits - s0.hits, s1.misses - s0.misses
    h2d = s1.bytes_h2d - s0.bytes_h2d
    value = ws * w.T * K / wall
    cpu = stack_cpu_baseline(w, rank, args)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": 1e3 * wall / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded)",
        "config": {"workload": w.describe() + f", {w.slots} device slots, drift every {synth.DRIFT_EVERY} steps",
                   "tokens_per_step": w.T, "weights": "int8 block-32 + fp16 scales",
                   "pool_gb": w.slots * rb / 1e9, "host_images": n_img,
                   "host_mapping": "(l*E + e) mod host_images" if n_img < n_all else "one image per expert",
                   "timing": "wall clock per step (the host reads each layer's active list), x copied in and "
                             "the output copied out inside every step",
                   "parallelism": f"replicas x{ws}"},
        "slot_pool": {"policy": "LRU" if policy == L.MOE_SLOT_LRU else
                      f"decayed use count (half-life {args.half_life_steps:g} steps)",
                      "warm_profile": bool(args.warm_profile), "warm_loads": ts.n_warm,
                      "hit_rate": hits / max(1, hits + misses), "hits": hits, "misses": misses,
                      "evictions": s1.evictions - s0.evictions, "h2d_gbs": h2d / wall / 1e9,
                      "h2d_bytes_per_step": h2d / K, "cold_start_misses": s0.misses},
        "roofline": {"kernel": "miss copies (pinned host to device slots)", "bound": "pcie",
                     "achieved": h2d / wall / 1e9, "peak": pcie, "unit": "GB/s", "frac": h2d / wall / 1e9 / pcie,
                     "peak_kind": "measured 2 GB pinned H2D copy on this box", "traffic": None},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": w.T * w.d * 2 + h2d / K,
                "d2h_bytes_per_step": w.T * w.d * 2},
        "cpu_baseline": cpu,
        "gpu_launches": launches[0],
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--host-gb", type=float, default=24.0, help="pinned host memory for expert images (tiered)")
    ap.add_argument("--slot-policy", choices=["lru", "freq"], default="lru",
                    help="tiered: replacement policy of the slot pool (LRU, or decayed use count)")
    ap.add_argument("--half-life-steps", type=float, default=50.0, help="tiered, freq: half-life of the use counts")
    ap.add_argument("--warm-profile", action="store_true",
                    help="tiered: fill the pool from a usage profile before the first step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        from synth.workloads import WORKLOADS
        w = WORKLOADS[args.workload]
        if w.layers > 1:
            import torch
            if not torch.cuda.is_available():
                raise SystemExit("bench.py needs a CUDA device")
            torch.cuda.set_device(local)
            (run_tiered if w.slots else run_stack)(args, ws, rank, local, w)
        else:
            run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
