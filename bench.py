"""Benchmark of one sparse MoE layer's forward pass on B300 (the decode workload by default).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload decode]

A layer pass is the whole hot path (router + top-k, bucketing, slot-table lookup inside the
expert FFN, SwiGLU experts, combine) over one batch of T tokens, replayed from a CUDA graph of
the C-ABI calls. Pass i runs the weights of layer i % 4 (decode) on batch i % 16, so each pass
reads its own experts (about 200 MB) and a layer's router and shared expert come back only
after about 600 MB of other reads: the inputs are larger than L2 and nothing is flushed. A
timed step is R consecutive passes, with R chosen so that the K timed steps last at least
300 ms (clock samples every 100 ms fall inside them). Times are CUDA events on the launching
stream, and the maximum is taken over ranks. One JSON line is printed by rank 0; with the
default decode workload it also carries the prefill chunk's measurement (T = 8192) under
"prefill".

--impl reference times the CPU oracle on this host's cores instead, over the same
workload and metric: one oracle pass per worker process and step, one worker per core.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

# the CPU oracle runs one numpy thread per process: fix the BLAS thread count before numpy loads
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; decode HBM GB/s & prefill int8 TOPS as % of B300 peak"
DTYPE = "bf16 activations, int8 block-32 weights (fp16 scales) entering f16 tensor-core MMAs exactly, fp32 accumulation"
N_BATCHES = 16
ROT_LAYERS = 4         # decode: layers whose weights rotate between passes
MIN_TIMED_MS = 300.0   # the K timed steps last at least this long
MAX_ORACLE_WORKERS = 32

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the dominant kernel, from one ncu
# capture of the kernel as it is now built (None once the kernel has changed since). Decode: the
# capture's bytes per expert record it streamed (41 records: 40 routed + the shared one, input
# batch 2), scaled in the line by the records of an average launch. Prefill: the two GEMM launches
# (gate/up + SwiGLU, down) of one pass at T = 8192.
TRAFFIC = {
    "decode": {"per_record": (206_294_528 + 3_836_672) / 41},
    "decode_q2": {"per_record": (60_700_928 + 694_272) / 41},
    "prefill": {"per_launch": 2_091_546_000 + 250_737_408 + 1_000_237_000 + 326_405_376},
}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0.0)) or None,
                "measured")
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


def pcts(v) -> dict:
    """Median and 10th / 90th percentiles of a list of per-pass times (ms)."""
    a = np.asarray(v, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)), "p90": float(np.percentile(a, 90)),
            "n": int(a.size)}


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
            self.path = f"/tmp/moe_bench_clocks_{os.getpid()}_{time.monotonic_ns()}.csv"
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)  # nvidia-smi takes a moment to start sampling
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
        sm, mx, power, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [c.strip() for c in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx = float(f[2])
                    power.append(float(f[3]))
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
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "sm_mhz_min": min(sm), "power_w_max": max(power) if power else None}


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


_BARRIER = None


def _oracle_pool_init(barrier):
    global _BARRIER
    _BARRIER = barrier


def _oracle_worker(job):
    """One worker of the all-core oracle timing: its own batch, its experts made here; W warm-up
    passes, a barrier, then `steps` timed passes (or until `budget_s`). One numpy thread."""
    from oracle import moe_oracle as O
    from synth.workloads import WORKLOADS
    wname, batch, warm, steps, budget_s = job
    w = WORKLOADS[wname]
    router = w.router(0)
    x = w.x_f64(batch)[:ORACLE_MAX_TOKENS]
    need = set(O.select_topk(O.router_logits(x, router), w.k).reshape(-1).tolist())
    ex = {e: w.expert(0, e) for e in sorted(need | {w.E + s for s in range(w.n_shared)})}
    shared = [ex[w.E + s] for s in range(w.n_shared)]
    _BARRIER.wait()
    for _ in range(warm):
        O.moe_layer(x, router, w.k, lambda e: ex[e], shared)
    _BARRIER.wait()
    n, t0 = 0, time.perf_counter()
    while True:
        O.moe_layer(x, router, w.k, lambda e: ex[e], shared)
        n += 1
        el = time.perf_counter() - t0
        if (steps is not None and n >= steps) or (budget_s is not None and el >= budget_s):
            break
    return x.shape[0] * n, n, el


def oracle_workers() -> tuple[int, int]:
    """(workers the all-core timing uses, logical CPUs this process may run on)."""
    try:
        avail = len(os.sched_getaffinity(0))
    except Exception:
        avail = os.cpu_count() or 1
    return max(1, min(avail, MAX_ORACLE_WORKERS)), avail


def time_oracle_all_cores(wname: str, warm: int = 1, steps: int | None = None, budget_s: float | None = None):
    """The oracle as it stands, one single-threaded process per core, all timing at once (spawn
    processes). Returns (tokens/s over all workers, passes, seconds, workers, cpus)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    n, avail = oracle_workers()
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(n)
    jobs = [(wname, i % N_BATCHES, warm, steps, budget_s) for i in range(n)]
    with cf.ProcessPoolExecutor(max_workers=n, mp_context=ctx, initializer=_oracle_pool_init,
                                initargs=(barrier,)) as ex:
        res = list(ex.map(_oracle_worker, jobs))
    tokens = sum(r[0] for r in res)
    passes = sum(r[1] for r in res)
    el = max(r[2] for r in res)
    return tokens / el, passes, el, n, avail


def cpu_baseline_line(w, args) -> dict:
    """The oracle timed on this host: all cores (one process per core, the headline value) and
    one core."""
    tps_all, passes, el, n, avail = time_oracle_all_cores(w.name, budget_s=args.cpu_seconds)
    tps1, steps1, el1, _ = time_oracle(w, prepare_oracle(w, list(range(4))), budget_s=args.cpu_seconds)
    lw = w.layers
    return {"value": tps_all / lw, "unit": "tokens/s", "cores": n, "kind": "oracle", "nproc": avail,
            "sample": f"{passes} oracle passes ({el:.1f} s) of T={min(w.T, ORACLE_MAX_TOKENS)} tokens, one process "
                      f"per core on {n} of {avail} logical CPUs, each on its own batch"
                      + (f" (layer 0; tokens/s divided by the {lw} layers of a step)" if lw > 1 else ""),
            "single_core": {"value": tps1 / lw, "cores": 1,
                            "sample": f"{steps1} oracle passes ({el1:.1f} s) over 4 rotating batches"}}


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
    # each step: one oracle pass per worker (one per core), all at once; stop early after 150 s
    tps, passes, el, n, avail = time_oracle_all_cores(w.name, warm=W, steps=K, budget_s=150.0)
    steps = max(1, passes // n)
    sample = (f"{passes} oracle layer passes ({el:.1f} s) of T={min(w.T, ORACLE_MAX_TOKENS)} tokens, one process "
              f"per core on {n} of {avail} logical CPUs, each on its own batch")
    if w.layers > 1:
        tps /= w.layers
        sample += f" (layer 0); tokens/s divided by the {w.layers} layers of a step"
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps,
        "warmup": W, "ms_per_step": 1e3 * el / steps * w.layers, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": w.describe(), "tokens_per_step": min(w.T, ORACLE_MAX_TOKENS) * n},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": n, "kind": "oracle", "sample": sample,
                         "nproc": avail},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ one-layer workloads ----

def time_layer(w, dev, K: int, W: int, rot_layers: int, n_batches: int, ydt: int, min_ms: float, ws: int,
               e2e: bool) -> dict:
    """Times layer passes of the one-layer workload w on `dev`: pass i runs layer i % rot_layers
    on batch i % n_batches from a CUDA graph of the C-ABI calls. Region 1: K steps of R passes
    each (R so that the region lasts >= min_ms), the clocks sampled meanwhile. Region 2: the same
    passes as three graphs (route + bucketing, expert FFN, combine) with events between, for the
    expert FFN's own time. With e2e, also the passes through the public API with host buffers."""
    import torch
    from routed_expert_ffn_bucketing_b300 import _lib as L
    from routed_expert_ffn_bucketing_b300 import layer as lay
    from synth.device import DeviceLayer

    dls = [DeviceLayer(w, layer=l, device=str(dev)) for l in range(rot_layers)]
    xs = [dls[0].x(b) for b in range(n_batches)]
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    buf = lay.alloc_buffers(s, device=dev, ydt=ydt, odt=L.MOE_BF16, keep_logits=False)
    tables = [L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of, dl.shared_ptr, fmt=w.fmt) for dl in dls]
    stream = torch.cuda.current_stream(dev)
    xdt = L.MOE_BF16
    n_combo = rot_layers * n_batches // math.gcd(rot_layers, n_batches)
    combo = [(i % rot_layers, i % n_batches) for i in range(n_combo)]

    def seg_route(l, x):
        L.moe_route_permute(s, x, xdt, dls[l].router, buf.topk_idx, buf.topk_w, None, buf.counts, buf.offsets,
                            buf.sorted_pair, buf.inv_pos, buf.active, buf.ws, buf.ws_bytes, None)

    def seg_layer(l, x):  # the whole pass in one C-ABI call
        L.moe_layer_forward(s, x, xdt, dls[l].router, tables[l], L.MOE_MODE_AUTO, buf.topk_idx, buf.topk_w, None,
                            buf.counts, buf.offsets, buf.sorted_pair, buf.inv_pos, buf.active, buf.y_perm, buf.ydt,
                            None, buf.out, buf.odt, buf.ws, buf.ws_bytes, None)

    def seg_ffn(l, x):
        L.moe_expert_ffn(s, L.MOE_MODE_AUTO, x, xdt, tables[l], buf.offsets, buf.sorted_pair, buf.active,
                         buf.y_perm, buf.ydt, buf.ws, buf.ws_bytes, None)

    def seg_comb(l, x):
        L.moe_combine(s, buf.y_perm, buf.ydt, buf.inv_pos, buf.topk_w, None, buf.out, buf.odt, None)

    # active experts per pass (for the algorithmic byte count), from untimed eager passes
    n_active = []
    for l, b in combo:
        seg_layer(l, xs[b])
        torch.cuda.synchronize(dev)
        n_active.append(int(buf.active[0].item()))
        assert L.moe_read_status(buf.ws) == 0
    cap = torch.cuda.Stream(dev)
    layer_graphs, stage_graphs = [], []
    for l, b in combo:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            seg_layer(l, xs[b])
        layer_graphs.append(g)
        gs = []
        for seg in (seg_route, seg_ffn, seg_comb):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                seg(l, xs[b])
            gs.append(g)
        stage_graphs.append(gs)
    for i in range(max(W, 3) * n_combo):
        layer_graphs[i % n_combo].replay()
    torch.cuda.synchronize(dev)
    # passes per step: the K steps together last >= min_ms
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(4 * n_combo):
        layer_graphs[i % n_combo].replay()
    b_.record(stream)
    torch.cuda.synchronize(dev)
    est = a.elapsed_time(b_) / (4 * n_combo)
    R = max(1, math.ceil(min_ms / (K * est)))

    # ---- region 1: K steps of R passes
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(dev.index or 0)
    barrier(ws)
    torch.cuda.synchronize(dev)
    clocks.start()
    t_wall = time.perf_counter()
    p = 0
    for i in range(K):
        ev[i][0].record(stream)
        for _ in range(R):
            layer_graphs[p % n_combo].replay()
            p += 1
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    assert L.moe_read_status(buf.ws) == 0, "a kernel reported an error during the timed steps"
    step_ms = [x.elapsed_time(y) for x, y in ev]
    total_s = dist_max(sum(step_ms) / 1e3, ws, dev)

    # ---- region 2: stages, for the expert FFN's own time
    n2 = min(K * R, max(8 * n_combo, 256))
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n2)]
    torch.cuda.synchronize(dev)
    for i in range(n2):
        e = ev2[i]
        g_route, g_ffn, g_comb = stage_graphs[i % n_combo]
        e[0].record(stream)
        g_route.replay()
        e[1].record(stream)
        g_ffn.replay()
        e[2].record(stream)
        g_comb.replay()
        e[3].record(stream)
    torch.cuda.synchronize(dev)
    route_ms = [e[0].elapsed_time(e[1]) for e in ev2]
    ffn_ms = [e[1].elapsed_time(e[2]) for e in ev2]
    comb_ms = [e[2].elapsed_time(e[3]) for e in ev2]
    staged_ms = [e[0].elapsed_time(e[3]) for e in ev2]

    # ---- region 3 (decode shapes): the expert FFN kernel back to back, one launch per (layer,
    # batch) on that combination's routing (computed beforehand), all in one graph: the kernel's
    # own duration, without a graph launch around each launch. Consecutive launches read
    # different layers' records (about 200 MB each, L2 126 MB), so none finds its experts in L2
    b2b_ms = None
    if w.T <= 16:
        rbufs = []
        for l, b in combo:
            rb = lay.alloc_buffers(s, device=dev, ydt=ydt, odt=L.MOE_BF16, keep_logits=False)
            L.moe_route_permute(s, xs[b], xdt, dls[l].router, rb.topk_idx, rb.topk_w, None, rb.counts, rb.offsets,
                                rb.sorted_pair, rb.inv_pos, rb.active, rb.ws, rb.ws_bytes, None)
            rbufs.append(rb)
        torch.cuda.synchronize(dev)
        g3 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g3, stream=cap):
            for c, (l, b) in enumerate(combo):
                L.moe_expert_ffn(s, L.MOE_MODE_AUTO, xs[b], xdt, tables[l], rbufs[c].offsets, rbufs[c].sorted_pair,
                                 rbufs[c].active, buf.y_perm, buf.ydt, buf.ws, buf.ws_bytes, None)
        for _ in range(2):
            g3.replay()
        torch.cuda.synchronize(dev)
        n3 = max(4, n2 // n_combo)
        a3, b3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a3.record(stream)
        for _ in range(n3):
            g3.replay()
        b3.record(stream)
        torch.cuda.synchronize(dev)
        assert L.moe_read_status(buf.ws) == 0, "a kernel reported an error during the back-to-back launches"
        b2b_ms = a3.elapsed_time(b3) / (n3 * n_combo)
        del g3, rbufs

    res = {"R": R, "K": K, "step_ms": step_ms, "total_s": total_s, "wall": wall, "clocks": clk,
           "pass_ms": [t / R for t in step_ms], "n_active": [n_active[i % n_combo] for i in range(n2)],
           "n_active_mean": float(np.mean(n_active)), "route_ms": route_ms, "ffn_ms": ffn_ms, "comb_ms": comb_ms,
           "staged_ms": staged_ms, "n_combo": n_combo, "ffn_b2b_ms": b2b_ms}

    if e2e:
        # the same passes through the public API with host buffers, per pass: the pinned x copied
        # in, the C-ABI calls on the device copy and the bf16 output copied back, all three captured
        # in one CUDA graph per (layer, batch), then the stream waited for
        x_host = [x.cpu().pin_memory() for x in xs]
        out_host = torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory()
        x_dev = torch.empty_like(xs[0])
        e2e_graphs = []
        for l, b in combo:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                x_dev.copy_(x_host[b], non_blocking=True)
                seg_layer(l, x_dev)
                out_host.copy_(buf.out, non_blocking=True)
            e2e_graphs.append(g)
        n_e2e = min(K * R, 4000)
        e2e_s = 0.0
        for i in range(W + n_e2e):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            e2e_graphs[i % n_combo].replay()
            stream.synchronize()
            if i >= W:
                e2e_s += time.perf_counter() - t0
        res["e2e_s"] = dist_max(e2e_s, ws, dev)
        res["n_e2e"] = n_e2e
    del layer_graphs, stage_graphs
    return res


def run_ours(args, ws, rank, local):
    import torch
    from routed_expert_ffn_bucketing_b300 import _lib as L
    from synth.workloads import WORKLOADS

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    K, W = args.steps, args.warmup
    hbm_peak, bf16_peak, bf16_sus, peak_kind = peaks()
    prefill = w.T > 16
    r = time_layer(w, dev, K, W, rot_layers=1 if prefill else ROT_LAYERS, n_batches=4 if prefill else N_BATCHES,
                   ydt=L.MOE_BF16 if prefill else L.MOE_F32, min_ms=MIN_TIMED_MS, ws=ws, e2e=True)
    R = r["R"]
    value = ws * w.T * K * R / r["total_s"]
    line_roof, extra = layer_roofline(w, r, hbm_peak, bf16_peak, bf16_sus, peak_kind)
    e2e = {"value": ws * w.T * r["n_e2e"] / r["e2e_s"], "unit": "tokens/s", "h2d_bytes_per_step": w.T * w.d * 2,
           "d2h_bytes_per_step": w.T * w.d * 2, "passes": r["n_e2e"],
           "launch": "per pass: one CUDA graph of the pinned x copy in, the C-ABI call and the bf16 output copy "
                     "out, then the stream synchronised"}
    nested = None
    if not prefill and not args.no_prefill and args.workload == "decode":
        torch.cuda.empty_cache()
        wp = WORKLOADS["prefill"]
        rp = time_layer(wp, dev, 10, 3, rot_layers=1, n_batches=4, ydt=L.MOE_BF16, min_ms=MIN_TIMED_MS, ws=ws,
                        e2e=False)
        roof_p, extra_p = layer_roofline(wp, rp, hbm_peak, bf16_peak, bf16_sus, peak_kind)
        nested = {"workload": wp.describe(), "value": ws * wp.T * 10 * rp["R"] / rp["total_s"], "unit": "tokens/s",
                  "steps": 10, "passes_per_step": rp["R"], "ms_per_pass": pcts(rp["pass_ms"]),
                  "roofline": roof_p, **extra_p, "clocks": rp["clocks"],
                  "gpu_launches": 12 * 10 * rp["R"]}
    nested_q2 = None
    if not prefill and not args.no_q2 and args.workload == "decode":
        # the same decode pass on 2-bit expert records (2.5 bits per weight)
        torch.cuda.empty_cache()
        wq = WORKLOADS["decode_q2"]
        rq = time_layer(wq, dev, K, W, rot_layers=ROT_LAYERS, n_batches=N_BATCHES, ydt=L.MOE_F32,
                        min_ms=MIN_TIMED_MS, ws=ws, e2e=False)
        roof_q, extra_q = layer_roofline(wq, rq, hbm_peak, bf16_peak, bf16_sus, peak_kind)
        nested_q2 = {"workload": wq.describe(), "value": ws * wq.T * K * rq["R"] / rq["total_s"], "unit": "tokens/s",
                     "record_bytes": wq.record_bytes, "steps": K, "passes_per_step": rq["R"],
                     "ms_per_pass": pcts(rq["pass_ms"]), "roofline": roof_q, **extra_q, "clocks": rq["clocks"],
                     "gpu_launches": 4 * K * rq["R"]}
    nested_more = {}
    if not prefill and not args.no_stack and args.workload == "decode":
        # the 48-layer stack and the tiered slot pool, short runs, each line's own fields kept
        import copy
        keep = ("workload", "value", "unit", "steps", "warmup", "ms_per_step", "roofline", "e2e", "slot_pool",
                "gpu_launches", "clocks")
        runs = [("stack", "stack", dict(steps=10, warmup=3)),
                ("tiered", "tiered", dict(steps=40, warmup=5, host_gb=8.0)),
                ("tiered_count_warm_split", "tiered",
                 dict(steps=40, warmup=5, host_gb=8.0, slot_policy="freq", warm_profile=True, pcie_frac=0.6,
                      host_threads=8)),
                ("tiered_q2", "tiered_q2", dict(steps=40, warmup=5, host_gb=8.0))]
        for key, wname, over in runs:
            torch.cuda.empty_cache()
            sub_args = copy.copy(args)
            sub_args.no_cpu_baseline = True
            for k_, v_ in over.items():
                setattr(sub_args, k_, v_)
            wn = WORKLOADS[wname]
            ln = (run_tiered if wn.slots else run_stack)(sub_args, ws, rank, local, wn, nested=True)
            if ln is not None:
                cfg = ln["config"]
                nested_more[key] = {"workload": cfg["workload"], **{k_: ln[k_] for k_ in keep[1:] if k_ in ln}}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_line(w, args)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": sum(r["step_ms"]) / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE, "data": "synthetic (seeded)",
        "config": {"workload": w.describe(), "tokens_per_pass": w.T, "passes_per_step": R,
                   "tokens_per_step": w.T * R, "weights": "int8 block-32 + fp16 scales", "activations": "bf16",
                   "l2": ("inputs larger than L2: pass i runs layer i % 4's weights (4 x 2.57 GB resident) on batch "
                          "i % 16, about 200 MB of experts per pass; no flush" if not prefill else
                          "inputs larger than L2: each pass reads all 513 experts (2.57 GB); no flush"),
                   "layers_rotated": 1 if prefill else ROT_LAYERS, "batches": 4 if prefill else N_BATCHES,
                   "mean_active_experts": r["n_active_mean"],
                   "launch": "one CUDA graph of the one C-ABI call of a pass, moe_layer_forward (stages_ms: "
                             "moe_route_permute, moe_expert_ffn, moe_combine, one graph per stage, events between)",
                   "parallelism": f"replicas x{ws}"},
        "ms_per_pass": pcts(r["pass_ms"]),
        "roofline": line_roof,
        **extra,
        "wall_s": r["wall"],
        "e2e": e2e,
        "cpu_baseline": cpu,
        # kernels per pass: decode 4 (router GEMV, top-k with bucketing, persistent expert FFN,
        # combine); prefill 12 (router weight split, router GEMM, top-k, 3 bucketing, 5 expert
        # FFN, combine)
        "gpu_launches": (12 if prefill else 4) * K * R,
        "clocks": r["clocks"],
    }
    if nested is not None:
        line["prefill"] = nested
    if nested_q2 is not None:
        line["decode_q2"] = nested_q2
    line.update(nested_more)
    print(json.dumps(line), flush=True)


def layer_roofline(w, r, hbm_peak, bf16_peak, bf16_sus, peak_kind):
    """The expert FFN's roofline entry for a one-layer workload, from time_layer's region 2."""
    ffn_ms = r["ffn_ms"]
    n = len(ffn_ms)
    rows = w.P + w.T * w.n_shared
    stages = {"route_permute": pcts(r["route_ms"]), "expert_ffn": pcts(ffn_ms), "combine": pcts(r["comb_ms"]),
              "pass_as_three_graphs": pcts(r["staged_ms"])}
    if w.T > 16:
        # tensor-bound: algorithmic FLOPs of the expert FFN (gate, up and down over every row)
        flops = 2.0 * rows * 3 * w.d * w.f
        tflops = flops / (sum(ffn_ms) / 1e3 / n) / 1e12
        router_flops = 2.0 * w.T * w.d * w.E
        roof = {"kernel": "moe_expert_ffn (tcgen05 grouped GEMM: gate/up + SwiGLU, down)", "bound": "tensor",
                "achieved": tflops, "peak": bf16_peak, "unit": "TFLOP/s", "frac": tflops / bf16_peak,
                "peak_kind": f"{peak_kind} dense bf16 burst (f16 has the same dense rate)",
                "frac_of_sustained": tflops / bf16_sus if bf16_sus else None,
                "int8_peak": None,
                "int8_note": "tcgen05.mma kind::i8 does not exist for sm_103a (ptxas: Feature '.kind::i8' not "
                             "supported on .target 'sm_103a'); the int8 codes enter f16 MMAs exactly",
                "traffic": (TRAFFIC["prefill"] or {}).get("per_launch"),
                "traffic_kernels": "prefill_gemm_kernel<0> + <1> (ncu, one pass)",
                "flops_per_launch": flops, "ms_per_launch": sum(ffn_ms) / n}
        extra = {"stages_ms": stages,
                 "router": {"ms": pcts(r["route_ms"])["median"], "flops": router_flops,
                            "tflops": router_flops / (np.median(r["route_ms"]) / 1e3) / 1e12,
                            "note": "route_permute stage: router GEMM + top-k + bucketing"}}
    else:
        small = w.T * w.d * 2 + rows * w.d * 4
        byts = [(na + w.n_shared) * w.record_bytes + small for na in r["n_active"]]
        # the kernel's launch duration: from the back-to-back launches when measured, else from
        # the stage graphs (which add a graph launch to every launch)
        per_launch_ms = r["ffn_b2b_ms"] if r.get("ffn_b2b_ms") else sum(ffn_ms) / n
        achieved = float(np.mean(byts)) / (per_launch_ms / 1e3) / 1e9
        roof = {"kernel": "moe_expert_ffn (persistent kernel: gate/up + SwiGLU, down)", "bound": "hbm",
                "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                "peak_kind": f"{peak_kind} copy bandwidth", "frac_of_8tbs": achieved / 8000.0,
                "traffic": (TRAFFIC.get(w.name) or {}).get("per_record", 0.0) * float(np.mean(r["n_active"]) + w.n_shared)
                if TRAFFIC.get(w.name) else None,
                "bytes_per_launch": float(np.mean(byts)),
                "ms_per_launch": per_launch_ms,
                "timing": "CUDA events around one graph of the kernel launched back to back on each (layer, "
                          "batch)'s routing, replayed; per launch = total / launches"
                if r.get("ffn_b2b_ms") else "CUDA events around a graph of the one launch",
                "ms_per_launch_stage_graph": sum(ffn_ms) / n}
        router_bytes = w.d * w.E * 4
        step_bytes = [(na + w.n_shared) * w.record_bytes + small + router_bytes for na in r["n_active"]]
        extra = {"stages_ms": stages,
                 "pass_hbm_gbs": float(np.mean(step_bytes)) / (np.mean(r["pass_ms"]) / 1e3) / 1e9}
    return roof, extra


# ------------------------------------------------------------------ multi-layer workloads ---

def stack_cpu_baseline(w, rank, args):
    """The oracle on one layer (layer 0's router and experts) at T tokens, extrapolated to the
    L-layer step by dividing its tokens/s by L."""
    if rank != 0 or args.no_cpu_baseline:
        return None
    return cpu_baseline_line(w, args)


def run_stack(args, ws, rank, local, w, nested: bool = False):
    """L resident layers on a residual stream; one CUDA graph of the whole L-layer step."""
    import torch
    from routed_expert_ffn_bucketing_b300 import _lib as L
    from routed_expert_ffn_bucketing_b300.stack import DecodeStack, LayerWeights
    from synth.device import DeviceLayer

    dev = torch.device("cuda", local)
    K, W = args.steps, args.warmup
    hbm_peak, _, _, peak_kind = peaks()
    need = w.layers * (w.E + w.n_shared) * w.record_bytes
    free, _ = torch.cuda.mem_get_info(dev)
    if need > free - (4 << 30):
        raise SystemExit(f"stack workload needs {need / 1e9:.1f} GB of device memory, {free / 1e9:.1f} GB free")
    dls = [DeviceLayer(w, layer=l, device=str(dev)) for l in range(w.layers)]
    s = L.shape(w.T, w.d, w.f, w.E, w.k, w.n_shared)
    st = DecodeStack(s, [LayerWeights(dl.router, L.expert_table(dl.pool, dl.slot_bytes, dl.n_slots, dl.slot_of,
                                                                dl.shared_ptr)) for dl in dls], device=dev,
                     native=not args.python_loop)
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

    # end to end: per step one CUDA graph of the pinned x copy in, the stack's calls and the bf16
    # output copy out, then the stream waited for
    x_host = [x.cpu().pin_memory() for x in xs]
    out_host = torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(xs[0])
    e2e_graphs = []
    for b in range(n_batches):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            x_dev.copy_(x_host[b], non_blocking=True)
            st.forward(x_dev)
            out_host.copy_(st.resid, non_blocking=True)
        e2e_graphs.append(g)
    K_e2e = min(K, 50)
    e2e_s = 0.0
    for i in range(W + K_e2e):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e2e_graphs[i % n_batches].replay()
        stream.synchronize()
        if i >= W:
            e2e_s += time.perf_counter() - t0
    e2e_s = dist_max(e2e_s, ws, dev)
    cpu = stack_cpu_baseline(w, rank, args)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": sum(step_ms) / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE, "data": "synthetic (seeded)",
        "config": {"workload": w.describe(), "tokens_per_step": w.T, "weights": "int8 block-32 + fp16 scales",
                   "resident_gb": need / 1e9, "activations": "bf16 residual stream",
                   "l2": "inputs larger than L2 (each step reads every layer's selected experts, ~10 GB)",
                   "batches": n_batches, "mean_active_experts_per_layer": float(np.mean(n_active)),
                   "launch": ("one CUDA graph of one moe_stack_forward call: per layer norm, router GEMV, top-k "
                              "with bucketing, expert FFN, combine, all in one chain of programmatic dependents"
                              if st.native else
                              f"one CUDA graph of the {2 * w.layers} C-ABI calls of a step (per layer: moe_rms_norm, "
                              "then moe_layer_forward: route, bucketing, expert FFN, combine)"),
                   "block": "pre-norm residual: x + MoE(rms_norm(x)), eps 1e-6, no gain",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"kernel": f"whole {w.layers}-layer step (route, permute, expert FFN, combine per layer)",
                     "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_kind": f"{peak_kind} copy bandwidth", "traffic": None,
                     "bytes_per_step": float(np.mean(step_bytes)), "ms_per_step": sum(step_ms) / K},
        "e2e": {"value": ws * w.T * K_e2e / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": w.T * w.d * 2,
                "d2h_bytes_per_step": w.T * w.d * 2, "steps": K_e2e,
                "launch": "per step: one CUDA graph of the pinned x copy in, the stack's C-ABI calls and the bf16 "
                          "output copy out, then the stream synchronised"},
        "cpu_baseline": cpu,
        "gpu_launches": 5 * w.layers * K,  # per layer: norm, router GEMV, top-k with bucketing, expert FFN, combine
        "clocks": clk,
    }
    if nested:
        return line
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
        fill_expert_records(w.seed, l, e, n, w.d, w.f, tmp.data_ptr(), rb, w.expert_sigma, fmt=w.fmt)
        host[i:i + n].copy_(tmp[:n])
        i += n
    torch.cuda.synchronize(dev)
    return host


def run_tiered(args, ws, rank, local, w, nested: bool = False):
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
            fill_expert_records(w.seed, l, w.E, w.n_shared, w.d, w.f, t.data_ptr(), rb, w.expert_sigma, fmt=w.fmt)
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
    # the library's executor runs the step (moe_tiered_forward); early routing needs the Python loop
    native = not args.prefetch and not args.python_loop
    ts = TieredStack(s, w.layers, routers, h_records, w.slots, rb, shared, device=dev, policy=policy,
                     half_life_steps=args.half_life_steps, profile=profile, fmt=w.fmt, native=native)
    if args.host_threads:
        ts.host_threads = args.host_threads
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
    host_experts = [0]

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
            y = ts.forward(x_dev, prefetch=args.prefetch, prefetch_top=args.prefetch_top, pcie_frac=args.pcie_frac)
            host_experts[0] += sum(ts.layer_host)
            if e2e:
                out_host.copy_(y, non_blocking=True)
            torch.cuda.synchronize(dev)
            wall += time.perf_counter() - t0
            # per layer: norm, router GEMV, top-k with bucketing, expert FFN, combine; with misses one
            # more expert FFN (the missed experts after their copies)
            launches[0] += sum(5 + (m > 0) for m in ts.layer_misses)
            if args.prefetch:  # the next layer's router GEMV and top-k with bucketing
                launches[0] += 2 * (w.layers - 1)
        return wall

    try:
        run(0, W, False)
        launches[0] = 0
        host_experts[0] = 0
        ts.host_seconds = 0.0
        s0 = L.slot_table_stats(ts.table)
        pf0 = L.slot_table_prefetch_stats(ts.table)
        clocks = ClockSampler(local)
        barrier(ws)
        clocks.start()
        wall = run(W, K, True)
        barrier(ws)
        clk = clocks.stop()
        s1 = L.slot_table_stats(ts.table)
        pf1 = L.slot_table_prefetch_stats(ts.table)
        st_words = (L.moe_read_status(ts.buf.ws), L.moe_read_status(ts.ws_miss), L.moe_read_status(ts.pbuf.ws))
        assert not any(st_words), f"a kernel reported an error during the timed steps: {st_words}"
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
        "dtype": DTYPE, "data": "synthetic (seeded)",
        "config": {"workload": w.describe() + f", {w.slots} device slots, drift every {synth.DRIFT_EVERY} steps",
                   "tokens_per_step": w.T,
                   "weights": "int8 block-32 + fp16 scales" if w.fmt == 0 else
                              "2-bit block-32 codes + fp16 scales (2.5 bits per weight)",
                   "record_bytes": rb, "pool_gb": w.slots * rb / 1e9, "host_images": n_img,
                   "host_mapping": "(l*E + e) mod host_images" if n_img < n_all else "one image per expert",
                   "timing": "wall clock per step (the host reads each layer's active list), x copied in and "
                             "the output copied out inside every step",
                   "executor": "moe_tiered_forward (C++)" if native else "TieredStack Python loop",
                   "parallelism": f"replicas x{ws}"},
        "slot_pool": {"policy": "LRU" if policy == L.MOE_SLOT_LRU else
                      f"decayed use count (half-life {args.half_life_steps:g} steps)",
                      "warm_profile": bool(args.warm_profile), "warm_loads": ts.n_warm,
                      "hit_rate": hits / max(1, hits + misses), "hits": hits, "misses": misses,
                      "evictions": s1.evictions - s0.evictions, "h2d_gbs": h2d / wall / 1e9,
                      "h2d_bytes_per_step": h2d / K, "cold_start_misses": s0.misses,
                      "pcie_frac": args.pcie_frac, "host_computed_experts": host_experts[0],
                      "host_threads": ts.host_threads,
                      "host_ffn_ms_per_step": 1e3 * ts.host_seconds / K,
                      "early_routing_prefetch": bool(args.prefetch), "prefetch_top": args.prefetch_top,
                      "prefetch_loads": pf1[0] - pf0[0],
                      "prefetch_used": pf1[1] - pf0[1]},
        "roofline": {"kernel": "miss copies (pinned host to device slots)", "bound": "pcie",
                     "achieved": h2d / wall / 1e9, "peak": pcie, "unit": "GB/s", "frac": h2d / wall / 1e9 / pcie,
                     "peak_kind": "measured 2 GB pinned H2D copy on this box", "traffic": None},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": w.T * w.d * 2 + h2d / K,
                "d2h_bytes_per_step": w.T * w.d * 2},
        "cpu_baseline": cpu,
        "gpu_launches": launches[0],
        "clocks": clk,
    }
    if nested:
        return line
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="decode: skip the nested prefill measurement")
    ap.add_argument("--no-q2", action="store_true", help="decode: skip the nested 2-bit-format measurement")
    ap.add_argument("--no-stack", action="store_true",
                    help="decode: skip the nested 48-layer stack and tiered slot-pool measurements")
    ap.add_argument("--host-gb", type=float, default=24.0, help="pinned host memory for expert images (tiered)")
    ap.add_argument("--slot-policy", choices=["lru", "freq"], default="lru",
                    help="tiered: replacement policy of the slot pool (LRU, or decayed use count)")
    ap.add_argument("--half-life-steps", type=float, default=50.0, help="tiered, freq: half-life of the use counts")
    ap.add_argument("--warm-profile", action="store_true",
                    help="tiered: fill the pool from a usage profile before the first step")
    ap.add_argument("--prefetch", action="store_true",
                    help="tiered: route layer l+1 on layer l's input and copy its experts during layer l")
    ap.add_argument("--pcie-frac", type=float, default=1.0,
                    help="tiered: share of each layer's missed experts copied to the device; the host computes the rest")
    ap.add_argument("--host-threads", type=int, default=0,
                    help="tiered, pcie-frac < 1: threads of the host expert FFN (0: three quarters of the cores)")
    ap.add_argument("--python-loop", action="store_true",
                    help="stack / tiered: run the step as per-layer calls (stack) or with TieredStack's Python loop "
                         "(tiered) instead of the library's executor")
    ap.add_argument("--prefetch-top", type=int, default=None,
                    help="tiered, prefetch: load only each token's first N predicted experts")
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
