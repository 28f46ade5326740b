"""Benchmark of the NVFP4 + LoRA + AQN-RMSNorm linear on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step is one pass of the decode hot path over one batch of synthetic input:
the 7B-shaped 3584x3584 projection (NVFP4 weights, LoRA r=32, lambda=2, AQN
sigma=1e-2, 0.1% outliers x20) at every batch size of its sweep M in
{1, 8, 16, 32, 64}, each call RMSNorm-AQN prologue + NVFP4 main loop + LoRA
epilogue.  Weights rotate through enough distinct copies (> 2x L2) that every
call streams its weights from HBM.  The metric is HBM GB/s of algorithmic bytes
(9P/16 + 4 + 2r(d_i+d_o) + 2M(d_i+d_o) + 8 d_i per call).

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step); the line reports bytes of all ranks over the
slowest rank's time.

--impl reference times the plain CPU oracle on the host cores on a bounded
sample of the same workload (test infrastructure, used only for this leg and
the cpu_baseline object).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NVFP4+LoRA linear: HBM GB/s (% of ~8 TB/s) at M<=64; TFLOPS at M=4096"


def algorithmic_bytes(M, d_i, d_o, r):
    P = d_o * d_i
    return 9 * P // 16 + 4 + 2 * r * (d_i + d_o) + 2 * M * (d_i + d_o) + 8 * d_i


def algorithmic_flops(M, d_i, d_o, r):
    return 2 * M * d_o * d_i + 2 * M * r * (d_i + d_o)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def profile_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or None when
    there is none or the kernel's source has changed since the counters were taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(f"{kernel}@{workload}")
        if e is None:
            return None
        with open(os.path.join(ROOT, e["src"]), "rb") as f:
            if hashlib.sha1(f.read()).hexdigest() != e["src_sha1"]:
                return None
        return e.get("dram_bytes_per_launch")
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.file is None:
            return None
        try:
            rows = [l.strip().split(",") for l in open(self.file.name) if l.strip()]
            os.unlink(self.file.name)
        except Exception:
            return None
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except Exception:
                continue
            for name, v in zip(names[1:], r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        # NCCL between GPUs; gloo on a host without one (the reference arm's other ranks
        # and the multi-rank tests on CPU)
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float, device):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import torch

    from precision_linear_gb300 import binding as pl
    from precision_linear_gb300 import synthetic

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = synthetic.WORKLOADS[args.workload]
    p = wl.projs[0]
    d_i, d_o, r = p.d_i, p.d_o, wl.r
    Ms = list(wl.Ms)
    # distinct weight copies so that every call reads its weights from HBM
    L2 = 129 * 2 ** 20
    per_copy = 9 * d_i * d_o // 16
    n_sets = max(2, (4 * L2) // (per_copy * len(Ms)) + 1)
    sets = []
    base = synthetic.projection_case(d_o, d_i, max(Ms), r, wl.sigma, wl.seed, wl.outlier_frac, device="cpu")
    W_dev = base["W"].to(dev)
    codes0, scales0, sg0 = pl.nvfp4_quantize(W_dev)
    torch.cuda.synchronize()
    # each step's inputs and results sit in one device buffer apiece (views per call), so the
    # end-to-end leg moves a step's inputs and results with one copy each way
    x_off = [sum(Ms[:j]) for j in range(len(Ms))]
    x_bufs, y_bufs = [], []
    for i in range(n_sets):
        xb = torch.empty(sum(Ms), d_i, dtype=torch.bfloat16, device=dev)
        yb = torch.empty(sum(Ms), d_o, dtype=torch.bfloat16, device=dev)
        x_bufs.append(xb)
        y_bufs.append(yb)
        calls = []
        for j, M in enumerate(Ms):
            xv = xb[x_off[j]:x_off[j] + M]
            xv.copy_(base["x"][:M])
            calls.append(dict(M=M, codes=codes0.clone(), scales=scales0.clone(), s_g=sg0.clone(),
                              x=xv, A=base["A"].to(dev), B=base["B"].to(dev),
                              w_norm=base["w_norm"].to(dev), z=base["z"].to(dev),
                              y=yb[x_off[j]:x_off[j] + M]))
        sets.append(calls)
    ws = pl.Workspace(dev)
    ws.get(max(pl.workspace_bytes(M, d_i, d_o, r) for M in Ms))

    def one_call(c, stream_x=None):
        pl.nvfp4_lora_linear(c["x"], c["codes"], c["scales"], c["s_g"], c["A"], c["B"], wl.lam, c["w_norm"],
                             c["z"], synthetic.EPS, out=c["y"], workspace=ws)

    def batch_call(calls):
        """The step's calls as one batch of independent problems (one prologue + one main kernel)."""
        pl.nvfp4_lora_linear_batch([dict(x=c["x"], codes=c["codes"], scales=c["scales"], s_g=c["s_g"], A=c["A"],
                                         B=c["B"], lam=wl.lam, w_norm=c["w_norm"], z=c["z"]) for c in calls],
                                   synthetic.EPS, outs=[c["y"] for c in calls], workspace=ws)

    def step(k, form):
        if form == "batch":
            batch_call(sets[k])
        else:
            for c in sets[k]:
                one_call(c)

    # CUDA graphs per form: one per copy set (= one step), and one "round" graph holding a
    # step on every copy set, so that the GPU runs far ahead of the host
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)  # every launch, replay and event below is on this stream
    n_round = len(sets)
    forms = {}
    with torch.cuda.stream(stream):
        for form in ("separate", "batch"):
            for k in range(n_round):  # warm (tensor-map encode, attribute set-up, workspace size) outside capture
                step(k, form)
        torch.cuda.synchronize()
        for form in ("separate", "batch"):
            graphs = []
            for k in range(n_round):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    step(k, form)
                graphs.append(g)
            round_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(round_graph, stream=stream):
                for k in range(n_round):
                    step(k, form)
            forms[form] = (graphs, round_graph)
    torch.cuda.synchronize()

    def run_steps(k, form):
        """Exactly k steps of one form: whole rounds, then single-step graphs for the rest."""
        graphs, round_graph = forms[form]
        for _ in range(k // n_round):
            round_graph.replay()
        for i in range(k % n_round):
            graphs[i].replay()

    paths = {M: pl.linear_path(M, d_i, d_o, r) for M in Ms}
    launches = {"separate": sum(1 if paths[M] == 2 else 2 for M in Ms),  # fused kernel, or prologue + main
                "batch": 2}
    step_bytes = sum(algorithmic_bytes(M, d_i, d_o, r) for M in Ms)
    step_flops = sum(algorithmic_flops(M, d_i, d_o, r) for M in Ms)

    # the faster form is the headline; the other is reported beside it
    form_ms = {}
    for form in forms:
        run_steps(args.warmup, form)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_steps(4 * n_round, form)
        e1.record(stream)
        torch.cuda.synchronize()
        form_ms[form] = e0.elapsed_time(e1) / (4 * n_round)
    form = min(form_ms, key=form_ms.get)
    run_steps(args.warmup, form)
    torch.cuda.synchronize()

    # ---- timed region: K steps (clocks sampled from a 1 s soak just before it through its end)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < 1.0:
            run_steps(20 * n_round, form)
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        run_steps(args.steps, form)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(world, ms, dev)
    clocks = clk.summary()
    total_bytes = step_bytes * args.steps * world
    value = total_bytes / (ms * 1e-3) / 1e9
    forms_out = {f: {"ms_per_step": round(v, 5), "GBps": round(step_bytes / (v * 1e-3) / 1e9, 1),
                     "tokens_per_s": round(sum(Ms) / (v * 1e-3), 1), "gpu_launches_per_step": launches[f]}
                 for f, v in form_ms.items()}

    # ---- per-M call durations (the roofline of the dominant kernel)
    per_m = {}
    reps = 20
    for j, M in enumerate(Ms):
        g = torch.cuda.CUDAGraph()  # this M on every copy set, back to back
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for k in range(len(sets)):
                    one_call(sets[k][j])
        torch.cuda.synchronize()
        for k in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * len(sets))
        b = algorithmic_bytes(M, d_i, d_o, r)
        per_m[str(M)] = {"us_per_call": round(us, 3), "GBps": round(b / (us * 1e-6) / 1e9, 1),
                         "TFLOPs": round(algorithmic_flops(M, d_i, d_o, r) / (us * 1e-6) / 1e12, 2),
                         "tokens_per_s_per_projection": round(M / (us * 1e-6), 1)}
    dom = max(per_m, key=lambda k: per_m[k]["us_per_call"])
    hbm_peak, _, peak_kind = measured_peaks()
    # the dominant kernel over the timed region: separate calls -- the decode kernel of every
    # call, algorithmic bytes per launch (the sweep's mean) over its mean launch duration;
    # batch -- the main kernel of the batch (every call's weight tiles), the step's bytes over
    # the step's time (the prologue's time included); both from CUDA events on the launching
    # stream around the K steps, i.e. the step's GB/s
    if form == "batch":
        kern, per_launch, n_launch = "k_tc_decode (+ k_pro_rows)", step_bytes, 1
        traffic = profile_traffic("k_tc_decode", f"{args.workload}/batch")
    else:
        kern = "k_fused_decode" if all(v == 2 for v in paths.values()) else "decode kernels"
        per_launch, n_launch = round(step_bytes / len(Ms)), len(Ms)
        traffic_m = [profile_traffic(kern, f"{args.workload}/M{M}") for M in Ms]
        traffic = round(sum(traffic_m) / len(Ms)) if all(t is not None for t in traffic_m) else None
    roofline = {"bound": "hbm", "kernel": kern, "form": form, "bytes_per_launch": per_launch,
                "launch_us": round(ms * 1e3 / (args.steps * n_launch), 3),
                "achieved": round(value / world, 2), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(value / world / hbm_peak, 4), "peak_kind": peak_kind, "traffic": traffic,
                "slowest_single_call": {"M": int(dom), "GBps": per_m[dom]["GBps"],
                                        "frac": round(per_m[dom]["GBps"] / hbm_peak, 4)}}

    # ---- end to end through the public API with host buffers
    e2e = None
    if rank == 0 or world > 1:
        hx = torch.empty(sum(Ms), d_i, dtype=torch.bfloat16).pin_memory()  # a step's inputs, packed
        hy = torch.empty(sum(Ms), d_o, dtype=torch.bfloat16).pin_memory()  # a step's results, packed
        for j, M in enumerate(Ms):
            hx[x_off[j]:x_off[j] + M].copy_(base["x"][:M])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        bi = sum(2 * M * d_i for M in Ms)
        bo = sum(2 * M * d_o for M in Ms)

        def e2e_step(k):
            x_bufs[k].copy_(hx, non_blocking=True)  # H2D of the step's inputs
            step(k, form)
            hy.copy_(y_bufs[k], non_blocking=True)  # D2H of the step's results

        copy_stream = torch.cuda.Stream(dev)

        def e2e_round():
            """Every copy set once, the next step's H2D and this step's D2H on a copy stream,
            overlapping the calls: the H2D of step k + 1 runs under the calls of step k."""
            n = len(sets)
            fork = torch.cuda.Event()
            fork.record(stream)
            copy_stream.wait_event(fork)
            h2d = [torch.cuda.Event() for _ in range(n)]
            done = [torch.cuda.Event() for _ in range(n)]
            with torch.cuda.stream(copy_stream):
                x_bufs[0].copy_(hx, non_blocking=True)
                h2d[0].record(copy_stream)
            for k in range(n):
                stream.wait_event(h2d[k])
                step(k, form)
                done[k].record(stream)
                with torch.cuda.stream(copy_stream):
                    if k + 1 < n:
                        x_bufs[k + 1].copy_(hx, non_blocking=True)
                        h2d[k + 1].record(copy_stream)
                    copy_stream.wait_event(done[k])
                    hy.copy_(y_bufs[k], non_blocking=True)
            join = torch.cuda.Event()
            join.record(copy_stream)
            stream.wait_event(join)

        with torch.cuda.stream(stream):
            eg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(eg, stream=stream):
                e2e_round()
            e1g = []
            for k in range(len(sets)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    e2e_step(k)
                e1g.append(g)
            for _ in range(max(1, args.warmup // n_round)):
                eg.replay()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(args.steps // n_round):
                eg.replay()
            for i in range(args.steps % n_round):
                e1g[i].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = max_over_ranks(world, e0.elapsed_time(e1), dev)
        e2e = {"value": round(step_bytes * args.steps * world / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": round(ms_e2e / args.steps, 4),
               "copies": "per step one H2D of its inputs and one D2H of its results, pinned host buffers, through "
                         "the public binding; on a copy stream so that step k+1's H2D overlaps step k's calls"}

    layer_dec = None
    if not args.no_layer:
        layer_dec = bench_layer_decode(dev, stream)

    prefill = None
    if not args.no_prefill:
        prefill = bench_prefill(dev, stream)
        _, bf16_peak, bf16_kind = measured_peaks()
        prefill["roofline"] = {"bound": "tensor", "kernel": "row prologue + LoRA down + k_gemm_nvfp4 (whole call)",
                               "achieved": prefill["layer_TFLOPs"], "peak": bf16_peak, "unit": "TFLOP/s",
                               "frac": round(prefill["layer_TFLOPs"] / bf16_peak, 4), "peak_kind": bf16_kind,
                               "peak_note": "dense BF16 cuBLAS burst; the path computes in f16 (same tensor rate)"}

    def guarded(fn):
        try:
            return fn(dev, stream)
        except Exception as e:  # reported, never allowed to cost the line
            return {"error": f"{type(e).__name__}: {e}"}

    extras = None if args.no_extras else guarded(bench_noise_and_fold)
    stack = None if args.no_stack else guarded(bench_stack_32b)
    w8 = None if args.no_extras else guarded(bench_w8a8)
    bwd = None if args.no_extras else guarded(bench_backward)
    quant = None if args.no_extras else guarded(bench_quantize_layer)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args, budget_s=args.cpu_seconds)
        cpu["one_thread"] = cpu_baseline_threads(args, 1, budget_s=args.cpu_seconds)
        try:
            cpu["larger_workloads"] = oracle_layer_timings(budget_s=args.cpu_seconds * 4)
        except Exception as e:
            cpu["larger_workloads"] = {"error": f"{type(e).__name__}: {e}"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": args.workload, "d_i": d_i, "d_o": d_o, "r": r, "lambda": wl.lam,
                       "sigma": wl.sigma, "M_sweep": Ms,
                       "step": ("the five calls of the sweep (independent problems, each its own weight copy and "
                                "input) as one pl_nvfp4_lora_linear_batch call: one prologue + one main kernel"
                                if form == "batch" else "one pl_nvfp4_lora_linear call per M"),
                       "forms": forms_out,
                       "l2": f"{len(sets)} rotating weight copy sets ({len(sets) * len(Ms)} copies, "
                             f"{len(sets) * len(Ms) * per_copy / 2**20:.0f} MiB > 2x L2)",
                       "graphs": f"CUDA graphs of {len(sets)} steps (one per copy set) replayed back to back",
                       "parallelism": f"replicas x{world}"},
            "tflops": round(step_flops * args.steps * world / (ms * 1e-3) / 1e12, 2),
            "per_M": per_m,
            "roofline": roofline,
            "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu, "layer_decode": layer_dec, "prefill": prefill,
            "aqn_and_uaq": extras, "stack_32b": stack, "w8a8": w8, "backward": bwd, "quantize_layer_7b": quant,
            "gpu_launches": launches[form] * args.steps,
        }
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------- AQN draw, UAQ fold
def _graph_us(stream, fn, calls: int = 20, replays: int = 10) -> float:
    """Mean us per call of fn(k) over CUDA graphs of `calls` calls (after one eager pass)."""
    import torch
    with torch.cuda.stream(stream):
        for k in range(3):
            fn(k)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(calls):
                fn(k)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (calls * replays)


def bench_noise_and_fold(dev, stream):
    """The AQN noise draw (per norm state; 64 per-token states; 4096 per-token states of a
    4096-token batch) and the UAQ-folded quantiser next to the plain one, on the 7B
    shapes; us per call from CUDA graphs, GB/s of the bytes each writes or moves."""
    import torch

    from precision_linear_gb300 import binding as pl
    from precision_linear_gb300 import synthetic

    out = {"noise": {}, "quantize": {}}
    for n, d in ((1, 3584), (64, 5120), (4096, 3584)):
        z = torch.empty(n, d, dtype=torch.float32, device=dev)
        us = _graph_us(stream, lambda k: pl.aqn_noise(d, 1, 0, k * n, n, 0.01, out=z))
        out["noise"][f"{n}x{d}"] = {"us": round(us, 2), "GBps_written": round(4 * n * d / (us * 1e3), 1)}
    for d_o, d_i in ((3584, 3584), (18944, 3584)):
        W = synthetic.weight(d_o, d_i, seed=d_o + d_i).to(dev)
        bufs = [pl.nvfp4_quantize(W) for _ in range(2)]
        P = d_o * d_i
        nbytes = 2 * P + 2 * P + 9 * P // 16  # the amax pass, the block pass, the packed output
        plain = _graph_us(stream, lambda k: pl.nvfp4_quantize(W, *bufs[k % 2]), calls=10, replays=5)
        fold = _graph_us(stream, lambda k: pl.nvfp4_quantize_uaq(W, 1.5, *bufs[k % 2]), calls=10, replays=5)
        out["quantize"][f"{d_o}x{d_i}"] = {"plain_us": round(plain, 2), "uaq_us": round(fold, 2),
                                           "plain_GBps": round(nbytes / (plain * 1e3), 1),
                                           "uaq_GBps": round(nbytes / (fold * 1e3), 1)}
        del W, bufs
    torch.cuda.synchronize()
    return out


# ------------------------------------------------------------------------- 7B layer decode
def layer_on_device(cases: dict, dev, keep_weights_on_host: bool = False) -> dict:
    """synthetic.layer_case moved to the device, each distinct tensor once: the
    projections that share a norm keep sharing one device copy of its input."""
    moved = {}

    def mv(t):
        if t is None:
            return None
        if id(t) not in moved:
            moved[id(t)] = t.to(dev)
        return moved[id(t)]

    return {name: {k: (v if (k == "W" and keep_weights_on_host) else mv(v)) for k, v in c.items()}
            for name, c in cases.items()}


def bench_layer_decode(dev, stream, replays: int = 20):
    """The Qwen2.5-7B-shaped decoder-layer projection set at decode batch sizes: the seven
    projections of one layer back to back (q/k/v on norm 1, gate/up on norm 2, o and down
    plain), two weight copies of the layer alternating (262 MB > L2), CUDA graphs; per M
    the layer's time and HBM GB/s of its algorithmic bytes."""
    import torch

    from precision_linear_gb300 import binding as pl
    from precision_linear_gb300 import synthetic

    wl = synthetic.WORKLOADS["layer_7b"]
    r = wl.r
    Mmax = max(wl.Ms)
    ws = pl.Workspace(dev)
    ws.get(max(pl.workspace_bytes(M, p.d_i, p.d_o, r) for M in wl.Ms for p in wl.projs))
    cases = layer_on_device(synthetic.layer_case(wl, 0, Mmax), dev)  # q/k/v and gate/up share their norm's input
    projs = []
    for p in wl.projs:
        c = cases[p.name]
        codes, scales, s_g = pl.nvfp4_quantize(c.pop("W"))
        projs.append(dict(p=p, copies=[(codes, scales, s_g), (codes.clone(), scales.clone(), s_g.clone())], **c))
    ws.get(max(pl.workspace_bytes(M, p.d_i, p.d_o, r) for M in wl.Ms for p in wl.projs) + (64 << 20))
    torch.cuda.synchronize()
    by_name = {q["p"].name: q for q in projs}
    groups = [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]]
    out = {}
    with torch.cuda.stream(stream):
        for M in wl.Ms:
            ys = {q["p"].name: torch.empty(M, q["p"].d_o, dtype=torch.bfloat16, device=dev) for q in projs}

            def separate(k):
                for q in projs:
                    codes, scales, s_g = q["copies"][k]
                    pl.nvfp4_lora_linear(q["x"][:M], codes, scales, s_g, q["A"], q["B"], wl.lam, q["w_norm"], q["z"],
                                         synthetic.EPS, out=ys[q["p"].name], workspace=ws)

            def grouped(k):
                for gn in groups:
                    q0 = by_name[gn[0]]
                    lst = [dict(zip(("codes", "scales", "s_g"), by_name[n]["copies"][k]), A=by_name[n]["A"],
                                B=by_name[n]["B"], lam=wl.lam) for n in gn]
                    pl.nvfp4_lora_linear_group(q0["x"][:M], lst, q0["w_norm"], q0["z"], synthetic.EPS,
                                               outs=[ys[n] for n in gn], workspace=ws)

            nbytes = sum(algorithmic_bytes(M, q["p"].d_i, q["p"].d_o, r) for q in projs)
            e = {}
            for name, fn in (("separate", separate), ("grouped", grouped)):
                fn(0)
                fn(1)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    fn(0)
                    fn(1)
                g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(replays):
                    g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                us = e0.elapsed_time(e1) * 1e3 / (2 * replays)
                e[name] = {"us_per_layer": round(us, 1), "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                           "tokens_per_s_per_layer": round(M / (us * 1e-6), 1)}
                del g
            best = min(e.values(), key=lambda v: v["us_per_layer"])
            out[str(M)] = {"us_per_layer": best["us_per_layer"], "GBps": best["GBps"],
                           "frac_of_hbm": round(best["GBps"] / measured_peaks()[0], 4), **e,
                           "paths": {q["p"].name: pl.linear_path(M, q["p"].d_i, q["p"].d_o, r) for q in projs}}
    torch.cuda.synchronize()
    return {"workload": "layer_7b (Qwen2.5-7B decoder-layer projection set, r=32; q/k/v and gate/up share their "
                        "norm's input)", "per_M": out,
            "forms": "separate: seven calls; grouped: q/k/v, o, gate/up, down as four group calls",
            "timing": f"CUDA events around {replays} replays of a CUDA graph of two layers (two weight copies)"}


# ------------------------------------------------------------------------- large-M path
def bench_prefill(dev, stream, reps: int = 5, replays: int = 3):
    """The Qwen2.5-7B-shaped layer set at M = 4096 (log-prob recompute): every projection
    through the large-M tensor-core path, timed with CUDA events on the launching stream,
    as seven separate calls and as four calls with q/k/v and gate/up grouped on their
    norm's shared input; returns per-projection, per-call and whole-layer TFLOPS."""
    import torch

    from precision_linear_gb300 import binding as pl
    from precision_linear_gb300 import synthetic

    wl = synthetic.WORKLOADS["prefill_7b"]
    M, r = wl.Ms[0], wl.r
    ws = pl.Workspace(dev)
    cases = layer_on_device(synthetic.layer_case(wl, 0, M), dev, keep_weights_on_host=True)
    proj = {}
    with torch.cuda.stream(stream):
        for p in wl.projs:
            c = cases[p.name]
            W = c["W"].to(dev)
            codes, scales, s_g = pl.nvfp4_quantize(W)
            del W
            proj[p.name] = dict(p=p, codes=codes, scales=scales, s_g=s_g, x=c["x"], A=c["A"], B=c["B"],
                                w_norm=c["w_norm"], z=c["z"],
                                y=torch.empty(M, p.d_o, dtype=torch.bfloat16, device=dev))
    torch.cuda.synchronize()

    def time_call(call):
        with torch.cuda.stream(stream):
            for _ in range(2):
                call()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()  # reps calls back to back, free of host launch gaps
            with torch.cuda.graph(g, stream=stream):
                for _ in range(reps):
                    call()
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(replays):
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            del g
        return e0.elapsed_time(e1) / (reps * replays)

    # seven separate calls
    out, tot_flops, tot_ms = {}, 0, 0.0
    for name, q in proj.items():
        p = q["p"]
        ws.get(pl.workspace_bytes(M, p.d_i, p.d_o, r))
        ms = time_call(lambda q=q: pl.nvfp4_lora_linear(q["x"], q["codes"], q["scales"], q["s_g"], q["A"], q["B"],
                                                        wl.lam, q["w_norm"], q["z"], synthetic.EPS, out=q["y"],
                                                        workspace=ws))
        fl = algorithmic_flops(M, p.d_i, p.d_o, r)
        out[name] = {"d_i": p.d_i, "d_o": p.d_o, "us_per_call": round(ms * 1e3, 1),
                     "TFLOPs": round(fl / (ms * 1e-3) / 1e12, 1), "path": pl.linear_path(M, p.d_i, p.d_o, r)}
        tot_flops += fl
        tot_ms += ms

    # four calls: q/k/v and gate/up as groups on their norm's input
    groups = [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]]
    grouped, g_ms = {}, 0.0
    for names in groups:
        members = [proj[n] for n in names]
        c0 = members[0]
        specs = [dict(codes=q["codes"], scales=q["scales"], s_g=q["s_g"], A=q["A"], B=q["B"], lam=wl.lam)
                 for q in members]
        outs = [q["y"] for q in members]
        if len(names) > 1:  # the binding sizes the workspace in the eager warm-up calls
            call = lambda c0=c0, specs=specs, outs=outs: pl.nvfp4_lora_linear_group(
                c0["x"], specs, c0["w_norm"], c0["z"], synthetic.EPS, outs=outs, workspace=ws)
        else:
            q = c0
            ws.get(pl.workspace_bytes(M, q["p"].d_i, q["p"].d_o, r))
            call = lambda q=q: pl.nvfp4_lora_linear(q["x"], q["codes"], q["scales"], q["s_g"], q["A"], q["B"], wl.lam,
                                                    q["w_norm"], q["z"], synthetic.EPS, out=q["y"], workspace=ws)
        ms = time_call(call)
        fl = sum(algorithmic_flops(M, q["p"].d_i, q["p"].d_o, r) for q in members)
        grouped["/".join(names)] = {"us_per_call": round(ms * 1e3, 1), "TFLOPs": round(fl / (ms * 1e-3) / 1e12, 1)}
        g_ms += ms
    torch.cuda.synchronize()
    sep = {"layer_us": round(tot_ms * 1e3, 1), "layer_TFLOPs": round(tot_flops / (tot_ms * 1e-3) / 1e12, 1)}
    grp = {"layer_us": round(g_ms * 1e3, 1), "layer_TFLOPs": round(tot_flops / (g_ms * 1e-3) / 1e12, 1),
           "calls": grouped}
    best = grp if g_ms < tot_ms else sep
    return {"workload": "prefill_7b (Qwen2.5-7B layer set, M=4096, r=32)", "M": M,
            "layer_us": best["layer_us"], "layer_TFLOPs": best["layer_TFLOPs"],
            "form": "grouped" if best is grp else "separate",
            "separate": sep, "grouped": grp, "per_proj": out,
            "timing": f"CUDA events around {replays} replays of a CUDA graph of {reps} calls "
                      f"(after 2 eager warm-up calls and one replay)"}


# ------------------------------------------------------------------------- 32B decode stack
def _layer_weights_on_gpu(wl, layer, dev):
    """NVFP4 weights and adapters of one layer, drawn on the device from the layer's seeds
    (the seeded CUDA generator of synthetic.py) and quantised by the library."""
    from precision_linear_gb300 import binding as pl
    from precision_linear_gb300 import synthetic
    out = {}
    for i, p in enumerate(wl.projs):
        sd = synthetic.proj_seed(wl, layer, i)
        W = synthetic.weight(p.d_o, p.d_i, sd, wl.outlier_frac, device=dev)
        codes, scales, s_g = pl.nvfp4_quantize(W)
        del W
        A, B = synthetic.lora(p.d_o, p.d_i, wl.r, sd, device=dev)
        out[p.name] = dict(codes=codes, scales=scales, s_g=s_g, A=A, B=B, lam=wl.lam)
    return out


def bench_stack_32b(dev, stream, replays: int = 3):
    """One decode step through the 64 layers of the Qwen2.5-32B-shaped stack (18.7 GB of
    distinct NVFP4 weights, no reuse), at M in {1, 16, 64}: per layer q/k/v on the attention
    norm's input, o on a plain input, gate/up on the FFN norm's input, down on a plain input.
    Two launch forms: every projection its own call, and the projections behind one norm as
    one group call.  GB/s of algorithmic bytes, tokens/s = M / step time."""
    import torch

    from precision_linear_gb300 import binding as pl
    from precision_linear_gb300 import synthetic

    wl = synthetic.WORKLOADS["stack_32b"]
    Mmax = max(wl.Ms)
    layers = [_layer_weights_on_gpu(wl, l, dev) for l in range(wl.layers)]
    torch.cuda.synchronize()
    # activations: one draw per input shape, shared by the layers (they do not change the
    # weight stream, which is what the step measures)
    act = synthetic.layer_case(wl, 0, Mmax)
    inp = {}
    for p in wl.projs:
        c = act[p.name]
        inp[p.name] = dict(x=c["x"].to(dev), w_norm=c["w_norm"].to(dev) if c["w_norm"] is not None else None,
                           z=c["z"].to(dev) if c["z"] is not None else None)
    for nm in ("k", "v"):  # the shared norm input stays one tensor
        inp[nm] = inp["q"]
    inp["up"] = inp["gate"]
    ws = pl.Workspace(dev)
    ws.get(256 << 20)
    groups = [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]]
    per_layer_bytes = {M: sum(algorithmic_bytes(M, p.d_i, p.d_o, wl.r) for p in wl.projs) for M in wl.Ms}
    res = {}
    with torch.cuda.stream(stream):
        for M in wl.Ms:
            ys = {p.name: torch.empty(M, p.d_o, dtype=torch.bfloat16, device=dev) for p in wl.projs}

            def separate():
                for L in layers:
                    for p in wl.projs:
                        q, a = L[p.name], inp[p.name]
                        pl.nvfp4_lora_linear(a["x"][:M], q["codes"], q["scales"], q["s_g"], q["A"], q["B"], q["lam"],
                                             a["w_norm"], a["z"], synthetic.EPS, out=ys[p.name], workspace=ws)

            def grouped():
                for L in layers:
                    for gnames in groups:
                        a = inp[gnames[0]]
                        pl.nvfp4_lora_linear_group(a["x"][:M], [L[n] for n in gnames], a["w_norm"], a["z"],
                                                   synthetic.EPS, outs=[ys[n] for n in gnames], workspace=ws)

            out = {}
            for name, fn in (("separate", separate), ("grouped", grouped)):
                fn()
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    fn()
                g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(replays):
                    g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / replays
                nb = per_layer_bytes[M] * wl.layers
                out[name] = {"ms_per_step": round(ms, 3), "GBps": round(nb / (ms * 1e-3) / 1e9, 1),
                             "tokens_per_s": round(M / (ms * 1e-3), 1)}
                del g
            best = max(out.values(), key=lambda v: v["GBps"])
            out["best_frac_of_hbm"] = round(best["GBps"] / measured_peaks()[0], 4)
            res[str(M)] = out
    del layers
    torch.cuda.synchronize()
    return {"workload": "stack_32b (Qwen2.5-32B-shaped decode step, 64 layers, r=32, sigma=5e-3)",
            "weights_GB": round(sum(9 * p.d_o * p.d_i // 16 for p in wl.projs) * wl.layers / 1e9, 2),
            "per_M": res, "timing": f"CUDA events around {replays} replays of a CUDA graph of one 64-layer step"}


# ------------------------------------------------------------------------- W8A8 and backward
def bench_w8a8(dev, stream):
    """The FP8 W8A8 rollout linear on the 7B layer set: decode (M in {8, 64}, one call per
    projection, two weight copies, HBM GB/s) and M = 4096 (TFLOP/s)."""
    import torch

    from precision_linear_gb300 import binding as pl
    from precision_linear_gb300 import synthetic

    wl = synthetic.WORKLOADS["layer_7b"]
    cases = layer_on_device(synthetic.layer_case(wl, 0, 4096), dev)
    projs = {}
    for p in wl.projs:
        c = cases[p.name]
        codes, s_w = pl.w8a8_quantize_weight(c.pop("W"))
        projs[p.name] = dict(p=p, copies=[(codes, s_w), (codes.clone(), s_w.clone())], **c)
    ws = pl.Workspace(dev)
    ws.get(max(pl.lib().pl_w8a8_workspace_bytes(4096, p.d_i, p.d_o, wl.r) for p in wl.projs))
    out = {}
    with torch.cuda.stream(stream):
        for M in (8, 64, 4096):
            ys = {n: torch.empty(M, q["p"].d_o, dtype=torch.bfloat16, device=dev) for n, q in projs.items()}

            def layer(k):
                for n, q in projs.items():
                    codes, s_w = q["copies"][k % 2]
                    pl.w8a8_lora_linear(q["x"][:M], codes, s_w, q["A"], q["B"], wl.lam, q["w_norm"], q["z"],
                                        synthetic.EPS, out=ys[n], workspace=ws)

            us = _graph_us(stream, layer, calls=2, replays=5 if M == 4096 else 20) / 1  # per layer
            nbytes = sum(M * (q["p"].d_i + q["p"].d_o) * 2 + q["p"].d_o * (q["p"].d_i + 4) +
                         2 * wl.r * (q["p"].d_i + q["p"].d_o) + 8 * q["p"].d_i for q in projs.values())
            flops = sum(algorithmic_flops(M, q["p"].d_i, q["p"].d_o, wl.r) for q in projs.values())
            e = {"us_per_layer": round(us, 1), "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                 "TFLOPs": round(flops / (us * 1e-6) / 1e12, 1)}
            out[str(M)] = e
    torch.cuda.synchronize()
    return {"workload": "layer_7b, FP8 E4M3 W8A8 (per-channel weight, per-token activation scales) + LoRA r=32",
            "per_M": out, "bytes": "d_o (d_i + 4) weight + scale bytes, adapters, activations in and out",
            "timing": "CUDA events around replays of a CUDA graph of two layers (two weight copies)"}


def bench_backward(dev, stream):
    """The frozen-backbone backward (dx through the norm, dA, dB) of the 7B layer set at
    M = 4096 (the log-prob / backward phase), TFLOP/s of 2 M (d_o d_i + r (d_i + d_o)) for dx
    plus the adapter gradients' 4 M r (d_i + d_o)."""
    import torch

    from precision_linear_gb300 import binding as pl
    from precision_linear_gb300 import synthetic

    wl = synthetic.WORKLOADS["prefill_7b"]
    M = wl.Ms[0]
    cases = layer_on_device(synthetic.layer_case(wl, 0, M), dev)
    ws = pl.Workspace(dev)
    out, tot_us, tot_fl = {}, 0.0, 0
    gen = torch.Generator(device=dev)
    gen.manual_seed(77)
    with torch.cuda.stream(stream):
        for p in wl.projs:
            c = cases[p.name]
            codes, scales, s_g = pl.nvfp4_quantize(c["W"])
            g = torch.randn(M, p.d_o, generator=gen, device=dev).to(torch.bfloat16)

            def call(k):
                pl.nvfp4_lora_linear_backward(g, c["x"], codes, scales, s_g, c["A"], c["B"], wl.lam, c["w_norm"],
                                              c["z"], synthetic.EPS, workspace=ws)

            call(0)
            torch.cuda.synchronize()
            us = _graph_us(stream, call, calls=2, replays=3)
            fl = 2 * M * (p.d_o * p.d_i + wl.r * (p.d_i + p.d_o)) + 4 * M * wl.r * (p.d_i + p.d_o)
            out[p.name] = {"us_per_call": round(us, 1), "TFLOPs": round(fl / (us * 1e-6) / 1e12, 1)}
            tot_us += us
            tot_fl += fl
            del codes, scales, s_g, g
    torch.cuda.synchronize()
    return {"workload": "prefill_7b layer set, backward at M=4096 (dx, dA, dB)", "per_proj": out,
            "layer_us": round(tot_us, 1), "layer_TFLOPs": round(tot_fl / (tot_us * 1e-6) / 1e12, 1)}


def bench_quantize_layer(dev, stream):
    """BF16 -> NVFP4 of all seven 7B weight matrices (466 MB of BF16): bytes are the two reads
    of 2P and the 9P/16 written, per matrix and in total."""
    import torch

    from precision_linear_gb300 import binding as pl
    from precision_linear_gb300 import synthetic

    wl = synthetic.WORKLOADS["layer_7b"]
    Ws = [synthetic.weight(p.d_o, p.d_i, synthetic.proj_seed(wl, 0, i), device=dev) for i, p in enumerate(wl.projs)]
    bufs = [pl.nvfp4_quantize(W) for W in Ws]

    def all7(k):
        for W, b in zip(Ws, bufs):
            pl.nvfp4_quantize(W, *b)

    us = _graph_us(stream, all7, calls=2, replays=5)
    P = sum(W.numel() for W in Ws)
    nbytes = 2 * P + 2 * P + 9 * P // 16
    res = {"bf16_MB": round(2 * P / 1e6, 1), "us_per_layer": round(us, 1), "GBps": round(nbytes / (us * 1e3), 1),
           "frac_of_hbm": round(nbytes / (us * 1e3) / measured_peaks()[0], 4)}
    del Ws, bufs
    torch.cuda.synchronize()
    return res


# ------------------------------------------------------------------------- oracle timing
def cpu_baseline(args, budget_s: float = 15.0, max_calls: int | None = None):
    """The CPU oracle, as it stands, on a bounded sample of the same workload:
    calls of the M sweep in order until the time budget (or call budget) is spent."""
    import numpy as np

    from oracle import linear as olin
    from oracle import nvfp4 as onv
    from precision_linear_gb300 import synthetic

    wl = synthetic.WORKLOADS[args.workload]
    p = wl.projs[0]
    d_i, d_o, r = p.d_i, p.d_o, wl.r
    c = synthetic.projection_case(d_o, d_i, max(wl.Ms), r, wl.sigma, wl.seed, wl.outlier_frac)
    f = lambda t: t.float().numpy()
    packed, sb, s_g = onv.quantize(f(c["W"]))
    x, A, B, w, z = (f(c[k]).astype(np.float64) for k in ("x", "A", "B", "w_norm", "z"))
    done_bytes, t0, calls = 0, time.perf_counter(), 0
    while True:
        M = wl.Ms[calls % len(wl.Ms)]
        olin.nvfp4_lora_linear(x[:M], packed, sb, s_g, A, B, wl.lam, w, z, synthetic.EPS)
        done_bytes += algorithmic_bytes(M, d_i, d_o, r)
        calls += 1
        if (max_calls is not None and calls >= max_calls) or time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    try:
        from threadpoolctl import threadpool_info
        cores = max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:  # not installed: the BLAS pool's size as the environment sets it, else every core
        cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)))
    return {"value": round(done_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{calls} oracle calls over the M sweep {list(wl.Ms)} of {args.workload} "
                      f"(dequantise + FP64 RMSNorm-AQN + FP64 matmul + LoRA), {dt:.1f} s"}


def cpu_baseline_threads(args, threads: int, budget_s: float = 12.0):
    """cpu_baseline in a child process whose BLAS and OpenMP pools are pinned to `threads`."""
    env = dict(os.environ, OMP_NUM_THREADS=str(threads), OPENBLAS_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads))
    code = ("import json, sys; sys.path.insert(0, %r); import bench, argparse; "
            "a = argparse.Namespace(workload=%r); print(json.dumps(bench.cpu_baseline(a, budget_s=%r)))"
            % (ROOT, args.workload, budget_s))
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                             timeout=budget_s * 4 + 60)
        res = json.loads(out.stdout.strip().splitlines()[-1])
        res["cores"] = threads
        return res
    except Exception as e:
        return {"error": f"{type(e).__name__}: {e}"}


def oracle_layer_timings(budget_s: float = 60.0):
    """The oracle on the larger workloads, within a time budget (as it stands; reported, not a
    target): the 7B layer set at M = 64 (dequantise + FP64 RMSNorm-AQN + FP64 matmul + LoRA per
    projection), the FP64 matmul of the 7B layer set at M = 4096, and sampled layers of the
    32B stack at M = 16 extrapolated x64.  Timing only: the packed weights are seeded random
    bytes of the NVFP4 layout (valid codes and finite scales), since the oracle's own quantiser
    would take minutes on these sizes and the linear's cost does not depend on the values."""
    import numpy as np

    from oracle import linear as olin
    from oracle import nvfp4 as onv
    from precision_linear_gb300 import synthetic

    rng = np.random.default_rng(0)

    def packed_weight(d_o, d_i):
        codes = rng.integers(0, 256, size=(d_o, d_i // 2), dtype=np.uint8)
        scales = rng.integers(0x20, 0x50, size=(d_o, d_i // 16), dtype=np.uint8)  # finite, moderate scales
        return codes, scales, np.float32(1e-3)

    def layer(wl, M, seed):
        t = 0.0
        for p in wl.projs:
            codes, scales, s_g = packed_weight(p.d_o, p.d_i)
            x = rng.standard_normal((M, p.d_i))
            A = rng.standard_normal((wl.r, p.d_i)) * 0.02
            B = rng.standard_normal((p.d_o, wl.r)) * 0.02
            w = 1 + 0.1 * rng.standard_normal(p.d_i) if p.norm else None
            z = wl.sigma * rng.standard_normal(p.d_i) if p.norm else None
            t0 = time.perf_counter()
            olin.nvfp4_lora_linear(x, codes, scales, s_g, A, B, wl.lam, w, z, synthetic.EPS)
            t += time.perf_counter() - t0
        return t

    out = {"cores": os.cpu_count(), "kind": "oracle"}
    start = time.perf_counter()
    wl3 = synthetic.WORKLOADS["layer_7b"]
    # config 4 first: the FP64 matmul of the whole layer set at M = 4096 (weights dequantised
    # in FP64, untimed), then config 3: the full oracle of the layer set at M = 64
    fl, t4, n4 = 0, 0.0, 0
    for p in wl3.projs:
        codes, scales, s_g = packed_weight(p.d_o, p.d_i)
        W = onv.dequantize(codes, scales, s_g)
        h = rng.standard_normal((4096, p.d_i))
        t0 = time.perf_counter()
        h @ W.T
        t4 += time.perf_counter() - t0
        fl += 2 * 4096 * p.d_i * p.d_o
        n4 += 1
        del W, h
    out["prefill_7b_M4096_fp64_matmul"] = {"s": round(t4, 2), "TFLOPs": round(fl / max(t4, 1e-9) / 1e12, 4),
                                           "projections": n4}
    t3 = layer(wl3, 64, 1)
    b3 = sum(algorithmic_bytes(64, p.d_i, p.d_o, wl3.r) for p in wl3.projs)
    out["layer_7b_M64"] = {"s_per_layer": round(t3, 2), "GBps": round(b3 / t3 / 1e9, 4)}
    wl5 = synthetic.WORKLOADS["stack_32b"]
    done, t5 = [], 0.0
    for lay in (0, 31, 63):
        if done and time.perf_counter() - start + t5 / len(done) > budget_s:
            break
        t5 += layer(wl5, 16, 5000 + lay)
        done.append(lay)
    b5 = sum(algorithmic_bytes(16, p.d_i, p.d_o, wl5.r) for p in wl5.projs) * wl5.layers
    step = t5 / len(done) * wl5.layers
    out["stack_32b_M16"] = {"layers_timed": done, "s_per_step_extrapolated_x64": round(step, 1),
                            "GBps": round(b5 / step / 1e9, 4), "tokens_per_s": round(16 / step, 4)}
    out["wall_s"] = round(time.perf_counter() - start, 1)
    return out


def synthetic_ms(args):
    from precision_linear_gb300 import synthetic
    return synthetic.WORKLOADS[args.workload].Ms


def run_reference(args, world, rank):
    if rank != 0:
        return
    # each step: one oracle call (one M of the sweep), so K + W steps stay within minutes
    per_step = max(0.05, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(args, budget_s=per_step, max_calls=1)
    vals, t0 = [], time.perf_counter()
    res = None
    for _ in range(args.steps):
        res = cpu_baseline(args, budget_s=per_step, max_calls=len(synthetic_ms(args)))
        vals.append(res["value"])
    dt = time.perf_counter() - t0
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload,
                       "step": f"oracle sample: up to one call per M of the sweep, <= {per_step:.2f} s"},
            "cpu_baseline": {"value": round(value, 4), "kind": res["kind"], "cores": res["cores"],
                             "sample": res["sample"]},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_proj_7b")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the M=4096 layer-set measurement")
    ap.add_argument("--no-layer", action="store_true", help="skip the 7B decoder-layer decode measurement")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the AQN draw, UAQ quantiser, W8A8, backward and layer quantiser timings")
    ap.add_argument("--no-stack", action="store_true", help="skip the 64-layer 32B-shaped decode step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        from precision_linear_gb300 import build
        if rank == 0:
            build.build()
        barrier(world)
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
