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

    # CUDA graphs: one per copy set (= one step), and one "round" graph holding a
    # step on every copy set, so that the GPU runs far ahead of the host
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)  # every launch, replay and event below is on this stream
    graphs = []
    with torch.cuda.stream(stream):
        for calls in sets:  # warm (tensor-map encode, attribute set-up) outside capture
            for c in calls:
                one_call(c)
        torch.cuda.synchronize()
        for calls in sets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for c in calls:
                    one_call(c)
            graphs.append(g)
        round_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(round_graph, stream=stream):
            for calls in sets:
                for c in calls:
                    one_call(c)
    torch.cuda.synchronize()
    n_round = len(sets)

    def run_steps(k):
        """Exactly k steps: whole rounds, then single-step graphs for the rest."""
        for _ in range(k // n_round):
            round_graph.replay()
        for i in range(k % n_round):
            graphs[i].replay()
    paths = {M: pl.linear_path(M, d_i, d_o, r) for M in Ms}
    launches_per_call = {M: (1 if paths[M] == 2 else 2) for M in Ms}  # fused kernel, or prologue + main
    step_bytes = sum(algorithmic_bytes(M, d_i, d_o, r) for M in Ms)
    step_flops = sum(algorithmic_flops(M, d_i, d_o, r) for M in Ms)

    run_steps(args.warmup)
    torch.cuda.synchronize()

    # ---- timed region: K steps (clocks sampled from a 1 s soak just before it through its end)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t_soak = time.perf_counter()
        i = 0
        while time.perf_counter() - t_soak < 1.0:
            run_steps(20 * n_round)
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        run_steps(args.steps)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(world, ms, dev)
    clocks = clk.summary()
    total_bytes = step_bytes * args.steps * world
    value = total_bytes / (ms * 1e-3) / 1e9

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
                         "TFLOPs": round(algorithmic_flops(M, d_i, d_o, r) / (us * 1e-6) / 1e12, 2)}
    dom = max(per_m, key=lambda k: per_m[k]["us_per_call"])
    hbm_peak, _, peak_kind = measured_peaks()
    achieved = per_m[dom]["GBps"]

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
            for c in sets[k]:
                one_call(c)
            hy.copy_(y_bufs[k], non_blocking=True)  # D2H of the step's results

        with torch.cuda.stream(stream):
            eg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(eg, stream=stream):
                for k in range(len(sets)):
                    e2e_step(k)
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
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": round(ms_e2e / args.steps, 4)}

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

    extras = None
    if not args.no_extras:
        try:
            extras = bench_noise_and_fold(dev, stream)
        except Exception as e:  # reported, never allowed to cost the line
            extras = {"error": f"{type(e).__name__}: {e}"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args, budget_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": args.workload, "d_i": d_i, "d_o": d_o, "r": r, "lambda": wl.lam,
                       "sigma": wl.sigma, "M_sweep": Ms, "step": "one call per M (one fused kernel per call)" if all(v == 2 for v in paths.values()) else "one call per M",
                       "l2": f"{len(sets)} rotating weight copy sets ({len(sets) * len(Ms)} copies, "
                             f"{len(sets) * len(Ms) * per_copy / 2**20:.0f} MiB > 2x L2)",
                       "graphs": f"CUDA graphs of {len(sets)} steps (one per copy set) replayed back to back",
                       "parallelism": f"replicas x{world}"},
            "tflops": round(step_flops * args.steps * world / (ms * 1e-3) / 1e12, 2),
            "per_M": per_m,
            "roofline": {"bound": "hbm", "kernel": ("k_fused_decode" if paths[int(dom)] == 2 else "k_act + k_tc_decode")
                         + " (CUDA events around each call on its stream)",
                         "M": int(dom), "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                         "traffic": profile_traffic("k_fused_decode" if paths[int(dom)] == 2 else "k_tc_decode",
                                                    f"{args.workload}/M{dom}")},
            "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu, "layer_decode": layer_dec, "prefill": prefill,
            "aqn_and_uaq": extras,
            "gpu_launches": sum(launches_per_call.values()) * args.steps,
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
    torch.cuda.synchronize()
    out = {}
    with torch.cuda.stream(stream):
        for M in wl.Ms:
            ys = [torch.empty(M, q["p"].d_o, dtype=torch.bfloat16, device=dev) for q in projs]

            def layer(k):
                for q, y in zip(projs, ys):
                    codes, scales, s_g = q["copies"][k]
                    pl.nvfp4_lora_linear(q["x"][:M], codes, scales, s_g, q["A"], q["B"], wl.lam, q["w_norm"], q["z"],
                                         synthetic.EPS, out=y, workspace=ws)

            layer(0)
            layer(1)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                layer(0)
                layer(1)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(replays):
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (2 * replays)
            nbytes = sum(algorithmic_bytes(M, q["p"].d_i, q["p"].d_o, r) for q in projs)
            out[str(M)] = {"us_per_layer": round(us, 1), "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                           "paths": {q["p"].name: pl.linear_path(M, q["p"].d_i, q["p"].d_o, r) for q in projs}}
    torch.cuda.synchronize()
    return {"workload": "layer_7b (Qwen2.5-7B decoder-layer projection set, r=32)", "per_M": out,
            "timing": f"CUDA events around {replays} replays of a CUDA graph of two layers (two weight copies)"}


# ------------------------------------------------------------------------- large-M path
def bench_prefill(dev, stream, reps: int = 5, replays: int = 3):
    """The Qwen2.5-7B-shaped layer set at M = 4096 (log-prob recompute): every
    projection through the large-M tensor-core path, timed with CUDA events on the
    launching stream; returns per-projection and whole-layer TFLOPS."""
    import torch

    from precision_linear_gb300 import binding as pl
    from precision_linear_gb300 import synthetic

    wl = synthetic.WORKLOADS["prefill_7b"]
    M, r = wl.Ms[0], wl.r
    ws = pl.Workspace(dev)
    out, tot_flops, tot_ms = {}, 0, 0.0
    cases = layer_on_device(synthetic.layer_case(wl, 0, M), dev, keep_weights_on_host=True)
    with torch.cuda.stream(stream):
        for p in wl.projs:
            c = cases[p.name]
            W = c["W"].to(dev)
            codes, scales, s_g = pl.nvfp4_quantize(W)
            del W
            x, A, B, w_norm, z = c["x"], c["A"], c["B"], c["w_norm"], c["z"]
            y = torch.empty(M, p.d_o, dtype=torch.bfloat16, device=dev)
            ws.get(pl.workspace_bytes(M, p.d_i, p.d_o, r))

            def call():
                pl.nvfp4_lora_linear(x, codes, scales, s_g, A, B, wl.lam, w_norm, z, synthetic.EPS, out=y, workspace=ws)

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
            ms = e0.elapsed_time(e1) / (reps * replays)
            del g
            fl = algorithmic_flops(M, p.d_i, p.d_o, r)
            out[p.name] = {"d_i": p.d_i, "d_o": p.d_o, "us_per_call": round(ms * 1e3, 1),
                           "TFLOPs": round(fl / (ms * 1e-3) / 1e12, 1), "path": pl.linear_path(M, p.d_i, p.d_o, r)}
            tot_flops += fl
            tot_ms += ms
            del codes, scales, s_g, x, A, B, w_norm, z, y
            cases[p.name] = None
    torch.cuda.synchronize()
    return {"workload": "prefill_7b (Qwen2.5-7B layer set, M=4096, r=32)", "M": M,
            "layer_us": round(tot_ms * 1e3, 1), "layer_TFLOPs": round(tot_flops / (tot_ms * 1e-3) / 1e12, 1),
            "per_proj": out, "timing": f"CUDA events around {replays} replays of a CUDA graph of {reps} calls per "
                                       f"projection (after 2 eager warm-up calls and one replay)"}


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
    except Exception:
        cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": round(done_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{calls} oracle calls over the M sweep {list(wl.Ms)} of {args.workload} "
                      f"(dequantise + FP64 RMSNorm-AQN + FP64 matmul + LoRA), {dt:.1f} s"}


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
    ap.add_argument("--no-extras", action="store_true", help="skip the AQN draw and UAQ quantiser timings")
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
