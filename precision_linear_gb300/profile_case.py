"""A small, self-contained run of one library call for profilers (ncu).

    python -m precision_linear_gb300.profile_case --op linear --workload decode_proj_7b --M 64 --calls 6
    python -m precision_linear_gb300.profile_case --op quantize --workload decode_proj_7b --calls 3
    python -m precision_linear_gb300.profile_case --op w8a8 --workload prefill_7b --M 4096 --calls 2
    python -m precision_linear_gb300.profile_case --op backward --workload prefill_7b --M 4096 --calls 2
    python -m precision_linear_gb300.profile_case --op group --workload layer_7b --proj 4 --M 8 --calls 3

It draws the seeded workload, quantises its weight once, makes enough distinct
weight copies that the set is larger than L2 (so each profiled launch reads its
weights from DRAM), then issues `--calls` back-to-back calls over the copies
and synchronises.  Nothing is timed here; use bench.py for numbers.
"""

from __future__ import annotations

import argparse

import torch

from . import binding as pl
from . import synthetic


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["linear", "quantize", "rmsnorm", "w8a8", "backward", "group", "batch"], default="linear")
    ap.add_argument("--workload", default="decode_proj_7b")
    ap.add_argument("--proj", type=int, default=0, help="index of the projection in the workload")
    ap.add_argument("--M", type=int, default=64)
    ap.add_argument("--calls", type=int, default=6)
    ap.add_argument("--copies", type=int, default=0, help="distinct weight copies (0: enough for > 2x L2)")
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    wl = synthetic.WORKLOADS[a.workload]
    p = wl.projs[a.proj]
    c = synthetic.projection_case(p.d_o, p.d_i, a.M, wl.r, wl.sigma, wl.seed, wl.outlier_frac, device="cpu")
    g = {k: v.to(dev) for k, v in c.items()}
    if a.op == "quantize":
        for _ in range(a.calls):
            pl.nvfp4_quantize(g["W"])
        torch.cuda.synchronize()
        return
    if a.op == "rmsnorm":
        for _ in range(a.calls):
            pl.rmsnorm_aqn(g["x"], g["w_norm"], g["z"], synthetic.EPS)
        torch.cuda.synchronize()
        return
    if a.op == "w8a8":
        codes, s_w = pl.w8a8_quantize_weight(g["W"])
        for _ in range(a.calls):
            pl.w8a8_lora_linear(g["x"], codes, s_w, g["A"], g["B"], wl.lam, g["w_norm"], g["z"], synthetic.EPS)
        torch.cuda.synchronize()
        return
    if a.op == "backward":
        codes, scales, s_g = pl.nvfp4_quantize(g["W"])
        gr = torch.randn(a.M, p.d_o, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).to(dev)
        for _ in range(a.calls):
            pl.nvfp4_lora_linear_backward(gr, g["x"], codes, scales, s_g, g["A"], g["B"], wl.lam, g["w_norm"], g["z"],
                                          synthetic.EPS)
        torch.cuda.synchronize()
        return
    if a.op == "batch":  # the workload's projection at every M of its sweep, one batch call per weight set
        batches = []
        per = 9 * p.d_o * p.d_i // 16 * len(wl.Ms)
        for k in range(a.copies or max(2, (2 * 129 * 2 ** 20) // per + 1)):  # weight sets larger than 2x L2
            calls = []
            for M in wl.Ms:
                cc = synthetic.projection_case(p.d_o, p.d_i, M, wl.r, wl.sigma, wl.seed + M, wl.outlier_frac)
                co, sc, sg = pl.nvfp4_quantize(cc["W"].to(dev))
                calls.append(dict(x=cc["x"].to(dev), codes=co, scales=sc, s_g=sg, A=cc["A"].to(dev),
                                  B=cc["B"].to(dev), lam=wl.lam, w_norm=cc["w_norm"].to(dev), z=cc["z"].to(dev)))
            batches.append(calls)
        for i in range(a.calls):
            pl.nvfp4_lora_linear_batch(batches[i % len(batches)], synthetic.EPS)
        torch.cuda.synchronize()
        return
    if a.op == "group":  # the projections of the workload behind the same norm as --proj, one group call
        cases = synthetic.layer_case(wl, 0, a.M)
        names = [q.name for q in wl.projs if q.norm == p.norm and q.norm is not None] or [p.name]
        c0 = cases[names[0]]
        projs = []
        for n in names:
            cc, ss, sg = pl.nvfp4_quantize(cases[n]["W"].to(dev))
            projs.append(dict(codes=cc, scales=ss, s_g=sg, A=cases[n]["A"].to(dev), B=cases[n]["B"].to(dev),
                              lam=wl.lam))
        x, w, z = c0["x"].to(dev), c0["w_norm"].to(dev), c0["z"].to(dev)
        for _ in range(a.calls):
            pl.nvfp4_lora_linear_group(x, projs, w, z, synthetic.EPS)
        torch.cuda.synchronize()
        return
    codes, scales, s_g = pl.nvfp4_quantize(g["W"])
    per = codes.numel() + scales.numel()
    n = a.copies or max(2, (2 * 129 * 2 ** 20) // per + 1)
    copies = [(codes.clone(), scales.clone(), s_g.clone()) for _ in range(n)]
    norm = p.norm is not None
    ws = pl.Workspace(dev)
    y = torch.empty(a.M, p.d_o, dtype=torch.bfloat16, device=dev)
    for i in range(a.calls):
        cc, ss, sg = copies[i % n]
        pl.nvfp4_lora_linear(g["x"], cc, ss, sg, g["A"], g["B"], wl.lam, g["w_norm"] if norm else None,
                             g["z"] if norm else None, synthetic.EPS, out=y, workspace=ws)
    torch.cuda.synchronize()


if __name__ == "__main__":
    main()
