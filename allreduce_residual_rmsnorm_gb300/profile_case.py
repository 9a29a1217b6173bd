"""Run one kernel variant on one synthetic workload, for profiler captures.

    python -m allreduce_residual_rmsnorm_gb300.profile_case --variant cta \
        --ranks 8 --tokens 2048 --hidden 7168 --pattern res_nvfp4 --iters 5

Inputs are seeded and generated on the CPU (workloads.py), staged once into
the workspace buffer region (Lamport slots when --lamport), then the fused
call (or the plain R-way sum with --sum N) runs --iters times.  Prints the
average device time per call (CUDA events) -- under a profiler that number is
not a measurement.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main(argv=None):
    import torch

    from allreduce_residual_rmsnorm_gb300 import binding as B
    from allreduce_residual_rmsnorm_gb300 import build as BUILD
    from allreduce_residual_rmsnorm_gb300 import workloads as W

    p = argparse.ArgumentParser()
    p.add_argument("--variant", default="auto", choices=["auto", "warp", "cta", "pipe"])
    p.add_argument("--ranks", type=int, default=8)
    p.add_argument("--tokens", type=int, default=2048)
    p.add_argument("--hidden", type=int, default=7168)
    p.add_argument("--pattern", default="res_nvfp4", choices=sorted(B.PATTERNS))
    p.add_argument("--dtype", default="bf16", choices=["bf16", "fp16", "fp32"])
    p.add_argument("--cluster", type=int, default=0)
    p.add_argument("--pdl", type=int, default=0)
    p.add_argument("--lamport", action="store_true")
    p.add_argument("--sum", type=int, default=0, help="plain R-way fp16 sum of N elements instead")
    p.add_argument("--iters", type=int, default=5)
    a = p.parse_args(argv)

    BUILD.build()
    B.load()
    dev = torch.device("cuda", 0)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if a.sum:
        x = W.make_sum_inputs(W.SumWorkload("s", R=a.ranks, N=a.sum)).to(dev)
        out = torch.empty(a.sum, dtype=torch.float16, device=dev)
        bufs = [x[r] for r in range(a.ranks)]
        B.ar_fusion_sum(bufs, out)
        ev0.record()
        for _ in range(a.iters):
            B.ar_fusion_sum(bufs, out)
        ev1.record()
        ev1.synchronize()
        print(f"sum R={a.ranks} N={a.sum}: {ev0.elapsed_time(ev1) * 1e3 / a.iters:.1f} us/call")
        return
    w = W.FusedWorkload("case", R=a.ranks, T=a.tokens, H=a.hidden, dtype=a.dtype,
                        pattern=a.pattern, heavy_frac=0.01)
    inp = W.make_fused_inputs(w)
    dt = {"bf16": B.AR_DT_BF16, "fp16": B.AR_DT_FP16, "fp32": B.AR_DT_FP32}[a.dtype]
    P, X, G = inp.partials.to(dev), inp.residual.to(dev), inp.gamma.to(dev)
    ws = B.ar_fusion_workspace_create(w.R, w.T, w.H, dt)
    B.ar_fusion_workspace_set_variant(ws, {"auto": B.AR_VARIANT_AUTO, "warp": B.AR_VARIANT_WARP_ROW,
                                           "cta": B.AR_VARIANT_CTA_ROW,
                                           "pipe": B.AR_VARIANT_BULK_PIPE}[a.variant])
    B.ar_fusion_workspace_set_launch(ws, a.cluster, a.pdl)
    mode = B.AR_MODE_LAMPORT if a.lamport else B.AR_MODE_BUFFER
    B.ar_fusion_workspace_set_mode(ws, mode)
    pat = B.PATTERNS[a.pattern]
    res, nrm = torch.empty_like(X), torch.empty_like(X)
    q = sf = sc = None
    if pat & B.AR_QUANT_FP8:
        q = torch.empty(w.T, w.H, dtype=torch.uint8, device=dev)
    if pat & B.AR_QUANT_NVFP4:
        q = torch.empty(w.T, w.H // 2, dtype=torch.uint8, device=dev)
        sf = torch.empty(w.T, w.H // 16, dtype=torch.uint8, device=dev)
    if q is not None:
        sc = torch.tensor([1.0], device=dev)

    def stage():
        for r in range(w.R):
            B.ar_fusion_workspace_stage(ws, r, P[r], mode=mode)

    stage()
    B.ar_fusion_run(ws, None, X, G, w.eps, pat, res, nrm, q, sf, sc)   # untimed: module load
    torch.cuda.synchronize()
    total = 0.0
    for _ in range(a.iters):
        if a.lamport:
            stage()
        ev0.record()
        B.ar_fusion_run(ws, None, X, G, w.eps, pat, res, nrm, q, sf, sc)
        ev1.record()
        ev1.synchronize()
        total += ev0.elapsed_time(ev1)
    rc, detail = B.ar_fusion_workspace_status(ws)
    last = B.ar_fusion_workspace_info(ws)["last_variant"]
    print(f"R={w.R} T={w.T} H={w.H} {a.pattern} variant={last} status={rc}: "
          f"{total * 1e3 / a.iters:.1f} us/call")
    B.ar_fusion_workspace_destroy(ws)
    if rc != 0:
        raise SystemExit(f"device status {rc} (detail {detail})")


if __name__ == "__main__":
    main()
