"""Seeded random configurations of the fused call against the oracle: ranks,
tokens, hidden size, element type, output pattern, kernel variant, staged or
caller partials, accumulation, NVFP4 scale layout, clusters and PDL drawn
together, so that combinations no hand-written case names are exercised."""
import random

import numpy as np
import pytest
import torch

import oracle
import parity as PY
from allreduce_residual_rmsnorm_gb300 import binding as B
from allreduce_residual_rmsnorm_gb300 import workloads as W
from test_parity_gpu import make_ws

PATTERNS = [W.RES_NORM, W.NORM, W.RES_QUANT_FP8, W.RES_QUANT_NVFP4, W.RES_NORM_FP8,
            W.RES_NORM_NVFP4]
VARIANTS = [B.AR_VARIANT_AUTO, B.AR_VARIANT_WARP_ROW, B.AR_VARIANT_CTA_ROW, B.AR_VARIANT_BULK_PIPE]


def draw(seed):
    rng = random.Random(seed)
    R = rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16])
    H = 16 * rng.choice([1, 3, 32, 40, 64, 65, 256, 448, 449, 512, 513, 640, 1024, 2048])
    T = rng.choice([1, 2, 7, 31, 64, 128, 129, 200, 333])
    while R * T * H > 3_000_000 and T > 1:
        T //= 2
    return dict(R=R, T=T, H=H, dtype=rng.choice(["bf16", "fp16", "fp32"]),
                pattern=rng.choice(PATTERNS), variant=rng.choice(VARIANTS),
                staged=rng.random() < 0.5, acc=rng.random() < 0.2,
                swizzled=rng.random() < 0.3, cluster=rng.choice([0, 0, 0, 2, 4]),
                pdl=int(rng.random() < 0.3), heavy=rng.random() < 0.3, seed=seed)


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(100))
def test_random_configuration_matches_oracle(seed):
    c = draw(seed)
    w = W.FusedWorkload(f"fuzz{seed}", R=c["R"], T=c["T"], H=c["H"], dtype=c["dtype"],
                        pattern=c["pattern"], heavy_frac=0.01 if c["heavy"] else 0.0,
                        eps=1e-5, seed=seed)
    acc = B.AR_ACC_ELEMENT if (c["acc"] and c["dtype"] != "fp32") else B.AR_ACC_FP32
    inp = W.make_fused_inputs(w)
    lam = c["staged"] and w.T <= B.AR_ONESHOT_MAX_TOKENS
    exp = PY.oracle_expected(w, inp, lamport_flip=lam, acc=acc)
    ws = make_ws(w)
    B.ar_fusion_workspace_set_variant(ws, c["variant"])
    B.ar_fusion_workspace_set_launch(ws, c["cluster"], c["pdl"])
    B.ar_fusion_workspace_set_accumulate(ws, acc)
    pat = B.PATTERNS[w.pattern]
    swz = c["swizzled"] and bool(pat & B.AR_QUANT_NVFP4)
    if swz:
        B.ar_fusion_workspace_set_scale_layout(ws, B.AR_SF_SWIZZLED)
    dev = "cuda"
    P = inp.partials.to(dev)
    X, G = inp.residual.to(dev), inp.gamma.to(dev)
    res = torch.full((w.T, w.H), float("nan"), dtype=X.dtype, device=dev)
    nrm = torch.full((w.T, w.H), float("nan"), dtype=X.dtype, device=dev)
    q = sf = sc = None
    if pat & B.AR_QUANT_FP8:
        q = torch.full((w.T, w.H), 0xAA, dtype=torch.uint8, device=dev)
    if pat & B.AR_QUANT_NVFP4:
        q = torch.full((w.T, w.H // 2), 0xAA, dtype=torch.uint8, device=dev)
        # the tile layout's padding is not written: zeros, as in the oracle's copy
        n_sf = B.swizzled_scale_bytes(w.T, w.H) if swz else w.T * (w.H // 16)
        sf = torch.full((n_sf,), 0 if swz else 0xAA, dtype=torch.uint8, device=dev)
    if q is not None:
        sc = torch.tensor([exp["scale"]], dtype=torch.float32, device=dev)
    if c["staged"]:
        for r in range(w.R):
            B.ar_fusion_workspace_stage(ws, r, P[r])
        parts = None
    else:
        parts = [P[r] for r in range(w.R)]
    B.ar_fusion_run(ws, parts, X, G, w.eps, pat, residual_out=res, norm_out=nrm, quant_out=q,
                    scale_out=sf, scale_factor=sc)
    torch.cuda.synchronize()
    rc, detail = B.ar_fusion_workspace_status(ws)
    assert rc == 0, (c, rc, detail)
    got = {"residual": W.bits(res.cpu()) if pat & B.AR_RESIDUAL_OUT else None,
           "norm": W.bits(nrm.cpu()) if pat & B.AR_NORM_OUT else None}
    if q is not None:
        got["quant"] = q.cpu().numpy()
    if sf is not None:
        got["sf"] = sf.cpu().numpy()
        if swz:
            exp = dict(exp, sf=oracle.swizzle_scales(exp["sf"]))
        else:
            got["sf"] = got["sf"].reshape(w.T, w.H // 16)
    stats = PY.check_all(w, got, exp)
    assert stats.get("residual_mismatch", 0) == 0, (c, stats)
    assert stats.get("norm_mismatch", 0) <= max(1, w.T * w.H // 1000), (c, stats)
    B.ar_fusion_workspace_destroy(ws)


def test_draws_cover_the_space():
    cs = [draw(s) for s in range(100)]
    assert {c["dtype"] for c in cs} == {"bf16", "fp16", "fp32"}
    assert {c["variant"] for c in cs} == set(VARIANTS)
    assert {c["pattern"] for c in cs} == set(PATTERNS)
    assert any(c["staged"] and c["T"] <= 128 for c in cs)
    assert any(c["swizzled"] and "nvfp4" in c["pattern"] for c in cs)
    assert np.mean([c["cluster"] > 0 for c in cs]) > 0.1
