"""Helpers shared by the GPU parity tests: run a workload through the C ABI
and through the CPU oracle, and compare under the stated tolerances.

Tolerances (per element): |g - o| <= atol + rtol * |o| with (2e-2, 1e-2) for
bf16, (5e-3, 5e-3) for fp16 and (1e-5, 1e-5) for fp32.  The same two numbers
also bound, separately, the maximum absolute error and the maximum relative
error of each output (the relative one over expected values in the normal
range of the element type: a subnormal value's last bit is a large fraction
of it).  Quantised codes must be bit-exact except that at most 0.1% may
differ by one code step.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from allreduce_residual_rmsnorm_gb300 import binding as B
from allreduce_residual_rmsnorm_gb300 import workloads as W

TOL = {"bf16": (2e-2, 1e-2), "fp16": (5e-3, 5e-3), "fp32": (1e-5, 1e-5)}
ODT = {"bf16": oracle.BF16, "fp16": oracle.FP16}
BDT = {"bf16": B.AR_DT_BF16, "fp16": B.AR_DT_FP16, "fp32": B.AR_DT_FP32}


def to_float(bits16: np.ndarray, dtype: str) -> np.ndarray:
    return W.from_bits(bits16, dtype).float().numpy()


def oracle_expected_f32(w: W.FusedWorkload, inp: W.FusedInputs, lamport_flip: bool = False):
    """oracle_expected for fp32 elements (residual / norm as uint32 bits)."""
    P = inp.partials.numpy()
    if lamport_flip:
        P = oracle.lamport_flip(P.view(np.uint16)).view(np.float32)
    res, nrm, rstd = oracle.fused_f32(P, inp.residual.numpy(), inp.gamma.numpy(), inp.eps)
    out = {"residual": res.view(np.uint32), "norm": nrm.view(np.uint32), "rstd": rstd}
    pat = B.PATTERNS[w.pattern]
    if pat & (B.AR_QUANT_FP8 | B.AR_QUANT_NVFP4):
        amax = oracle.amax_f32(nrm)
        out["amax"] = amax
        if pat & B.AR_QUANT_FP8:
            out["scale"] = oracle.fp8_inv_scale(amax)
            out["quant"] = oracle.quant_fp8_f32(nrm, out["scale"])
        else:
            out["scale"] = oracle.nvfp4_global_scale(amax)
            out["quant"], out["sf"] = oracle.quant_nvfp4_f32(nrm, out["scale"])
    return out


def oracle_expected(w: W.FusedWorkload, inp: W.FusedInputs, lamport_flip: bool = False,
                    acc: int = 0):
    """Oracle outputs for the workload: dict with residual, norm, amax and,
    when quantised, the scale passed to both sides and the codes."""
    if w.dtype == "fp32":
        return oracle_expected_f32(w, inp, lamport_flip)
    odt = ODT[w.dtype]
    P = W.bits(inp.partials)
    if lamport_flip:
        P = oracle.lamport_flip(P)
    res, nrm, rstd = oracle.fused(odt, P, W.bits(inp.residual), W.bits(inp.gamma), inp.eps,
                                  acc=acc)
    out = {"residual": res, "norm": nrm, "rstd": rstd}
    pat = B.PATTERNS[w.pattern]
    if pat & (B.AR_QUANT_FP8 | B.AR_QUANT_NVFP4):
        amax = oracle.amax(odt, nrm)
        out["amax"] = amax
        if pat & B.AR_QUANT_FP8:
            out["scale"] = oracle.fp8_inv_scale(amax)
            out["quant"] = oracle.quant_fp8(odt, nrm, out["scale"])
        else:
            out["scale"] = oracle.nvfp4_global_scale(amax)
            out["quant"], out["sf"] = oracle.quant_nvfp4(odt, nrm, out["scale"])
    return out


def run_gpu(ws, w: W.FusedWorkload, inp: W.FusedInputs, scale: float | None = None,
            staged: bool = False, pattern: int | None = None, dev="cuda"):
    """Run the fused call; returns dict of host numpy outputs."""
    pat = B.PATTERNS[w.pattern] if pattern is None else pattern
    P = inp.partials.to(dev)
    X = inp.residual.to(dev)
    G = inp.gamma.to(dev)
    T, H = w.T, w.H
    res = torch.full((T, H), float("nan"), dtype=X.dtype, device=dev)
    nrm = torch.full((T, H), float("nan"), dtype=X.dtype, device=dev)
    quant = sf = sc = None
    if pat & B.AR_QUANT_FP8:
        quant = torch.full((T, H), 0xAA, dtype=torch.uint8, device=dev)
    if pat & B.AR_QUANT_NVFP4:
        quant = torch.full((T, H // 2), 0xAA, dtype=torch.uint8, device=dev)
        sf = torch.full((T, max(H // 16, 1)), 0xAA, dtype=torch.uint8, device=dev)
    if pat & (B.AR_QUANT_FP8 | B.AR_QUANT_NVFP4):
        sc = torch.tensor([scale], dtype=torch.float32, device=dev)
    if staged:
        for r in range(w.R):
            B.ar_fusion_workspace_stage(ws, r, P[r])
        parts = None
    else:
        parts = [P[r] for r in range(w.R)]
    B.ar_fusion_run(ws, parts, X, G, inp.eps, pat, residual_out=res, norm_out=nrm,
                    quant_out=quant, scale_out=sf, scale_factor=sc)
    torch.cuda.synchronize()
    out = {"residual": W.bits(res.cpu()) if pat & B.AR_RESIDUAL_OUT else None,
           "norm": W.bits(nrm.cpu()) if pat & B.AR_NORM_OUT else None}
    if quant is not None:
        out["quant"] = quant.cpu().numpy()
    if sf is not None:
        out["sf"] = sf.cpu().numpy()
    return out


MIN_NORMAL = {"bf16": 2.0 ** -126, "fp16": 2.0 ** -14, "fp32": 2.0 ** -126}


def error_stats(got_bits, exp_bits, dtype: str):
    """(max abs error, max rel error over normal-range expected values)."""
    g = to_float(got_bits, dtype).astype(np.float64)
    o = to_float(exp_bits, dtype).astype(np.float64)
    err = np.abs(g - o)
    err[np.isnan(g) & np.isnan(o)] = 0.0
    nrm = np.abs(o) >= MIN_NORMAL[dtype]
    rel = err[nrm] / np.abs(o[nrm])
    return float(np.max(err, initial=0.0)), float(np.max(rel, initial=0.0))


def assert_close16(got_bits, exp_bits, dtype: str, what: str, require_exact_frac: float = 0.0,
                   errors: dict | None = None):
    atol, rtol = TOL[dtype]
    g = to_float(got_bits, dtype)
    o = to_float(exp_bits, dtype)
    err = np.abs(g - o)
    bad = ~(err <= atol + rtol * np.abs(o))
    assert not bad.any(), (f"{what}: {bad.sum()} elements outside tolerance; max abs err "
                           f"{np.nanmax(err)} at {np.argwhere(bad)[:5].tolist()}")
    max_abs, max_rel = error_stats(got_bits, exp_bits, dtype)
    assert max_abs <= atol, f"{what}: max abs error {max_abs} > {atol}"
    assert max_rel <= rtol, f"{what}: max rel error {max_rel} > {rtol}"
    if errors is not None:
        errors[what] = {"max_abs_err": max_abs, "max_rel_err": max_rel}
    mism = np.count_nonzero(got_bits != exp_bits)
    return mism


def e4m3_step(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Code distance of E4M3 bytes (0x00 and 0x80 are the same value)."""
    def key(c):
        c = c.astype(np.int32)
        m = c & 0x7f
        return np.where(c & 0x80, -m, m)
    return np.abs(key(a) - key(b))


def e2m1_step(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def key(c):
        c = c.astype(np.int32)
        m = c & 0x7
        return np.where(c & 0x8, -m, m)
    return np.abs(key(a) - key(b))


def assert_codes(got: np.ndarray, exp: np.ndarray, kind: str, what: str):
    if kind == "e4m3":
        d = e4m3_step(got, exp)
    else:  # packed e2m1 pairs
        d = np.maximum(e2m1_step(got & 0xf, exp & 0xf), e2m1_step(got >> 4, exp >> 4))
    n_off = np.count_nonzero(d)
    assert d.max(initial=0) <= 1, f"{what}: code differs by {d.max()} steps"
    assert n_off <= max(0, int(0.001 * d.size)), f"{what}: {n_off} of {d.size} codes differ"
    return n_off


def check_all(w: W.FusedWorkload, got: dict, exp: dict):
    """Apply every rule; returns a dict of mismatch counts (for reporting)."""
    stats = {}
    errs = {}
    pat = B.PATTERNS[w.pattern]
    if pat & B.AR_RESIDUAL_OUT:
        stats["residual_mismatch"] = assert_close16(got["residual"], exp["residual"], w.dtype,
                                                    "residual_out", errors=errs)
    if pat & B.AR_NORM_OUT:
        stats["norm_mismatch"] = assert_close16(got["norm"], exp["norm"], w.dtype, "norm_out",
                                                errors=errs)
    stats["errors"] = errs
    if pat & B.AR_QUANT_FP8:
        stats["fp8_off"] = assert_codes(got["quant"], exp["quant"], "e4m3", "fp8 codes")
    if pat & B.AR_QUANT_NVFP4:
        stats["sf_off"] = assert_codes(got["sf"], exp["sf"], "e4m3", "nvfp4 scales")
        stats["fp4_off"] = assert_codes(got["quant"], exp["quant"], "e2m1", "nvfp4 codes")
    return stats
