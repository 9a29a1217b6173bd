"""ar_fusion_run_noalloc: the fused call for callers that may not allocate.

Some callers cannot call cudaMalloc: a plugin running inside a framework that
owns the whole device-memory budget (it sizes one pool at start-up and forbids
side allocations), or code on a latency-critical path where cudaMalloc /
cudaFree, which can synchronise the device, are not allowed.  For them the
library keeps the one-shot scratch (three slots and their state) in a fixed
device array and takes only inputs and outputs from the caller.

The GPU test calls the entry point through the C ABI twice in a row on fresh
inputs -- the second call uses the next scratch slot and depends on the first
call having cleaned up after itself -- and checks every output against the
workspace-based ar_fusion_run on the same inputs, under the same tolerances as
the other parity tests.  This file is collected last so that a run stopping at
the first failure has already run every other test; it also passes on its own
in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import parity as PY
from allreduce_residual_rmsnorm_gb300 import binding as B
from allreduce_residual_rmsnorm_gb300 import build as BUILD
from allreduce_residual_rmsnorm_gb300 import workloads as W


def _outputs(w, dev="cuda"):
    T, H = w.T, w.H
    pat = B.PATTERNS[w.pattern]
    dt = W.torch_dtype(w.dtype)
    out = {"residual": torch.full((T, H), float("nan"), dtype=dt, device=dev),
           "norm": torch.full((T, H), float("nan"), dtype=dt, device=dev),
           "quant": None, "sf": None}
    if pat & B.AR_QUANT_FP8:
        out["quant"] = torch.full((T, H), 0xAA, dtype=torch.uint8, device=dev)
    if pat & B.AR_QUANT_NVFP4:
        out["quant"] = torch.full((T, H // 2), 0xAA, dtype=torch.uint8, device=dev)
        out["sf"] = torch.full((T, H // 16), 0xAA, dtype=torch.uint8, device=dev)
    return out


def _host(out, pat):
    return {"residual": W.bits(out["residual"].cpu()) if pat & B.AR_RESIDUAL_OUT else None,
            "norm": W.bits(out["norm"].cpu()) if pat & B.AR_NORM_OUT else None,
            "quant": out["quant"].cpu().numpy() if out["quant"] is not None else None,
            "sf": out["sf"].cpu().numpy() if out["sf"] is not None else None}


CASES = [
    W.TINY,                                                             # 2 x 16 x 512
    W.FusedWorkload("noalloc_nvfp4", R=8, T=32, H=2048, pattern=W.RES_NORM_NVFP4, heavy_frac=0.01),
    W.FusedWorkload("noalloc_fp8", R=4, T=24, H=4096, pattern=W.RES_QUANT_FP8),
    W.FusedWorkload("noalloc_fp32_nvfp4", R=4, T=16, H=4096, dtype="fp32",
                    pattern=W.RES_NORM_NVFP4),                           # 1 MiB per slot
]


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_workspace_call_twice(w):
    B.load()
    L = B.lib()
    pat = B.PATTERNS[w.pattern]
    dtype = PY.BDT[w.dtype]
    ws = B.ar_fusion_workspace_create(w.R, w.T, w.H, dtype)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        inp = W.make_fused_inputs(w.with_(seed=1000 + call))
        P = inp.partials.cuda()
        X = inp.residual.cuda()
        G = inp.gamma.cuda()
        scale = torch.tensor([2688.0 / 6.0 if pat & B.AR_QUANT_NVFP4 else 64.0], device="cuda")
        ref = _outputs(w)
        B.ar_fusion_run(ws, [P[r] for r in range(w.R)], X, G, w.eps, pat, ref["residual"],
                        ref["norm"], ref["quant"], ref["sf"], scale)
        got = _outputs(w)
        parts = (ctypes.c_void_p * w.R)(*[P[r].data_ptr() for r in range(w.R)])

        def ptr(t):
            return None if t is None else t.data_ptr()

        rc = L.ar_fusion_run_noalloc(parts, w.R, w.T, w.H, dtype, X.data_ptr(),
                                     G.data_ptr(), ctypes.c_float(w.eps), pat,
                                     ptr(got["residual"]), ptr(got["norm"]), ptr(got["quant"]),
                                     ptr(got["sf"]), scale.data_ptr(), stream)
        assert rc == B.AR_OK, B.ar_fusion_last_error()
        torch.cuda.synchronize()
        exp_h, got_h = _host(ref, pat), _host(got, pat)
        if pat & B.AR_RESIDUAL_OUT:
            PY.assert_close16(got_h["residual"], exp_h["residual"], w.dtype,
                              f"residual (call {call})")
        if pat & B.AR_NORM_OUT:
            PY.assert_close16(got_h["norm"], exp_h["norm"], w.dtype, f"norm (call {call})")
        if pat & B.AR_QUANT_FP8:
            PY.assert_codes(got_h["quant"], exp_h["quant"], "e4m3", f"fp8 (call {call})")
        if pat & B.AR_QUANT_NVFP4:
            PY.assert_codes(got_h["sf"], exp_h["sf"], "e4m3", f"scales (call {call})")
            PY.assert_codes(got_h["quant"], exp_h["quant"], "e2m1", f"fp4 (call {call})")
    B.ar_fusion_workspace_destroy(ws)


def test_noalloc_rejects_sizes_beyond_the_scratch_before_any_cuda_call():
    BUILD.build()
    L = B.load()
    big = (ctypes.c_void_p * 8)(*([16] * 8))
    # 8 ranks x 128 tokens x 4096 x 2 bytes = 8 MiB > the 4 MiB slot
    rc = L.ar_fusion_run_noalloc(big, 8, 128, 4096, B.AR_DT_BF16, 16, 16, ctypes.c_float(1e-5),
                                 B.PATTERNS["res_norm"], 16, 16, None, None, None, None)
    assert rc == B.AR_ERR_CAPACITY
    assert "scratch" in B.ar_fusion_last_error()
    rc = L.ar_fusion_run_noalloc(big, 17, 1, 64, B.AR_DT_BF16, 16, 16, ctypes.c_float(1e-5),
                                 B.PATTERNS["res_norm"], 16, 16, None, None, None, None)
    assert rc == B.AR_ERR_UNSUPPORTED
    # fp32 elements count 4 bytes: 8 x 64 x 4096 x 4 = 8 MiB
    rc = L.ar_fusion_run_noalloc(big, 8, 64, 4096, B.AR_DT_FP32, 32, 32, ctypes.c_float(1e-5),
                                 B.PATTERNS["res_norm"], 32, 32, None, None, None, None)
    assert rc == B.AR_ERR_CAPACITY
    assert np.int64(B.AR_NOALLOC_SLOT_BYTES) == 4 << 20
