"""ar_fusion_run_noalloc: the fused call for callers that may not allocate.

Some callers cannot call cudaMalloc: a plugin running inside a framework that
owns the whole device-memory budget (it sizes one pool at start-up and forbids
side allocations), or code on a latency-critical path where cudaMalloc /
cudaFree, which can synchronise the device, are not allowed.  For them the
library keeps the one-shot scratch (three slots and their state) in a fixed
device array and takes only inputs and outputs from the caller.

The GPU tests call the entry point through the C ABI:
  - twice in a row on fresh inputs per case (the second call uses the next
    scratch slot and depends on the first call having cleaned up after
    itself), every output checked against the CPU oracle and against the
    workspace-based ar_fusion_run on the same inputs, under the same
    tolerances as the other parity tests;
  - in a sequence that changes element type, rank count and size from one
    call to the next on one stream (a bf16 call filling a whole slot followed
    by fp32 calls is the case where the retired slot's clear must use the
    previous call's element size), run twice; free device memory must not
    change during the second pass, and the status query must report no
    device-side error.
This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
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


def _ptr(t):
    return None if t is None else t.data_ptr()


class _Call:
    """One no-allocation call: device inputs, outputs and the oracle's result,
    all prepared before any call runs."""

    def __init__(self, w):
        self.w = w
        self.pat = B.PATTERNS[w.pattern]
        self.dtype = PY.BDT[w.dtype]
        self.inp = W.make_fused_inputs(w)
        # the one-shot path stages with the sentinel flip: the oracle sees it too
        self.exp = PY.oracle_expected(w, self.inp, lamport_flip=True)
        self.P = self.inp.partials.cuda()
        self.X = self.inp.residual.cuda()
        self.G = self.inp.gamma.cuda()
        s = self.exp.get("scale", 1.0)
        self.scale = torch.tensor([float(s)], dtype=torch.float32, device="cuda")
        self.got = _outputs(w)
        self.parts = (ctypes.c_void_p * w.R)(*[self.P[r].data_ptr() for r in range(w.R)])

    def run_noalloc(self, stream):
        w, g = self.w, self.got
        rc = B.lib().ar_fusion_run_noalloc(self.parts, w.R, w.T, w.H, self.dtype,
                                           self.X.data_ptr(), self.G.data_ptr(),
                                           ctypes.c_float(w.eps), self.pat, _ptr(g["residual"]),
                                           _ptr(g["norm"]), _ptr(g["quant"]), _ptr(g["sf"]),
                                           self.scale.data_ptr(), stream)
        assert rc == B.AR_OK, B.ar_fusion_last_error()

    def run_workspace(self):
        w = self.w
        ws = B.ar_fusion_workspace_create(w.R, w.T, w.H, self.dtype)
        ref = _outputs(w)
        B.ar_fusion_run(ws, [self.P[r] for r in range(w.R)], self.X, self.G, w.eps, self.pat,
                        ref["residual"], ref["norm"], ref["quant"], ref["sf"], self.scale)
        torch.cuda.synchronize()
        B.ar_fusion_workspace_destroy(ws)
        return _host(ref, self.pat)

    def check(self, what, against_workspace=True):
        got = _host(self.got, self.pat)
        PY.check_all(self.w, got, self.exp)
        if against_workspace:
            ref = self.run_workspace()
            for k in ("residual", "norm", "quant", "sf"):
                if got[k] is not None:
                    assert np.array_equal(got[k], ref[k]), \
                        f"{self.w.name} {what}: {k} differs from ar_fusion_run"


CASES = [
    W.TINY,                                                             # 2 x 16 x 512
    W.FusedWorkload("noalloc_nvfp4", R=8, T=32, H=2048, pattern=W.RES_NORM_NVFP4, heavy_frac=0.01),
    W.FusedWorkload("noalloc_fp8", R=4, T=24, H=4096, pattern=W.RES_QUANT_FP8),
    W.FusedWorkload("noalloc_fp32_nvfp4", R=4, T=16, H=4096, dtype="fp32",
                    pattern=W.RES_NORM_NVFP4),                           # 1 MiB per slot
]


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_oracle_and_workspace_call_twice(w):
    B.load()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        c = _Call(w.with_(seed=1000 + call))
        c.run_noalloc(stream)
        torch.cuda.synchronize()
        c.check(f"call {call}")
    assert B.ar_fusion_noalloc_status() == (B.AR_OK, -1)


# Consecutive calls change element type, ranks and size.  Slot bytes per call
# (R * T * H * element size): 4 MiB (the whole slot), 1 MiB, 256 KiB, 4 MiB,
# 32 KiB, 2 MiB.
MIXED = [
    W.FusedWorkload("mix_bf16_full_slot", R=8, T=128, H=2048, pattern=W.RES_NORM),
    W.FusedWorkload("mix_fp32_nvfp4", R=4, T=16, H=4096, dtype="fp32", pattern=W.RES_NORM_NVFP4),
    W.FusedWorkload("mix_fp16_fp8", R=2, T=64, H=1024, dtype="fp16", pattern=W.RES_QUANT_FP8),
    W.FusedWorkload("mix_fp32_full_slot", R=8, T=32, H=4096, dtype="fp32", pattern=W.RES_NORM),
    W.FusedWorkload("mix_bf16_tiny", R=2, T=16, H=512, pattern=W.NORM),
    W.FusedWorkload("mix_fp16_r16_nvfp4", R=16, T=8, H=8192, dtype="fp16",
                    pattern=W.RES_QUANT_NVFP4, heavy_frac=0.01),
]


def test_mixed_sequence_fits_the_scratch_slots():
    for w in MIXED:
        eb = 4 if w.dtype == "fp32" else 2
        assert w.R * w.T * w.H * eb <= B.AR_NOALLOC_SLOT_BYTES, w.name
    assert MIXED[0].R * MIXED[0].T * MIXED[0].H * 2 == B.AR_NOALLOC_SLOT_BYTES
    assert MIXED[1].dtype == "fp32" and MIXED[0].dtype == "bf16"


@pytest.mark.gpu
def test_noalloc_mixed_sequence_allocates_nothing_and_reports_no_error():
    B.load()
    stream = torch.cuda.current_stream().cuda_stream
    calls = [_Call(w.with_(seed=2000 + i)) for i, w in enumerate(MIXED)]
    torch.cuda.synchronize()
    # first pass: set-up (on a fresh process) and every kernel loaded
    for c in calls:
        c.run_noalloc(stream)
    torch.cuda.synchronize()
    for c in calls:
        c.check("first pass", against_workspace=False)
        for t in c.got.values():
            if t is not None:
                t.fill_(0x55 if t.dtype == torch.uint8 else float("nan"))
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for c in calls:
        c.run_noalloc(stream)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert B.ar_fusion_noalloc_status() == (B.AR_OK, -1)
    assert B.ar_fusion_noalloc_status() == (B.AR_OK, -1)
    for c in calls:
        c.check("second pass", against_workspace=True)


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
