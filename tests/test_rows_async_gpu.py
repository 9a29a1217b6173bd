"""GPU parity of the row kernel that copies each thread's next-row vectors into
shared memory (AR_VARIANT_CTA_ROW_ASYNC) against the CPU oracle: rank counts
1-8, ragged and one-vector rows, more rows than blocks, every output pattern,
staged buffer and caller partials, element-type accumulation, the calibration
pass, and the fallback to AUTO's choice where the kernel does not apply."""
import pytest
import torch

import parity as PY
from allreduce_residual_rmsnorm_gb300 import binding as B
from allreduce_residual_rmsnorm_gb300 import workloads as W
from test_parity_gpu import make_ws

pytestmark = pytest.mark.gpu


def run_async(w, staged, acc=B.AR_ACC_FP32, mode=B.AR_MODE_BUFFER):
    inp = W.make_fused_inputs(w)
    ws = make_ws(w)
    B.ar_fusion_workspace_set_variant(ws, B.AR_VARIANT_CTA_ROW_ASYNC)
    B.ar_fusion_workspace_set_mode(ws, mode)
    B.ar_fusion_workspace_set_accumulate(ws, acc)
    lam = staged and (mode == B.AR_MODE_LAMPORT or
                      (mode == B.AR_MODE_AUTO and w.T <= B.AR_ONESHOT_MAX_TOKENS))
    exp = PY.oracle_expected(w, inp, lamport_flip=lam, acc=acc)
    got = PY.run_gpu(ws, w, inp, scale=exp.get("scale"), staged=staged)
    rc, detail = B.ar_fusion_workspace_status(ws)
    assert rc == 0, (rc, detail)
    last = B.ar_fusion_workspace_info(ws)["last_variant"]
    stats = PY.check_all(w, got, exp)
    B.ar_fusion_workspace_destroy(ws)
    return stats, last


CASES = [
    # (R, T, H, dtype, pattern, staged)
    (1, 1, 8, "bf16", W.RES_NORM, False),
    (2, 7, 24, "fp16", W.NORM, True),
    (3, 5, 16, "bf16", W.RES_QUANT_NVFP4, False),
    (3, 300, 4096, "bf16", W.RES_NORM_FP8, True),
    (4, 333, 8192, "bf16", W.RES_NORM_FP8, True),
    (4, 200, 8184, "fp16", W.RES_NORM, False),
    (5, 200, 7168, "fp16", W.RES_QUANT_NVFP4, False),
    (6, 153, 6160, "bf16", W.RES_NORM_NVFP4, True),
    (7, 160, 1000, "bf16", W.RES_NORM, False),
    (8, 400, 7168, "bf16", W.RES_QUANT_NVFP4, True),
    (8, 333, 6152, "bf16", W.RES_NORM, True),
    (8, 152, 7168, "fp16", W.RES_NORM_FP8, False),
]


@pytest.mark.parametrize("R,T,H,dtype,pattern,staged", CASES)
def test_async_rows_match_oracle(R, T, H, dtype, pattern, staged):
    w = W.FusedWorkload(f"async_r{R}_t{T}_h{H}", R=R, T=T, H=H, dtype=dtype, pattern=pattern,
                        heavy_frac=0.01 if R == 8 else 0.0, eps=1e-5, seed=R * 7 + T)
    stats, last = run_async(w, staged)
    assert last == B.AR_VARIANT_CTA_ROW_ASYNC
    assert stats.get("residual_mismatch", 0) == 0, stats
    assert stats.get("norm_mismatch", 0) <= max(1, w.T * w.H // 100000), stats


def test_async_rows_full_fp8_configuration():
    # 4 ranks x 2048 tokens x hidden 8192, residual + norm + FP8 (1024 threads)
    stats, last = run_async(W.FP8_PREFILL, staged=True)
    assert last == B.AR_VARIANT_CTA_ROW_ASYNC
    assert stats["residual_mismatch"] == 0, stats
    assert stats["norm_mismatch"] <= 0.00001 * W.FP8_PREFILL.T * W.FP8_PREFILL.H, stats


def test_async_rows_full_nvfp4_configuration():
    # 8 ranks x 8192 tokens x hidden 7168, residual + NVFP4 (896 threads)
    stats, last = run_async(W.NVFP4_PREFILL, staged=True)
    assert last == B.AR_VARIANT_CTA_ROW_ASYNC
    assert stats["residual_mismatch"] == 0, stats


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_async_rows_element_type_accumulation(dtype):
    w = W.FusedWorkload(f"async_acc_{dtype}", R=6, T=300, H=3072, dtype=dtype,
                        pattern=W.RES_NORM_FP8, seed=11)
    stats, last = run_async(w, staged=False, acc=B.AR_ACC_ELEMENT)
    assert last == B.AR_VARIANT_CTA_ROW_ASYNC
    assert stats.get("residual_mismatch", 0) == 0, stats
    assert stats.get("norm_mismatch", 0) <= max(1, w.T * w.H // 100000), stats


def test_calibration_pass_with_the_async_variant_set():
    # the calibration pass runs the plain row kernel whatever the variant
    # setting; the setting must not change its result
    w = W.FP8_PREFILL.with_(T=256, seed=3)
    inp = W.make_fused_inputs(w)
    exp = PY.oracle_expected(w, inp)
    ws = make_ws(w)
    B.ar_fusion_workspace_set_variant(ws, B.AR_VARIANT_CTA_ROW_ASYNC)
    P = inp.partials.cuda()
    amax = torch.full((1,), -1.0, device="cuda")
    B.ar_fusion_norm_amax(ws, [P[r] for r in range(w.R)], inp.residual.cuda(), inp.gamma.cuda(),
                          w.eps, amax)
    torch.cuda.synchronize()
    assert float(amax.item()) == exp["amax"]
    B.ar_fusion_workspace_destroy(ws)


@pytest.mark.parametrize("R,T,H,dtype,mode,staged", [
    (8, 64, 4096, "bf16", B.AR_MODE_AUTO, True),      # Lamport slots
    (12, 40, 2048, "bf16", B.AR_MODE_BUFFER, False),  # more than 8 ranks
    (4, 40, 9216, "bf16", B.AR_MODE_BUFFER, False),   # more than one vector per thread
    (8, 40, 2048, "fp32", B.AR_MODE_BUFFER, False),   # fp32 elements
])
def test_async_rows_fall_back_where_they_do_not_apply(R, T, H, dtype, mode, staged):
    w = W.FusedWorkload(f"async_fb_r{R}_h{H}", R=R, T=T, H=H, dtype=dtype, pattern=W.RES_NORM)
    stats, last = run_async(w, staged, mode=mode)
    assert last != B.AR_VARIANT_CTA_ROW_ASYNC
    assert stats.get("residual_mismatch", 0) == 0, stats
    assert stats.get("norm_mismatch", 0) <= max(1, w.T * w.H // 100000), stats
