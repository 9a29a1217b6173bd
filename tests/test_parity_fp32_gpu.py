"""GPU parity for fp32 elements (the 4-byte exchange type of FlashInfer's
use_fp32_lamport workspaces) against the fp32 oracle: the fused call in every
launch shape, the Lamport slots, the plain sum.  Tolerance |g - o| <= 1e-5 +
1e-5 |o|; the rank sum and residual add are plain fp32 additions in rank
order on both sides, so residual_out must be bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import parity as PY
from allreduce_residual_rmsnorm_gb300 import binding as B
from allreduce_residual_rmsnorm_gb300 import workloads as W
from test_parity_gpu import make_ws, run_and_check

pytestmark = pytest.mark.gpu


def _norm_budget(w):
    # the sum of squares is a double-float pair on the GPU and fp64 in the
    # oracle: a row whose sum sits next to an fp32 rounding boundary can give
    # an rstd one ulp apart, and then every element of that row may differ by
    # an ulp (well inside the tolerance)
    return max(1, w.T * w.H // 1000)


@pytest.mark.parametrize("staged", [False, True])
def test_fp32_decode_r8_t128_h4096(staged):
    w = W.FP32_DECODE
    stats, _, _ = run_and_check(w, B.AR_VARIANT_AUTO, staged)
    assert stats["residual_mismatch"] == 0, stats
    assert stats["norm_mismatch"] <= _norm_budget(w), stats


@pytest.mark.parametrize("variant,staged", [(B.AR_VARIANT_AUTO, True), (B.AR_VARIANT_CTA_ROW, False),
                                            (B.AR_VARIANT_BULK_PIPE, False)])
def test_fp32_prefill_r8_t1024_h7168_nvfp4(variant, staged):
    # hidden 7168 = 896 vectors of 8 fp32: AUTO splits the row over a 2-CTA
    # cluster; the row kernel alone takes two vectors per thread
    w = W.FP32_PREFILL
    stats, _, _ = run_and_check(w, variant, staged)
    assert stats["residual_mismatch"] == 0, stats
    assert stats["norm_mismatch"] <= _norm_budget(w), stats


EDGE32 = [
    # (R, T, H, pattern)
    (1, 1, 8, W.RES_NORM), (3, 5, 24, W.NORM), (5, 3, 16, W.RES_QUANT_NVFP4),
    (16, 7, 520, W.RES_NORM_FP8), (2, 37, 1000, W.RES_QUANT_FP8), (7, 9, 1024, W.RES_NORM_NVFP4),
    (4, 13, 4104, W.RES_NORM), (8, 33, 2048, W.RES_NORM), (6, 17, 7176, W.RES_NORM_FP8),
    (2, 3, 32768, W.RES_QUANT_NVFP4), (16, 2, 32768, W.RES_NORM), (8, 200, 4096, W.RES_NORM_NVFP4),
    (1, 500, 16384, W.RES_QUANT_FP8), (2, 3, 20480, W.RES_NORM_FP8), (3, 9, 10240, W.RES_NORM_NVFP4),
]


@pytest.mark.parametrize("R,T,H,pattern", EDGE32)
@pytest.mark.parametrize("variant", [B.AR_VARIANT_AUTO, B.AR_VARIANT_WARP_ROW, B.AR_VARIANT_CTA_ROW,
                                     B.AR_VARIANT_BULK_PIPE])
def test_fp32_edge_shapes(R, T, H, pattern, variant):
    w = W.FusedWorkload(f"edge32_{R}_{T}_{H}", R=R, T=T, H=H, dtype="fp32", pattern=pattern,
                        eps=1e-5, seed=R * 1000 + T + 7)
    stats, _, _ = run_and_check(w, variant)
    assert stats.get("residual_mismatch", 0) == 0, stats
    assert stats.get("norm_mismatch", 0) <= _norm_budget(w), stats


@pytest.mark.parametrize("cluster", [2, 4])
@pytest.mark.parametrize("staged,pdl", [(False, 0), (True, 1)])
def test_fp32_cluster_split_rows(cluster, staged, pdl):
    w = W.FusedWorkload("fp32_cluster", R=8, T=40, H=4096, dtype="fp32",
                        pattern=W.RES_NORM_NVFP4, seed=77)
    stats, _, _ = run_and_check(w, B.AR_VARIANT_CTA_ROW, staged, cluster=cluster, pdl=pdl)
    assert stats["residual_mismatch"] == 0, stats
    assert stats["norm_mismatch"] <= _norm_budget(w), stats


def test_fp32_lamport_sequence_clears_retired_slot():
    w = W.FusedWorkload("fp32_lamport", R=4, T=16, H=1024, dtype="fp32", pattern=W.RES_NORM)
    ws = make_ws(w, mem=True)
    info = B.ar_fusion_workspace_info(ws)
    assert info["elem_bytes"] == 4
    assert info["lamport_comm_bytes"] == w.R * B.AR_ONESHOT_MAX_TOKENS * w.H * 4
    mem = ws.mem
    slot_b = info["lamport_comm_bytes"]
    lam_off = info["lamport"] - info["base"]
    flag = clear = 0
    for k in range(5):
        wk = w.with_(seed=300 + k, T=w.T - (k % 3))
        inp = W.make_fused_inputs(wk)
        exp = PY.oracle_expected(wk, inp, lamport_flip=True)
        got = PY.run_gpu(ws, wk, inp, staged=True)
        PY.check_all(wk, got, exp)
        assert np.array_equal(got["residual"], exp["residual"])
        st = B.ar_fusion_workspace_copy_state(ws)
        new_flag, new_clear, _, cl = oracle.lamport_step(flag, clear, wk.R, wk.T, wk.H)
        assert st["lamport_flag"] == new_flag and st["clear_size"] == new_clear
        assert st["calls"] == k + 1 and st["status"] == 0
        # clear_size counts elements: 4 bytes each here
        words = mem[lam_off + cl * slot_b: lam_off + cl * slot_b + clear * 4].view(torch.int32)
        assert bool((words == torch.tensor(-2 ** 31, dtype=torch.int32, device="cuda")).all())
        flag, clear = new_flag, new_clear
    B.ar_fusion_workspace_destroy(ws)


def test_fp32_negative_zero_partials_are_flipped_on_stage():
    # an fp32 -0.0 element is the sentinel word itself: staged into a Lamport
    # slot it becomes +0.0, which only changes the sign of an all-zero sum
    w = W.FusedWorkload("fp32_negzero", R=3, T=8, H=256, dtype="fp32", pattern=W.RES_NORM, seed=9)
    inp = W.make_fused_inputs(w)
    inp.partials[:, :, :16] = -0.0
    inp.residual[:, :8] = -0.0
    stats, got, exp = run_and_check(w, staged=True, inp=inp)
    assert stats["residual_mismatch"] == 0
    assert np.all(got["residual"].reshape(w.T, w.H)[:, :8] == 0)            # +0.0 words
    stats, got, _ = run_and_check(w, staged=False, inp=inp)
    assert stats["residual_mismatch"] == 0
    assert np.all(got["residual"].reshape(w.T, w.H)[:, :8] == 0x80000000)   # -0 + -0 = -0


def test_fp32_rejects_16_byte_aligned_pointers():
    w = W.FusedWorkload("fp32_align", R=2, T=4, H=64, dtype="fp32")
    ws = make_ws(w)
    big = torch.zeros(w.T * w.H + 8, device="cuda")
    X = big[4:4 + w.T * w.H].view(w.T, w.H)                  # 16 bytes past a 32-byte boundary
    G = torch.ones(w.H, device="cuda")
    P = [torch.zeros(w.T, w.H, device="cuda") for _ in range(w.R)]
    out = torch.empty(w.T, w.H, device="cuda")
    with pytest.raises(B.ArFusionError) as e:
        B.ar_fusion_run(ws, P, X, G, 1e-6, B.AR_NORM_OUT, norm_out=out)
    assert e.value.code == B.AR_ERR_INVALID
    with pytest.raises(B.ArFusionError) as e:
        B.ar_fusion_run(ws, [P[0], X], P[1], G, 1e-6, B.AR_NORM_OUT, norm_out=out)
    assert e.value.code == B.AR_ERR_INVALID
    B.ar_fusion_workspace_destroy(ws)


@pytest.mark.parametrize("R,N,offset", [(8, 1_000_003, 0), (3, 4099, 0), (16, 65536, 0),
                                        (5, 1001, 1), (2, 777, 4)])
def test_fp32_vector_sum(R, N, offset):
    g = torch.Generator().manual_seed(R * 7 + N)
    ins = (torch.rand(R, N + offset, generator=g) * 2 - 1)
    exp = oracle.vector_sum_f32(ins[:, offset:].numpy())
    dev = ins.cuda()
    out = torch.full((N + offset,), float("nan"), device="cuda")
    B.ar_fusion_sum([dev[r, offset:] for r in range(R)], out[offset:], n=N)
    torch.cuda.synchronize()
    assert np.array_equal(out[offset:].cpu().numpy().view(np.uint32), exp.view(np.uint32))
    # rounding to the element type after every add is the identity for fp32
    out.fill_(float("nan"))
    B.ar_fusion_sum_ex([dev[r, offset:] for r in range(R)], out[offset:], B.AR_ACC_ELEMENT, n=N)
    torch.cuda.synchronize()
    assert np.array_equal(out[offset:].cpu().numpy().view(np.uint32), exp.view(np.uint32))


@pytest.mark.parametrize("R,T,H,dtype,expect", [
    (8, 512, 16384, "bf16", B.AR_VARIANT_BULK_PIPE),    # two vectors per thread, 151 MB of inputs
    (16, 450, 7168, "bf16", B.AR_VARIANT_BULK_PIPE),    # 16 ranks of 14 KB rows, 110 MB
    (16, 400, 7168, "bf16", B.AR_VARIANT_CTA_ROW),      # 97.5 MB: below the 96 MiB threshold
    (16, 1024, 4096, "bf16", B.AR_VARIANT_CTA_ROW),     # 16 ranks of 8 KB rows
    (8, 1024, 7168, "bf16", B.AR_VARIANT_CTA_ROW),      # one vector per thread, 8 ranks
    (8, 512, 7168, "fp32", B.AR_VARIANT_BULK_PIPE),     # fp32: 896 vectors > 512 threads
    (8, 256, 7168, "fp32", B.AR_VARIANT_CTA_ROW),       # 66 MB
    (16, 512, 4096, "fp32", B.AR_VARIANT_BULK_PIPE),    # 16 ranks of 16 KB rows
    (4, 2048, 512, "bf16", B.AR_VARIANT_WARP_ROW),
    (2, 2048, 12288, "bf16", B.AR_VARIANT_CTA_ROW),     # two ranks: row kernel up to 2048 vectors
    (2, 1024, 20480, "bf16", B.AR_VARIANT_BULK_PIPE),   # beyond that the pipe
    (4, 1024, 12288, "bf16", B.AR_VARIANT_CTA_ROW),     # <= 4 ranks: row kernel up to 1536 vectors
    (4, 1024, 16384, "bf16", B.AR_VARIANT_BULK_PIPE),
    (2, 1024, 12288, "fp32", B.AR_VARIANT_BULK_PIPE),   # fp32: the pipe beyond 512 vectors
])
def test_automatic_variant_choice(R, T, H, dtype, expect):
    w = W.FusedWorkload(f"auto_{R}_{T}_{H}_{dtype}", R=R, T=T, H=H, dtype=dtype,
                        pattern=W.RES_NORM_NVFP4, seed=T + R)
    inp = W.make_fused_inputs(w)
    ws = make_ws(w)
    exp = PY.oracle_expected(w, inp)
    got = PY.run_gpu(ws, w, inp, scale=exp["scale"])
    stats = PY.check_all(w, got, exp)
    assert stats["residual_mismatch"] == 0, stats
    info = B.ar_fusion_workspace_info(ws)
    assert info["last_variant"] == expect
    assert info["last_cluster"] == 1
    B.ar_fusion_workspace_destroy(ws)


def test_fp32_norm_amax_matches_oracle():
    w = W.FusedWorkload("fp32_amax", R=4, T=96, H=2048, dtype="fp32", heavy_frac=0.01, seed=21,
                        pattern=W.RES_NORM_FP8)
    inp = W.make_fused_inputs(w)
    exp = PY.oracle_expected(w, inp)
    ws = make_ws(w)
    P = inp.partials.cuda()
    amax = torch.full((1,), -1.0, device="cuda")
    B.ar_fusion_norm_amax(ws, [P[r] for r in range(w.R)], inp.residual.cuda(), inp.gamma.cuda(),
                          w.eps, amax)
    torch.cuda.synchronize()
    assert float(amax.item()) == exp["amax"]
    B.ar_fusion_workspace_destroy(ws)


@pytest.mark.parametrize("variant", [B.AR_VARIANT_CTA_ROW, B.AR_VARIANT_BULK_PIPE])
def test_fp32_nvfp4_swizzled_scale_layout(variant):
    from test_parity_gpu import _run_nvfp4_swizzled
    w = W.FusedWorkload("fp32_swz", R=4, T=200, H=4096, dtype="fp32", pattern=W.RES_NORM_NVFP4,
                        heavy_frac=0.01, seed=33)
    exp, q, sf = _run_nvfp4_swizzled(w, variant)
    PY.assert_codes(q.cpu().numpy(), exp["quant"], "e2m1", "fp4 codes")
    PY.assert_codes(sf.cpu().numpy(), oracle.swizzle_scales(exp["sf"]), "e4m3", "swizzled scales")
