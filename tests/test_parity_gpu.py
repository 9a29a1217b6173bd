"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs, element by element.  Needs a GPU (marked ``gpu``)."""
import numpy as np
import pytest
import torch

import oracle
import parity as PY
from allreduce_residual_rmsnorm_gb300 import binding as B
from allreduce_residual_rmsnorm_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def make_ws(w, max_tokens=None, mem=False):
    maxT = max_tokens or max(w.T, 1)
    if mem:
        n = B.ar_fusion_workspace_bytes(w.R, maxT, w.H, PY.BDT[w.dtype])
        buf = torch.empty(n, dtype=torch.uint8, device="cuda")
        return B.ar_fusion_workspace_create(w.R, maxT, w.H, PY.BDT[w.dtype], device_mem=buf)
    return B.ar_fusion_workspace_create(w.R, maxT, w.H, PY.BDT[w.dtype])


def run_and_check(w, variant=B.AR_VARIANT_AUTO, staged=False, mode=B.AR_MODE_AUTO, inp=None,
                  max_tokens=None, cluster=0, pdl=1, acc=B.AR_ACC_FP32):
    inp = inp or W.make_fused_inputs(w)
    ws = make_ws(w, max_tokens)
    B.ar_fusion_workspace_set_variant(ws, variant)
    B.ar_fusion_workspace_set_mode(ws, mode)
    B.ar_fusion_workspace_set_launch(ws, cluster, pdl)
    B.ar_fusion_workspace_set_accumulate(ws, acc)
    lam = staged and (mode == B.AR_MODE_LAMPORT or
                      (mode == B.AR_MODE_AUTO and w.T <= B.AR_ONESHOT_MAX_TOKENS))
    exp = PY.oracle_expected(w, inp, lamport_flip=lam, acc=acc)
    got = PY.run_gpu(ws, w, inp, scale=exp.get("scale"), staged=staged)
    rc, detail = B.ar_fusion_workspace_status(ws)
    assert rc == 0, (rc, detail)
    stats = PY.check_all(w, got, exp)
    B.ar_fusion_workspace_destroy(ws)
    return stats, got, exp


# ------------------------------------------------------------ the five targets

@pytest.mark.parametrize("variant", [B.AR_VARIANT_AUTO, B.AR_VARIANT_WARP_ROW, B.AR_VARIANT_CTA_ROW])
@pytest.mark.parametrize("staged", [False, True])
def test_tiny_r2_t16_h512(variant, staged):
    stats, _, _ = run_and_check(W.TINY, variant, staged)
    print(W.TINY.name, stats)
    assert stats["residual_mismatch"] == 0 and stats["norm_mismatch"] == 0, stats


@pytest.mark.parametrize("staged", [False, True])
def test_decode_r8_t128_h4096(staged):
    stats, _, _ = run_and_check(W.DECODE, B.AR_VARIANT_AUTO, staged)
    print(W.DECODE.name, stats)
    assert stats["residual_mismatch"] == 0 and stats["norm_mismatch"] == 0, stats


@pytest.mark.parametrize("variant", [B.AR_VARIANT_AUTO, B.AR_VARIANT_CTA_ROW, B.AR_VARIANT_BULK_PIPE])
def test_fp8_r4_t2048_h8192(variant):
    stats, _, _ = run_and_check(W.FP8_PREFILL, variant, staged=True)
    print(W.FP8_PREFILL.name, stats)
    assert stats["residual_mismatch"] == 0, stats
    assert stats["norm_mismatch"] <= 0.00001 * W.FP8_PREFILL.T * W.FP8_PREFILL.H, stats


@pytest.mark.parametrize("variant,staged", [(B.AR_VARIANT_AUTO, True),
                                            (B.AR_VARIANT_CTA_ROW, False)])
def test_nvfp4_r8_t8192_h7168_full_size(variant, staged):
    # the benchmarked configuration, element by element over every output
    stats, _, _ = run_and_check(W.NVFP4_PREFILL, variant, staged)
    print(W.NVFP4_PREFILL.name, stats)
    assert stats["residual_mismatch"] == 0, stats


def test_nvfp4_with_norm_out_small():
    w = W.NVFP4_PREFILL.with_(T=300, pattern=W.RES_NORM_NVFP4)
    for variant in (B.AR_VARIANT_CTA_ROW, B.AR_VARIANT_BULK_PIPE):
        stats, _, _ = run_and_check(w, variant)
        assert stats["residual_mismatch"] == 0 and stats["norm_mismatch"] == 0, stats


# ------------------------------------------------------------------ edges

EDGE = [
    # (R, T, H, dtype, pattern)
    (1, 1, 8, "bf16", W.RES_NORM), (3, 5, 24, "bf16", W.NORM), (5, 3, 16, "fp16", W.RES_QUANT_NVFP4),
    (16, 7, 520, "bf16", W.RES_NORM_FP8), (2, 37, 1000, "fp16", W.RES_QUANT_FP8),
    (7, 9, 1024, "bf16", W.RES_NORM_NVFP4), (4, 13, 1032, "bf16", W.RES_NORM),
    (8, 33, 2048, "fp16", W.RES_NORM), (6, 17, 7176, "bf16", W.RES_NORM_FP8),
    (2, 3, 32768, "bf16", W.RES_QUANT_NVFP4), (16, 2, 32768, "fp16", W.RES_NORM),
    (3, 5, 20480, "bf16", W.RES_NORM_NVFP4), (5, 4, 16392, "fp16", W.RES_NORM),
    # three vectors per thread (<= 4 ranks, 1025..1536 vectors)
    (3, 7, 10240, "bf16", W.RES_NORM_NVFP4), (4, 33, 12288, "fp16", W.RES_NORM_FP8),
    (2, 9, 8200, "bf16", W.RES_NORM),
    (8, 200, 4096, "bf16", W.RES_NORM_NVFP4), (1, 500, 7168, "fp16", W.RES_QUANT_FP8),
    # two rows per SM (<= 4 ranks, 513..1023 vectors, <= 2304 rank-vectors,
    # at least 2 rows per SM); the last three stay one row per SM (next row
    # loaded ahead)
    (3, 320, 6128, "bf16", W.RES_NORM_NVFP4), (4, 350, 4104, "fp16", W.RES_NORM_FP8),
    (2, 400, 8184, "bf16", W.RES_QUANT_FP8), (3, 320, 6160, "bf16", W.RES_NORM_NVFP4),
    (2, 400, 8192, "fp16", W.RES_QUANT_FP8), (4, 333, 8192, "bf16", W.RES_NORM),
    # 449..512 vectors, one vector per thread: 6..8 ranks load the next row
    # ahead (more rows than SMs), 5 ranks run two rows per SM (at least 2
    # rows per SM); the last one has one row per block
    (8, 320, 4096, "bf16", W.RES_NORM_NVFP4), (6, 400, 3600, "fp16", W.RES_NORM_FP8),
    (7, 153, 4096, "bf16", W.RES_QUANT_NVFP4), (8, 303, 4096, "fp16", W.RES_NORM),
    (5, 310, 4000, "bf16", W.RES_NORM), (5, 200, 4096, "fp16", W.RES_NORM),
    (8, 152, 4096, "bf16", W.RES_NORM),
]


@pytest.mark.parametrize("R,T,H,dtype,pattern", EDGE)
@pytest.mark.parametrize("variant", [B.AR_VARIANT_AUTO, B.AR_VARIANT_WARP_ROW, B.AR_VARIANT_CTA_ROW,
                                     B.AR_VARIANT_BULK_PIPE])
def test_edge_shapes(R, T, H, dtype, pattern, variant):
    w = W.FusedWorkload(f"edge_{R}_{T}_{H}", R=R, T=T, H=H, dtype=dtype, pattern=pattern,
                        eps=1e-5, seed=R * 1000 + T)
    stats, _, _ = run_and_check(w, variant)
    assert stats.get("residual_mismatch", 0) == 0, stats
    assert stats.get("norm_mismatch", 0) <= max(1, T * H // 100000), stats


# ------------------------------------------- cluster-split rows, PDL launch

CLUSTER_CASES = [
    # (R, T, H, dtype, pattern)
    W.DECODE,                                                               # 8 x 128 x 4096
    W.FusedWorkload("cl_nvfp4", R=8, T=40, H=7168, pattern=W.RES_NORM_NVFP4, heavy_frac=0.01),
    W.FusedWorkload("cl_fp8", R=3, T=7, H=2064, pattern=W.RES_NORM_FP8, dtype="fp16", seed=3),
    W.FusedWorkload("cl_r16", R=16, T=5, H=8192, pattern=W.NORM, seed=4),
]


@pytest.mark.parametrize("w", CLUSTER_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("cluster", [2, 4, 8])
@pytest.mark.parametrize("staged,pdl", [(False, 0), (True, 1)])
def test_cluster_split_rows(w, cluster, staged, pdl):
    stats, _, _ = run_and_check(w, B.AR_VARIANT_CTA_ROW, staged, cluster=cluster, pdl=pdl)
    assert stats.get("residual_mismatch", 0) == 0, stats
    assert stats.get("norm_mismatch", 0) <= max(1, w.T * w.H // 100000), stats


def test_cluster_lamport_sequence_with_pdl():
    # several one-shot calls in a row with both launch options on: the slot
    # state machine and the retired-slot clear still hold
    w = W.DECODE.with_(T=48)
    ws = make_ws(w)
    B.ar_fusion_workspace_set_launch(ws, 4, 1)
    for k in range(5):
        wk = w.with_(seed=50 + k)
        inp = W.make_fused_inputs(wk)
        exp = PY.oracle_expected(wk, inp, lamport_flip=True)
        got = PY.run_gpu(ws, wk, inp, staged=True)
        PY.check_all(wk, got, exp)
        assert np.array_equal(got["residual"], exp["residual"])
        st = B.ar_fusion_workspace_copy_state(ws)
        assert st["lamport_flag"] == (k + 1) % 3 and st["status"] == 0 and st["counter"] == 0
    B.ar_fusion_workspace_destroy(ws)


def test_set_launch_rejects_bad_values():
    ws = make_ws(W.TINY)
    for cl, pdl in ((3, 0), (16, 0), (-1, 0), (2, 2)):
        with pytest.raises(B.ArFusionError) as e:
            B.ar_fusion_workspace_set_launch(ws, cl, pdl)
        assert e.value.code == B.AR_ERR_INVALID
    B.ar_fusion_workspace_destroy(ws)


# ---------------------------------------- element-type accumulation variant

ACC_CASES = [
    (W.TINY, B.AR_VARIANT_WARP_ROW, True),
    (W.DECODE, B.AR_VARIANT_CTA_ROW, True),
    (W.FusedWorkload("acc_fp16", R=5, T=300, H=3072, dtype="fp16", pattern=W.RES_NORM_FP8),
     B.AR_VARIANT_CTA_ROW, False),
    (W.FusedWorkload("acc_pipe", R=8, T=400, H=7168, pattern=W.RES_QUANT_NVFP4, heavy_frac=0.01),
     B.AR_VARIANT_BULK_PIPE, False),
    (W.FusedWorkload("acc_r16", R=16, T=33, H=1024, pattern=W.RES_NORM), B.AR_VARIANT_WARP_ROW, False),
    # 449..512 vectors: 8 ranks load the next row ahead, 5 ranks two rows per SM
    (W.FusedWorkload("acc_ahead", R=8, T=400, H=4096, pattern=W.RES_NORM_NVFP4),
     B.AR_VARIANT_AUTO, True),
    (W.FusedWorkload("acc_two_rows", R=5, T=320, H=3840, dtype="fp16", pattern=W.RES_QUANT_FP8),
     B.AR_VARIANT_AUTO, False),
]


@pytest.mark.parametrize("w,variant,staged", ACC_CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_element_type_accumulation(w, variant, staged):
    stats, _, _ = run_and_check(w, variant, staged, acc=B.AR_ACC_ELEMENT)
    assert stats.get("residual_mismatch", 0) == 0, stats
    assert stats.get("norm_mismatch", 0) <= max(1, w.T * w.H // 100000), stats


@pytest.mark.parametrize("R,N,dtype,offset", [(8, 1_000_003, "fp16", 0), (3, 4099, "bf16", 0),
                                               (16, 77777, "fp16", 1)])
def test_vector_sum_element_type_accumulation(R, N, dtype, offset):
    x = W.make_sum_inputs(W.SumWorkload("s", R=R, N=N + offset, dtype=dtype))
    exp = oracle.vector_sum(PY.ODT[dtype], W.bits(x[:, offset:]), acc=1)
    xd = x.cuda()
    out_full = torch.zeros(N + 8, dtype=xd.dtype, device="cuda")
    out = out_full[offset:offset + N]
    B.ar_fusion_sum_ex([xd[r, offset:] for r in range(R)], out, B.AR_ACC_ELEMENT)
    torch.cuda.synchronize()
    assert np.array_equal(W.bits(out.cpu()), exp)


# Values that stress the per-add rounding of the element-type sum: signed
# zeros, subnormals, neighbours one unit in the last place apart, exact halves
# of a unit (ties), the largest finite values and infinities.
SPECIALS = {
    "fp16": [0.0, -0.0, 2.0**-24, -2.0**-24, 3 * 2.0**-24, 2.0**-14, 1.0, 1 + 2.0**-10, 2.0**-11,
             -2.0**-11, 3 * 2.0**-12, 65504.0, -65504.0, 32768.0, float("inf"), float("-inf")],
    "bf16": [0.0, -0.0, 2.0**-133, -2.0**-133, 2.0**-126, 1.0, 1 + 2.0**-7, 2.0**-8, -2.0**-8,
             3 * 2.0**-10, 2.0**127 * 1.9921875, -2.0**127 * 1.9921875, 2.0**127, float("inf"),
             float("-inf")],
}


def special_draw(dtype, shape, seed, finite=False):
    pool = [v for v in SPECIALS[dtype] if not finite or abs(v) < 1e4]
    if not finite:
        pool.append(float("nan"))
    vals = torch.tensor(pool, dtype=W.torch_dtype(dtype))
    rng = np.random.default_rng(seed)
    x = vals[torch.from_numpy(rng.integers(0, len(pool), size=shape))]
    # a third of the elements ordinary values, so special and plain terms meet
    plain = torch.from_numpy(rng.uniform(-2, 2, size=shape)).to(x.dtype)
    return torch.where(torch.from_numpy(rng.random(shape) < 1 / 3), plain, x)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("R", [2, 5, 8])
def test_vector_sum_special_values(dtype, R):
    x = special_draw(dtype, (R, 40_003), seed=R)
    xd = x.cuda()
    for acc, oacc in ((B.AR_ACC_ELEMENT, 1), (B.AR_ACC_FP32, 0)):
        exp = oracle.vector_sum(PY.ODT[dtype], W.bits(x), acc=oacc)
        out = torch.empty(x.shape[1], dtype=x.dtype, device="cuda")
        B.ar_fusion_sum_ex([xd[r] for r in range(R)], out, acc)
        torch.cuda.synchronize()
        got = out.cpu()
        nan_e = torch.isnan(W.from_bits(exp, dtype)).numpy()
        assert np.array_equal(torch.isnan(got).numpy(), nan_e), (acc, "NaN positions")
        assert np.array_equal(W.bits(got)[~nan_e], exp[~nan_e]), acc


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("variant", [B.AR_VARIANT_WARP_ROW, B.AR_VARIANT_CTA_ROW,
                                     B.AR_VARIANT_BULK_PIPE])
def test_element_type_accumulation_special_partials(dtype, variant):
    # finite specials only: the row's norm stays finite
    w = W.FusedWorkload(f"acc_special_{dtype}", R=6, T=40, H=512 if variant == B.AR_VARIANT_WARP_ROW
                        else 2048, dtype=dtype, pattern=W.RES_NORM)
    inp = W.make_fused_inputs(w)
    inp.partials = special_draw(dtype, (w.R, w.T, w.H), seed=7, finite=True)
    for acc in (B.AR_ACC_ELEMENT, B.AR_ACC_FP32):
        stats, _, _ = run_and_check(w, variant, False, inp=inp, acc=acc)
        assert stats.get("residual_mismatch", 0) == 0, (acc, stats)
        assert stats.get("norm_mismatch", 0) <= max(1, w.T * w.H // 100000), (acc, stats)


@pytest.mark.parametrize("staged", [False, True])
def test_staged_buffer_mode_and_capacity(staged):
    w = W.DECODE.with_(T=100)
    stats, _, _ = run_and_check(w, B.AR_VARIANT_CTA_ROW, staged, mode=B.AR_MODE_BUFFER,
                                max_tokens=160)
    assert stats["residual_mismatch"] == 0


def test_zero_tokens_launches_nothing():
    w = W.TINY
    ws = make_ws(w)
    X = torch.empty(0, w.H, dtype=torch.bfloat16, device="cuda")
    G = torch.ones(w.H, dtype=torch.bfloat16, device="cuda")
    B.ar_fusion_run(ws, None, X, G, 1e-6, B.PATTERNS[w.pattern])
    B.ar_fusion_run(ws, [X, X], X, G, 1e-6, B.PATTERNS[w.pattern])
    st = B.ar_fusion_workspace_copy_state(ws)
    assert st["calls"] == 0 and st["lamport_flag"] == 0
    B.ar_fusion_workspace_destroy(ws)


def test_all_zero_inputs_nvfp4_and_fp8():
    for pat in (W.RES_NORM_NVFP4, W.RES_NORM_FP8):
        w = W.FusedWorkload("zeros", R=4, T=6, H=256, pattern=pat)
        inp = W.make_fused_inputs(w)
        inp.partials.zero_()
        inp.residual.zero_()
        stats, got, _ = run_and_check(w, inp=inp)
        assert np.all(got["quant"] == 0)
        if "sf" in got:
            assert np.all(got["sf"] == 0)


# ------------------------------------------------------- Lamport state machine

def test_lamport_sequence_state_and_retired_slot_clear():
    w = W.TINY
    ws = make_ws(w, mem=True)
    info = B.ar_fusion_workspace_info(ws)
    mem = ws.mem
    slot_b = info["lamport_comm_bytes"]
    lam_off = info["lamport"] - info["base"]
    flag = 0
    clear = 0
    for k in range(7):
        wk = w.with_(seed=100 + k, T=w.T - (k % 3))      # varying T changes clear sizes
        inp = W.make_fused_inputs(wk)
        exp = PY.oracle_expected(wk, inp, lamport_flip=True)
        got = PY.run_gpu(ws, wk, inp, staged=True)
        PY.check_all(wk, got, exp)
        assert np.array_equal(got["residual"], exp["residual"])
        st = B.ar_fusion_workspace_copy_state(ws)
        new_flag, new_clear, rd, cl = oracle.lamport_step(flag, clear, wk.R, wk.T, wk.H)
        assert st["lamport_flag"] == new_flag and st["clear_size"] == new_clear
        assert st["counter"] == 0 and st["calls"] == k + 1 and st["status"] == 0
        # the slot cleared by this call holds sentinel words over the previous clear size
        words = mem[lam_off + cl * slot_b: lam_off + cl * slot_b + clear * 2].view(torch.int32)
        assert bool((words == torch.tensor(-2 ** 31, dtype=torch.int32, device="cuda")).all())
        flag, clear = new_flag, new_clear
    B.ar_fusion_workspace_destroy(ws)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_lamport_sentinel_pairs_are_flipped_on_stage(dtype):
    w = W.TINY.with_(seed=5, dtype=dtype)
    inp = W.make_fused_inputs(w)
    p16 = inp.partials.view(torch.int16)
    p16[:, :, 0] = 0                       # (lo=+0, hi=-0): the -0.0f sentinel word
    p16[:, :, 1] = -32768
    p16[:, 3, 4] = -32768                  # low half -0 with a non-zero high half: kept
    stats, _, _ = run_and_check(w, staged=True, inp=inp)
    assert stats["residual_mismatch"] == 0
    stats, _, _ = run_and_check(w, staged=False, inp=inp)
    assert stats["residual_mismatch"] == 0


def test_lamport_wait_times_out_and_reset_recovers():
    w = W.TINY
    inp = W.make_fused_inputs(w)
    ws = make_ws(w)
    B.ar_fusion_workspace_set_timeout_ns(ws, 20_000_000)   # 20 ms bound per wait
    P = inp.partials.cuda()
    X, G = inp.residual.cuda(), inp.gamma.cuda()
    res, nrm = torch.empty_like(X), torch.empty_like(X)
    for r in range(w.R - 1):                # the last rank never arrives
        B.ar_fusion_workspace_stage(ws, r, P[r])
    B.ar_fusion_run(ws, None, X, G, w.eps, B.PATTERNS[w.pattern], residual_out=res, norm_out=nrm)
    rc, detail = B.ar_fusion_workspace_status(ws)
    assert rc == B.AR_ERR_TIMEOUT
    assert detail % 32 == w.R - 1 and 0 <= detail // 32 < w.T
    B.ar_fusion_workspace_reset(ws)
    assert B.ar_fusion_workspace_status(ws)[0] == 0
    got = PY.run_gpu(ws, w, inp, staged=True)
    exp = PY.oracle_expected(w, inp, lamport_flip=True)
    PY.check_all(w, got, exp)
    assert B.ar_fusion_workspace_status(ws)[0] == 0
    B.ar_fusion_workspace_destroy(ws)


def test_bulk_pipe_with_a_1ns_wait_bound_is_correct_or_reports_a_timeout():
    """The bulk-copy pipe with a 1 ns bound per stage wait.  Each wait first
    suspends in the barrier unit until its phase completes, so in practice no
    wait runs out; whichever happens, a call must either finish with the
    oracle's outputs and a clean status, or report AR_ERR_TIMEOUT from a
    consumer (-1) or producer (-2) wait and end (every copy it issued lands
    before its block exits: the producer's final wait for its copies keeps a
    floor of 200 ms).  After a reset, with the default bound, the workspace
    computes the oracle's outputs."""
    w = W.FusedWorkload("pipe_tiny_bound", R=8, T=304, H=16384, pattern=W.RES_NORM)
    inp = W.make_fused_inputs(w)
    exp = PY.oracle_expected(w, inp)
    ws = make_ws(w)
    B.ar_fusion_workspace_set_variant(ws, B.AR_VARIANT_BULK_PIPE)
    B.ar_fusion_workspace_set_timeout_ns(ws, 1)
    outcomes = []
    for _ in range(5):
        got = PY.run_gpu(ws, w, inp)
        assert B.ar_fusion_workspace_info(ws)["last_variant"] == B.AR_VARIANT_BULK_PIPE
        rc, detail = B.ar_fusion_workspace_status(ws)
        if rc == 0:
            PY.check_all(w, got, exp)
        else:
            assert rc == B.AR_ERR_TIMEOUT and detail in (-1, -2), (rc, detail)
            B.ar_fusion_workspace_reset(ws)
        outcomes.append(rc)
    B.ar_fusion_workspace_reset(ws)
    assert B.ar_fusion_workspace_status(ws)[0] == 0
    B.ar_fusion_workspace_set_timeout_ns(ws, 2_000_000_000)
    got = PY.run_gpu(ws, w, inp)
    PY.check_all(w, got, exp)
    assert B.ar_fusion_workspace_status(ws)[0] == 0
    B.ar_fusion_workspace_destroy(ws)


def test_lamport_wait_times_out_in_the_pipelined_row_and_reset_recovers():
    """At most 4 ranks, one vector per thread: the row's rank vectors are
    loaded ahead and polled in place.  A rank that never arrives makes that
    poll give up (AR_ERR_TIMEOUT naming the row and the rank); after a reset
    the workspace computes the oracle's outputs."""
    w = W.FusedWorkload("lam_pipe_timeout", R=4, T=64, H=4096, pattern=W.RES_NORM_FP8)
    inp = W.make_fused_inputs(w)
    ws = make_ws(w)
    B.ar_fusion_workspace_set_variant(ws, B.AR_VARIANT_CTA_ROW)
    B.ar_fusion_workspace_set_timeout_ns(ws, 20_000_000)    # 20 ms bound per wait
    P = inp.partials.cuda()
    X, G = inp.residual.cuda(), inp.gamma.cuda()
    res, nrm = torch.empty_like(X), torch.empty_like(X)
    q = torch.empty(w.T, w.H, dtype=torch.uint8, device="cuda")
    sc = torch.ones(1, device="cuda")
    for r in range(w.R - 1):                # rank 3 never arrives
        B.ar_fusion_workspace_stage(ws, r, P[r])
    B.ar_fusion_run(ws, None, X, G, w.eps, B.PATTERNS[w.pattern], residual_out=res, norm_out=nrm,
                    quant_out=q, scale_factor=sc)
    rc, detail = B.ar_fusion_workspace_status(ws)
    assert rc == B.AR_ERR_TIMEOUT
    assert detail % 32 == w.R - 1 and 0 <= detail // 32 < w.T
    assert B.ar_fusion_workspace_info(ws)["last_variant"] == B.AR_VARIANT_CTA_ROW
    B.ar_fusion_workspace_reset(ws)
    B.ar_fusion_workspace_set_timeout_ns(ws, 2_000_000_000)
    exp = PY.oracle_expected(w, inp, lamport_flip=True)
    got = PY.run_gpu(ws, w, inp, scale=exp["scale"], staged=True)
    PY.check_all(w, got, exp)
    assert B.ar_fusion_workspace_status(ws)[0] == 0
    B.ar_fusion_workspace_destroy(ws)


@pytest.mark.parametrize("R,T,H,dtype", [(4, 400, 4096, "bf16"), (2, 700, 8192, "fp16"),
                                         (3, 333, 2064, "bf16"), (8, 350, 4096, "bf16"),
                                         (6, 200, 3728, "fp16"), (3, 320, 5120, "bf16")])
def test_forced_lamport_with_several_rows_per_block(R, T, H, dtype):
    """Lamport mode forced beyond the one-shot token count: every block runs
    several rows, so the look-ahead loads of the next row are polling loads
    of the current slot (at shapes whose buffer-mode calls take a form
    compiled without the Lamport code, the plain row kernel runs)."""
    w = W.FusedWorkload(f"lam_rows_{R}_{T}_{H}", R=R, T=T, H=H, dtype=dtype,
                        pattern=W.RES_NORM_NVFP4, seed=R + T)
    stats, _, _ = run_and_check(w, B.AR_VARIANT_CTA_ROW, staged=True, mode=B.AR_MODE_LAMPORT)
    assert stats["residual_mismatch"] == 0, stats


def test_bound_run_repeats_the_call_it_was_made_for():
    """binding.bound_run marshals the arguments once; calling it launches the
    same call: the oracle's outputs, three times in a row on staged partials."""
    w = W.FusedWorkload("bound", R=8, T=300, H=7168, pattern=W.RES_QUANT_NVFP4, heavy_frac=0.01)
    inp = W.make_fused_inputs(w)
    exp = PY.oracle_expected(w, inp)
    ws = make_ws(w)
    P = inp.partials.cuda()
    X, G = inp.residual.cuda(), inp.gamma.cuda()
    for r in range(w.R):
        B.ar_fusion_workspace_stage(ws, r, P[r], mode=B.AR_MODE_BUFFER)
    res = torch.empty_like(X)
    q = torch.empty(w.T, w.H // 2, dtype=torch.uint8, device="cuda")
    sf = torch.empty(w.T, w.H // 16, dtype=torch.uint8, device="cuda")
    sc = torch.tensor([float(exp["scale"])], device="cuda")
    call = B.bound_run(ws, None, X, G, w.eps, B.PATTERNS[w.pattern], residual_out=res,
                       quant_out=q, scale_out=sf, scale_factor=sc)
    B.ar_fusion_workspace_set_mode(ws, B.AR_MODE_BUFFER)
    for _ in range(3):
        res.fill_(float("nan"))
        q.fill_(0xAA)
        sf.fill_(0xAA)
        call()
        torch.cuda.synchronize()
        got = {"residual": W.bits(res.cpu()), "quant": q.cpu().numpy(), "sf": sf.cpu().numpy()}
        PY.check_all(w, got, exp)
        assert np.array_equal(got["residual"], exp["residual"])
    assert B.ar_fusion_workspace_status(ws)[0] == 0
    B.ar_fusion_workspace_destroy(ws)


# --------------------------------------------------------------- ABI errors

def test_abi_errors_launch_nothing():
    w = W.TINY
    ws = make_ws(w)
    X = torch.randn(w.T, w.H, device="cuda").to(torch.bfloat16)
    G = torch.ones(w.H, dtype=torch.bfloat16, device="cuda")
    P = [torch.randn(w.T, w.H, device="cuda").to(torch.bfloat16) for _ in range(w.R)]
    out = torch.full((w.T, w.H), 7.0, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(w.T, w.H, dtype=torch.uint8, device="cuda")
    sc = torch.ones(1, device="cuda")
    L = B.lib()

    def expect(code, fn):
        with pytest.raises(B.ArFusionError) as e:
            fn()
        assert e.value.code == code, (e.value, code)

    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws, P, X, G, 1e-6, 0, out, out))
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws, P, X, G, 1e-6, B.AR_RESIDUAL_OUT, out, out))
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws, P, X, G, 1e-6, B.AR_NORM_OUT | B.AR_QUANT_FP8,
                                                     out, out, q, None, sc))
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws, P, X, G, 1e-6,
                                                     B.AR_RESIDUAL_OUT | B.AR_QUANT_FP8 | B.AR_QUANT_NVFP4,
                                                     out, out, q, q, sc))
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws, P, X, G, 1e-6, 16 | B.AR_NORM_OUT, out, out))
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws, P, X, G, 1e-6, B.PATTERNS["res_fp8"], out,
                                                     None, q, None, None))
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws, P, X, G, 1e-6, B.PATTERNS["res_nvfp4"], out,
                                                     None, q, None, sc))
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws, P, X, G, 1e-6, B.PATTERNS["res_norm"], None, out))
    # misaligned pointer
    Xo = torch.empty(w.T * w.H + 8, dtype=torch.bfloat16, device="cuda")[1:1 + w.T * w.H].view(w.T, w.H)
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws, P, Xo, G, 1e-6, B.PATTERNS["res_norm"], out, out))
    # dtype mismatch with the workspace
    Xh = X.half()
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws, [p.half() for p in P], Xh, G.half(), 1e-6,
                                                     B.PATTERNS["res_norm"], out.half(), out.half()))
    # staged: wrong rank count, capacity
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws, None, X, G, 1e-6, B.PATTERNS["res_norm"],
                                                     out, out, nranks=3))
    Xbig = torch.randn(w.T + 1, w.H, device="cuda").to(torch.bfloat16)
    outbig = torch.empty_like(Xbig)
    expect(B.AR_ERR_CAPACITY, lambda: B.ar_fusion_run(ws, None, Xbig, G, 1e-6, B.PATTERNS["res_norm"],
                                                      outbig, outbig))
    expect(B.AR_ERR_UNSUPPORTED, lambda: B.ar_fusion_run(ws, P * 9, X, G, 1e-6, B.PATTERNS["res_norm"],
                                                         out, out))
    expect(B.AR_ERR_CAPACITY, lambda: B.ar_fusion_workspace_stage(ws, 0, Xbig))
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_workspace_stage(ws, w.R, X))
    # NVFP4 needs hidden % 16 == 0
    ws2 = B.ar_fusion_workspace_create(2, 4, 24, B.AR_DT_BF16)
    X24 = torch.zeros(4, 24, dtype=torch.bfloat16, device="cuda")
    G24 = torch.ones(24, dtype=torch.bfloat16, device="cuda")
    expect(B.AR_ERR_INVALID, lambda: B.ar_fusion_run(ws2, [X24, X24], X24, G24, 1e-6, B.PATTERNS["res_nvfp4"],
                                                     X24, None, q, q, sc))
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a rejected call wrote an output"
    st = B.ar_fusion_workspace_copy_state(ws)
    assert st["calls"] == 0
    del L
    B.ar_fusion_workspace_destroy(ws2)
    B.ar_fusion_workspace_destroy(ws)


def test_outputs_stay_inside_their_bounds():
    # canary bands around every output in place of a memory checker
    w = W.FusedWorkload("canary", R=3, T=37, H=1040, pattern=W.RES_NORM_NVFP4, seed=3)
    inp = W.make_fused_inputs(w)
    exp = PY.oracle_expected(w, inp)
    for variant in (B.AR_VARIANT_WARP_ROW, B.AR_VARIANT_CTA_ROW, B.AR_VARIANT_BULK_PIPE):
        ws = make_ws(w)
        B.ar_fusion_workspace_set_variant(ws, variant)
        pad = 4096
        def band(n, dt):
            t = torch.full((n + 2 * pad,), 0x5A if dt == torch.uint8 else 1234.0, dtype=dt, device="cuda")
            return t, t[pad:pad + n]
        rb, res = band(w.T * w.H, torch.bfloat16)
        nb, nrm = band(w.T * w.H, torch.bfloat16)
        qb, q = band(w.T * w.H // 2, torch.uint8)
        sb, s = band(w.T * w.H // 16, torch.uint8)
        sc = torch.tensor([exp["scale"]], device="cuda")
        P = inp.partials.cuda()
        B.ar_fusion_run(ws, [P[r] for r in range(w.R)], inp.residual.cuda(), inp.gamma.cuda(), w.eps,
                        B.PATTERNS[w.pattern], res.view(w.T, w.H), nrm.view(w.T, w.H), q, s, sc)
        torch.cuda.synchronize()
        for full, dt in ((rb, torch.bfloat16), (nb, torch.bfloat16), (qb, torch.uint8), (sb, torch.uint8)):
            v = 0x5A if dt == torch.uint8 else 1234.0
            assert bool((full[:pad] == v).all()) and bool((full[-pad:] == v).all()), variant
        got = {"residual": W.bits(res.view(w.T, w.H).cpu()), "norm": W.bits(nrm.view(w.T, w.H).cpu()),
               "quant": q.view(w.T, -1).cpu().numpy(), "sf": s.view(w.T, -1).cpu().numpy()}
        PY.check_all(w, got, exp)
        B.ar_fusion_workspace_destroy(ws)


# ------------------------------------------- encoders over every bf16 value

def _gamma_probe(gamma_vals, pattern, scale, sign_seed=0):
    """A row of |y| = 1 with eps = 0 has rstd = 1, so n = sign * gamma exactly:
    gamma then carries the values the quantiser sees."""
    H = gamma_vals.numel()
    T = 2
    rng = torch.Generator().manual_seed(sign_seed)
    sign = torch.where(torch.rand(T, H, generator=rng) < 0.5, -1.0, 1.0)
    w = W.FusedWorkload("probe", R=1, T=T, H=H, eps=0.0, pattern=pattern)
    inp = W.FusedInputs(partials=sign.to(torch.bfloat16).unsqueeze(0).contiguous(),
                        residual=torch.zeros(T, H, dtype=torch.bfloat16),
                        gamma=gamma_vals.to(torch.bfloat16), eps=0.0)
    ws = make_ws(w)
    B.ar_fusion_workspace_set_variant(ws, B.AR_VARIANT_CTA_ROW)
    got = PY.run_gpu(ws, w, inp, scale=scale)
    B.ar_fusion_workspace_destroy(ws)
    n = W.bits((sign * gamma_vals.to(torch.bfloat16).float()).to(torch.bfloat16))
    assert np.array_equal(got["norm"], n)
    return got, n


@pytest.mark.parametrize("mult", [1.0, 0.5, 448.0 / 7.0, 2.0 ** -9])
def test_fp8_encoder_every_bf16_value(mult):
    allbits = torch.arange(0, 65536, dtype=torch.int32)
    finite = ((allbits >> 7) & 0xff) != 0xff
    vals = allbits[finite].to(torch.int16).view(torch.bfloat16)
    vals = torch.cat([vals, torch.zeros((-vals.numel()) % 32768, dtype=torch.bfloat16)])
    for chunk in vals.split(32768):
        got, n = _gamma_probe(chunk, W.RES_NORM_FP8, mult)
        exp = oracle.quant_fp8(oracle.BF16, n, np.float32(mult))
        assert np.array_equal(got["quant"], exp)


def test_nvfp4_encoder_many_values():
    g = torch.Generator().manual_seed(1)
    e = torch.rand(32768, generator=g) * 40 - 20
    vals = (torch.exp2(e) * torch.where(torch.rand(32768, generator=g) < 0.5, -1.0, 1.0))
    vals[::97] = 0.0
    for gs in (1.0, 2688.0 / 37.5, 3.0e5):
        got, n = _gamma_probe(vals, W.RES_NORM_NVFP4, gs)
        eq, es = oracle.quant_nvfp4(oracle.BF16, n, np.float32(gs))
        assert np.array_equal(got["sf"], es)
        assert np.array_equal(got["quant"], eq)


# -------------------------------------------------------------- calibration

def test_norm_amax_from_staged_buffer_partials():
    # partials == NULL: the calibration pass reads the buffer region (never the
    # Lamport slots, whose state it must leave alone)
    w = W.FP8_PREFILL.with_(T=200, seed=4)
    inp = W.make_fused_inputs(w)
    exp = PY.oracle_expected(w, inp)
    ws = make_ws(w)
    P = inp.partials.cuda()
    for r in range(w.R):
        B.ar_fusion_workspace_stage(ws, r, P[r], mode=B.AR_MODE_BUFFER)
    before = B.ar_fusion_workspace_copy_state(ws)
    amax = torch.full((1,), -1.0, device="cuda")
    B.ar_fusion_norm_amax(ws, None, inp.residual.cuda(), inp.gamma.cuda(), w.eps, amax)
    torch.cuda.synchronize()
    assert float(amax.item()) == exp["amax"]
    after = B.ar_fusion_workspace_copy_state(ws)
    assert after["calls"] == before["calls"] and after["lamport_flag"] == before["lamport_flag"]
    B.ar_fusion_workspace_destroy(ws)


def test_norm_amax_matches_oracle():
    for w in (W.FP8_PREFILL.with_(T=256), W.TINY):
        inp = W.make_fused_inputs(w)
        exp = PY.oracle_expected(w.with_(pattern=W.RES_NORM_FP8), inp)
        ws = make_ws(w)
        P = inp.partials.cuda()
        amax = torch.full((1,), -1.0, device="cuda")
        B.ar_fusion_norm_amax(ws, [P[r] for r in range(w.R)], inp.residual.cuda(), inp.gamma.cuda(),
                              w.eps, amax)
        torch.cuda.synchronize()
        assert float(amax.item()) == exp["amax"]
        B.ar_fusion_workspace_destroy(ws)


# ---------------------------------------------------------------- plain sum

@pytest.mark.parametrize("N", W.SUM_SIZES)
def test_vector_sum_sizes(N):
    w = W.SumWorkload(f"sum{N}", R=8, N=N)
    x = W.make_sum_inputs(w)
    exp = oracle.vector_sum(oracle.FP16, W.bits(x))
    xd = x.cuda()
    out = torch.full((N,), float("nan"), dtype=torch.float16, device="cuda")
    B.ar_fusion_sum([xd[r] for r in range(w.R)], out)
    torch.cuda.synchronize()
    got = W.bits(out.cpu())
    assert np.array_equal(got, exp), np.count_nonzero(got != exp)


@pytest.mark.parametrize("R,N,dtype,offset", [(1, 1000, "fp16", 0), (3, 4099, "bf16", 0),
                                               (16, 77777, "fp16", 0), (5, 12345, "bf16", 1),
                                               (2, 7, "fp16", 3)])
def test_vector_sum_ranks_types_and_misaligned(R, N, dtype, offset):
    x = W.make_sum_inputs(W.SumWorkload("s", R=R, N=N + offset, dtype=dtype))
    exp = oracle.vector_sum(PY.ODT[dtype], W.bits(x[:, offset:]))
    xd = x.cuda()
    out_full = torch.zeros(N + 8, dtype=xd.dtype, device="cuda")
    out = out_full[offset:offset + N]
    B.ar_fusion_sum([xd[r, offset:] for r in range(R)], out)
    torch.cuda.synchronize()
    assert np.array_equal(W.bits(out.cpu()), exp)
    assert bool((out_full[offset + N:] == 0).all())


@pytest.mark.parametrize("R,N,dtype,acc", [(8, 1_000_003, "fp16", 0), (3, 4099, "bf16", 0),
                                            (16, 77777, "fp16", 1), (5, 12345, "bf16", 1),
                                            (2, 40, "fp16", 0), (1, 33, "bf16", 0),
                                            (8, 25, "fp16", 0)])
def test_vector_sum_realigned_inputs(R, N, dtype, acc):
    """Every rank and the output at its own element offset (0..7): the inputs
    are read as aligned 16-byte blocks and realigned in registers; results
    bit-exact, nothing outside the output written."""
    rng = np.random.default_rng(R * 1000 + N)
    offs = rng.integers(0, 8, size=R)
    oo = int(rng.integers(0, 8))
    x = W.make_sum_inputs(W.SumWorkload("s", R=R, N=N + 8, dtype=dtype))
    views = np.stack([W.bits(x[r, offs[r]:offs[r] + N]) for r in range(R)])
    exp = oracle.vector_sum(PY.ODT[dtype], views, acc=acc)
    xd = x.cuda()
    out_full = torch.full((N + 16,), 7.0, dtype=xd.dtype, device="cuda")
    out = out_full[oo:oo + N]
    B.ar_fusion_sum_ex([xd[r, int(offs[r]):int(offs[r]) + N] for r in range(R)], out,
                       accumulate=B.AR_ACC_ELEMENT if acc else B.AR_ACC_FP32)
    torch.cuda.synchronize()
    assert np.array_equal(W.bits(out.cpu()), exp), np.count_nonzero(W.bits(out.cpu()) != exp)
    assert bool((out_full[:oo] == 7.0).all()) and bool((out_full[oo + N:] == 7.0).all())


@pytest.mark.parametrize("R,N,dtype,acc,pad", [(3, (1 << 25) + 13, "bf16", 0, 16),
                                                (8, (1 << 25) + 13, "fp16", 1, 16),
                                                (2, (1 << 25) + 5, "fp16", 0, 8)])
def test_vector_sum_large_sizes_with_32_byte_rows(R, N, dtype, acc, pad):
    """From 2^25 elements, 16-bit sums over 32-byte aligned buffers read 256
    bits per load (ragged tail summed element by element); rows aligned to 16
    bytes only (pad = 8 elements) keep the 128-bit path.  Bit-exact."""
    stride = (N + pad - 1) // pad * pad
    x = W.make_sum_inputs(W.SumWorkload("s", R=R, N=stride, dtype=dtype))
    exp = oracle.vector_sum(PY.ODT[dtype], W.bits(x[:, :N]), acc=acc)
    xd = x.cuda()
    out_full = torch.full((stride + 16,), 7.0, dtype=xd.dtype, device="cuda")
    out = out_full[:N]
    B.ar_fusion_sum_ex([xd[r, :N] for r in range(R)], out,
                       accumulate=B.AR_ACC_ELEMENT if acc else B.AR_ACC_FP32)
    torch.cuda.synchronize()
    got = W.bits(out.cpu())
    assert np.array_equal(got, exp), np.count_nonzero(got != exp)
    assert bool((out_full[N:] == 7.0).all())


# ------------------------------------------- NVFP4 scales in the tile layout

def _run_nvfp4_swizzled(w, variant, inp=None, gs=None):
    inp = inp or W.make_fused_inputs(w)
    exp = PY.oracle_expected(w, inp)
    gs = exp["scale"] if gs is None else gs
    ws = make_ws(w)
    B.ar_fusion_workspace_set_variant(ws, variant)
    B.ar_fusion_workspace_set_scale_layout(ws, B.AR_SF_SWIZZLED)
    P = inp.partials.cuda()
    X, G = inp.residual.cuda(), inp.gamma.cuda()
    res = torch.empty_like(X)
    nrm = torch.empty_like(X)
    q = torch.zeros(w.T, w.H // 2, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(B.swizzled_scale_bytes(w.T, w.H), dtype=torch.uint8, device="cuda")
    sc = torch.tensor([gs], dtype=torch.float32, device="cuda")
    B.ar_fusion_run(ws, [P[r] for r in range(w.R)], X, G, w.eps, B.PATTERNS[w.pattern],
                    residual_out=res, norm_out=nrm, quant_out=q, scale_out=sf, scale_factor=sc)
    torch.cuda.synchronize()
    B.ar_fusion_workspace_destroy(ws)
    return exp, q, sf


@pytest.mark.parametrize("variant", [B.AR_VARIANT_WARP_ROW, B.AR_VARIANT_CTA_ROW, B.AR_VARIANT_BULK_PIPE])
@pytest.mark.parametrize("R,T,H", [(4, 200, 512), (4, 300, 7168), (4, 128, 1040), (8, 320, 4096)])
def test_nvfp4_swizzled_scale_layout_matches_oracle(variant, R, T, H):
    w = W.FusedWorkload("swz", R=R, T=T, H=H, pattern=W.RES_NORM_NVFP4, heavy_frac=0.01, seed=T + H)
    exp, q, sf = _run_nvfp4_swizzled(w, variant)
    assert np.array_equal(q.cpu().numpy(), exp["quant"])
    assert np.array_equal(sf.cpu().numpy(), oracle.swizzle_scales(exp["sf"]))


def _scaled_mm_nvfp4(a_codes, a_sf_swz, b_codes, b_sf_swz):
    """NVFP4 x NVFP4 -> bf16 through PyTorch's block-scaled matmul (cuBLASLt),
    A [M, K/2] and B [N, K/2] packed codes, scales in the tile layout."""
    fp4 = getattr(torch, "float4_e2m1fn_x2", None)
    if fp4 is None:
        pytest.skip("this PyTorch has no float4_e2m1fn_x2")
    a = a_codes.view(fp4)
    b = b_codes.view(fp4).t()
    sa = a_sf_swz.view(torch.float8_e4m3fn)
    sb = b_sf_swz.view(torch.float8_e4m3fn)
    F = torch.nn.functional
    errors = []
    if hasattr(F, "scaled_mm") and hasattr(F, "ScalingType"):
        try:
            return F.scaled_mm(a, b, sa, F.ScalingType.BlockWise1x16, sb, F.ScalingType.BlockWise1x16,
                               swizzle_a=F.SwizzleType.SWIZZLE_32_4_4,
                               swizzle_b=F.SwizzleType.SWIZZLE_32_4_4, output_dtype=torch.bfloat16)
        except Exception as e:  # noqa: BLE001
            errors.append(repr(e))
    try:
        return torch._scaled_mm(a, b, sa, sb, out_dtype=torch.bfloat16)
    except Exception as e:  # noqa: BLE001
        errors.append(repr(e))
    pytest.skip("no usable NVFP4 block-scaled matmul in this PyTorch: " + " | ".join(errors)[:300])


@pytest.mark.parametrize("T", [256, 200])
def test_nvfp4_swizzled_output_feeds_a_block_scaled_matmul(T):
    # Independent consumer of both the codes (nibble order included) and the
    # tile layout: with B = identity in NVFP4 (code 1.0, every block scale 1.0)
    # the product is A's dequantised matrix val(code) * blockscale, exact in
    # bf16 -- any misplaced scale byte or swapped nibble changes it.
    H = 512
    w = W.FusedWorkload("swz_mm", R=8, T=T, H=H, pattern=W.RES_NORM_NVFP4, heavy_frac=0.01, seed=T)
    exp, q, sf = _run_nvfp4_swizzled(w, B.AR_VARIANT_CTA_ROW)
    codes = np.stack([exp["quant"] & 0xf, exp["quant"] >> 4], -1).reshape(T, H)
    deq = oracle.e2m1_decode(codes) * np.repeat(oracle.e4m3_decode(exp["sf"]), 16, axis=1)
    eye_codes = np.zeros((H, H), np.uint8)
    np.fill_diagonal(eye_codes, 0x2)                                  # E2M1 1.0
    b_packed = (eye_codes[:, 0::2] | (eye_codes[:, 1::2] << 4)).astype(np.uint8)
    b_sf = oracle.swizzle_scales(np.full((H, H // 16), 0x38, np.uint8))  # E4M3 1.0
    out = _scaled_mm_nvfp4(q, sf, torch.from_numpy(b_packed).cuda(), torch.from_numpy(b_sf).cuda())
    got = out.float().cpu().numpy()
    assert np.array_equal(got, deq.astype(np.float32))


# ------------------------------------------------------------- CUDA graphs

@pytest.mark.parametrize("pdl", [0, 1])
@pytest.mark.parametrize("w", [W.DECODE.with_(T=64), W.DECODE, W.TINY], ids=["t64", "t128", "tiny"])
def test_graph_replay_of_stage_and_run_advances_the_lamport_slots(pdl, w):
    # the slot index and clear size live on the device, so a captured
    # stage + run replays correctly: each replay reads the slot its staging
    # filled and clears the previous one (row blocks and one-row-per-warp
    # blocks; every block takes its slot ticket right after the state read)
    ws = make_ws(w)
    B.ar_fusion_workspace_set_launch(ws, 0, pdl)
    inp0 = W.make_fused_inputs(w)
    P = inp0.partials.cuda()
    X, G = inp0.residual.cuda(), inp0.gamma.cuda()
    res, nrm = torch.empty_like(X), torch.empty_like(X)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                 # warm-up outside the capture
        for r in range(w.R):
            B.ar_fusion_workspace_stage(ws, r, P[r], stream=side)
        B.ar_fusion_run(ws, None, X, G, w.eps, B.PATTERNS[w.pattern], res, nrm, stream=side)
    torch.cuda.synchronize()
    calls0 = B.ar_fusion_workspace_copy_state(ws)["calls"]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for r in range(w.R):
            B.ar_fusion_workspace_stage(ws, r, P[r], stream=side)
        B.ar_fusion_run(ws, None, X, G, w.eps, B.PATTERNS[w.pattern], res, nrm, stream=side)
    for k in range(5):
        inp = W.make_fused_inputs(w.with_(seed=500 + k))
        P.copy_(inp.partials)
        X.copy_(inp.residual)
        G.copy_(inp.gamma)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        exp = PY.oracle_expected(w, inp, lamport_flip=True)
        got = {"residual": W.bits(res.cpu()), "norm": W.bits(nrm.cpu())}
        stats = PY.check_all(w, got, exp)
        assert stats["residual_mismatch"] == 0, (k, stats)
        st = B.ar_fusion_workspace_copy_state(ws)
        assert st["calls"] == calls0 + k + 1 and st["status"] == 0
        assert st["lamport_flag"] == (calls0 + k + 1) % 3
    del g
    B.ar_fusion_workspace_destroy(ws)


# ------------------------------------------------- partials written in place

@pytest.mark.parametrize("mode", [B.AR_MODE_BUFFER, B.AR_MODE_LAMPORT])
def test_partials_written_in_place_at_partial_ptr(mode):
    # a producer writes each rank's block at ar_fusion_workspace_partial_ptr
    # (no staging kernel); the run then reads it.  In Lamport mode the
    # address moves with every call and the producer writes no -0.0f word.
    w = W.DECODE.with_(T=96)
    ws = make_ws(w, mem=True)
    B.ar_fusion_workspace_set_mode(ws, mode)
    info = B.ar_fusion_workspace_info(ws)
    mem = ws.mem
    addrs = set()
    for k in range(4):
        inp = W.make_fused_inputs(w.with_(seed=700 + k))
        for r in range(w.R):
            ptr = B.ar_fusion_workspace_partial_ptr(ws, r, w.T, mode)
            assert ptr % 16 == 0
            addrs.add(ptr)
            words = inp.partials[r].contiguous().view(torch.int32)
            if mode == B.AR_MODE_LAMPORT:
                words = torch.where(words == -2 ** 31, torch.zeros_like(words), words)
            block = words.view(torch.uint8).reshape(-1)
            off = ptr - info["base"]
            mem[off:off + block.numel()].copy_(block)
        X, G = inp.residual.cuda(), inp.gamma.cuda()
        res, nrm = torch.empty_like(X), torch.empty_like(X)
        B.ar_fusion_run(ws, None, X, G, w.eps, B.PATTERNS[w.pattern], res, nrm)
        torch.cuda.synchronize()
        exp = PY.oracle_expected(w, inp, lamport_flip=mode == B.AR_MODE_LAMPORT)
        got = {"residual": W.bits(res.cpu()), "norm": W.bits(nrm.cpu())}
        stats = PY.check_all(w, got, exp)
        assert stats["residual_mismatch"] == 0, (k, stats)
        st = B.ar_fusion_workspace_copy_state(ws)
        assert st["status"] == 0
        assert st["calls"] == (k + 1 if mode == B.AR_MODE_LAMPORT else 0)
    # buffer mode: one fixed region per rank; Lamport: the three slots rotate
    assert len(addrs) == (w.R if mode == B.AR_MODE_BUFFER else 3 * w.R)
    B.ar_fusion_workspace_destroy(ws)


@pytest.mark.parametrize("H", [1024, 512], ids=["row_blocks", "warp_rows"])
def test_long_mixed_sequence_keeps_the_lamport_invariants(H):
    # 60 calls on one workspace: Lamport calls of varying token counts mixed
    # with staged buffer-mode calls and caller-partial calls.  After every
    # Lamport call the slot the next Lamport call will read must hold only
    # sentinel words (its retired data was cleared two calls ago), and the
    # slot counter must count exactly the Lamport calls.  At H=512 the rows
    # go one per warp, and T=1, 5 and 100 leave warps without a row, which
    # still read the slot state and take part in the block's ticket.
    import random
    w = W.FusedWorkload("mixed", R=4, T=128, H=H, pattern=W.RES_NORM)
    ws = make_ws(w, mem=True)
    info = B.ar_fusion_workspace_info(ws)
    slot_b = info["lamport_comm_bytes"]
    lam_off = info["lamport"] - info["base"]
    sent = torch.tensor(-2 ** 31, dtype=torch.int32, device="cuda")
    rng = random.Random(3)
    lamport_calls = 0
    for k in range(60):
        kind = rng.choice(["lamport", "lamport", "buffer", "caller"])
        T = rng.choice([1, 5, 64, 100, 128])
        wk = w.with_(T=T, seed=900 + k)
        inp = W.make_fused_inputs(wk)
        if kind == "caller":
            got = PY.run_gpu(ws, wk, inp, staged=False)
            exp = PY.oracle_expected(wk, inp)
        else:
            mode = B.AR_MODE_LAMPORT if kind == "lamport" else B.AR_MODE_BUFFER
            B.ar_fusion_workspace_set_mode(ws, mode)
            got = PY.run_gpu(ws, wk, inp, staged=True)
            B.ar_fusion_workspace_set_mode(ws, B.AR_MODE_AUTO)
            exp = PY.oracle_expected(wk, inp, lamport_flip=kind == "lamport")
        stats = PY.check_all(wk, got, exp)
        assert stats["residual_mismatch"] == 0, (k, kind, T, stats)
        st = B.ar_fusion_workspace_copy_state(ws)
        assert st["status"] == 0, (k, st)
        if kind == "lamport":
            lamport_calls += 1
            nxt = st["lamport_flag"] % 3
            region = ws.mem[lam_off + nxt * slot_b: lam_off + (nxt + 1) * slot_b].view(torch.int32)
            assert bool((region == sent).all()), (k, "next slot not fully cleared")
        assert st["calls"] == lamport_calls and st["lamport_flag"] == lamport_calls % 3
    B.ar_fusion_workspace_destroy(ws)


def test_caller_partials_may_exceed_max_token_num():
    # max_token_num sizes the staging regions only: a call with caller
    # partials may pass more tokens; a staged one may not
    w = W.FusedWorkload("beyond_max", R=3, T=300, H=1024, pattern=W.RES_NORM, seed=11)
    inp = W.make_fused_inputs(w)
    ws = make_ws(w, max_tokens=64)
    got = PY.run_gpu(ws, w, inp, staged=False)
    stats = PY.check_all(w, got, PY.oracle_expected(w, inp))
    assert stats["residual_mismatch"] == 0
    X = inp.residual.cuda()
    with pytest.raises(B.ArFusionError) as e:
        B.ar_fusion_run(ws, None, X, inp.gamma.cuda(), w.eps, B.PATTERNS[w.pattern],
                        torch.empty_like(X), torch.empty_like(X))
    assert e.value.code == B.AR_ERR_CAPACITY
    B.ar_fusion_workspace_destroy(ws)


def test_two_workspaces_on_two_streams_run_independently():
    # each workspace owns its slots and state: Lamport calls on two streams,
    # issued alternately without ordering between the streams, stay correct
    ws_list, streams, cases = [], [], []
    for k, w in enumerate((W.DECODE.with_(T=96, seed=41), W.TINY.with_(seed=42, T=12))):
        ws_list.append(make_ws(w))
        streams.append(torch.cuda.Stream())
        cases.append(w)
    outs = []
    for step in range(6):
        for k, (ws, s, w) in enumerate(zip(ws_list, streams, cases)):
            wk = w.with_(seed=w.seed + 100 * step)
            inp = W.make_fused_inputs(wk)
            with torch.cuda.stream(s):
                P = inp.partials.cuda(non_blocking=False)
                X, G = inp.residual.cuda(), inp.gamma.cuda()
                res, nrm = torch.empty_like(X), torch.empty_like(X)
                for r in range(wk.R):
                    B.ar_fusion_workspace_stage(ws, r, P[r], stream=s)
                B.ar_fusion_run(ws, None, X, G, wk.eps, B.PATTERNS[wk.pattern], res, nrm, stream=s)
            outs.append((k, wk, inp, res, nrm, P, X, G))
    torch.cuda.synchronize()
    for k, wk, inp, res, nrm, *_ in outs:
        exp = PY.oracle_expected(wk, inp, lamport_flip=True)
        got = {"residual": W.bits(res.cpu()), "norm": W.bits(nrm.cpu())}
        stats = PY.check_all(wk, got, exp)
        assert stats["residual_mismatch"] == 0, (k, stats)
    for ws, s in zip(ws_list, streams):
        st = B.ar_fusion_workspace_copy_state(ws, stream=s)
        assert st["calls"] == 6 and st["status"] == 0
        B.ar_fusion_workspace_destroy(ws)
