"""The benchmark checks its own device outputs against the oracle with the
parity tests' rules, written out in bench.py.  Here those rules run on the
oracle's own outputs (which must pass) and on planted errors (which must
fail), without a GPU."""
import numpy as np

import bench
import oracle
from allreduce_residual_rmsnorm_gb300 import binding as B
from allreduce_residual_rmsnorm_gb300 import workloads as W


def _oracle_outputs(w, lamport=False):
    inp = W.make_fused_inputs(w)
    P = W.bits(inp.partials)
    if lamport:
        P = oracle.lamport_flip(P)
    res, nrm, _ = oracle.fused(oracle.BF16, P, W.bits(inp.residual), W.bits(inp.gamma), w.eps)
    return inp, res, nrm


def test_elem_rules_accept_the_oracle_and_reject_a_planted_error():
    w = W.TINY
    _, res, nrm = _oracle_outputs(w)
    st = bench.elem_stats(nrm, nrm, "bf16")
    assert st["ok"] and st["bit_mismatch"] == 0 and st["max_abs_err"] == 0.0
    bad = nrm.copy()
    f = W.from_bits(bad, "bf16").float().numpy()
    flat = f.reshape(-1)
    flat[int(np.argmax(np.abs(flat)))] *= 1.05
    bad = W.bits(__import__("torch").from_numpy(f).to(W.torch_dtype("bf16")))
    st = bench.elem_stats(bad, nrm, "bf16")
    assert not st["ok"] and st["outside_tol"] == 1
    assert st["max_rel_err"] > 0.03 and st["max_abs_err"] > 0.0
    # one last-bit difference stays within the tolerance but is counted
    one = res.copy()
    one[0, 0] ^= 1
    st = bench.elem_stats(one, res, "bf16")
    assert st["ok"] and st["bit_mismatch"] == 1


def test_code_rules():
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 256, size=(64, 512), dtype=np.uint8)
    assert bench.code_stats(codes, codes, "e4m3")["ok"]
    two = codes.copy()
    two[3, 5] = 0x21
    codes2 = codes.copy()
    codes2[3, 5] = 0x23                   # same sign, two code steps apart
    st = bench.code_stats(two, codes2, "e4m3")
    assert not st["ok"] and st["max_step"] == 2
    many = codes.copy()
    flat = many.reshape(-1)
    idx = rng.choice(flat.size, size=int(0.002 * flat.size) + 1, replace=False)
    flat[idx] = np.where((flat[idx] & 0x7F) < 0x7E, flat[idx] + 1, flat[idx] - 1)
    st = bench.code_stats(many, codes, "e4m3")
    assert st["max_step"] == 1 and not st["ok"]
    # E2M1 nibble pairs: a swapped pair is a large step
    fp4 = rng.integers(0, 256, size=(16, 64), dtype=np.uint8)
    sw = fp4.copy()
    sw[0, 0] = ((fp4[0, 0] & 0xF) << 4) | (fp4[0, 0] >> 4)
    lo, hi = fp4[0, 0] & 7, (fp4[0, 0] >> 4) & 7
    st = bench.code_stats(sw, fp4, "e2m1")
    assert st["ok"] == (abs(int(lo) - int(hi)) <= 1 and ((fp4[0, 0] ^ sw[0, 0]) & 0x88) == 0)
    # +0 and -0 are the same code value
    z = np.array([[0x00, 0x80]], np.uint8)
    assert bench.code_stats(z, z[:, ::-1].copy(), "e4m3")["ok"]


def test_oracle_parity_passes_the_oracle_outputs_and_flags_a_wrong_scale():
    oracle.build_oracle()
    w = W.TINY
    inp, res, nrm = _oracle_outputs(w, lamport=True)
    pat = B.PATTERNS[w.pattern]
    out = [{"entry": {"workload": w.name}, "w": w, "inp": inp, "lamport": True, "pattern": pat,
            "scale": None, "residual": res, "norm": nrm, "quant": None}]
    # the benchmarked workload's role, played by a small NVFP4 case
    w4 = W.FusedWorkload("small_nvfp4", R=4, T=8, H=256, pattern=W.RES_QUANT_NVFP4,
                         heavy_frac=0.01)
    inp4 = W.make_fused_inputs(w4)
    r4, n4, _ = oracle.fused(oracle.BF16, W.bits(inp4.partials), W.bits(inp4.residual),
                             W.bits(inp4.gamma), w4.eps)
    gs = bench.quant_scale(B.AR_QUANT_NVFP4, oracle.amax(oracle.BF16, n4), B)
    q4, sf4 = oracle.quant_nvfp4(oracle.BF16, n4, gs)
    head = {"w": w4, "inp": inp4, "pattern": B.PATTERNS[w4.pattern], "scale": gs,
            "residual": r4, "quant": q4, "sf": sf4}
    chk = bench.oracle_parity(out, head, threads=2)
    assert chk["ok"], chk
    assert chk[w4.name]["nvfp4_codes"]["off"] == 0 and chk[w4.name]["nvfp4_scales"]["off"] == 0
    wrong = dict(head, sf=np.where(sf4 > 0, sf4 + 1, sf4).astype(np.uint8))
    wrong["sf"][0, 0] = sf4[0, 0] + 3
    assert not bench.oracle_parity(out, wrong, threads=2)["ok"]


def test_quant_scale_follows_the_stated_roundings():
    a = np.float32(3.1)
    assert bench.quant_scale(B.AR_QUANT_FP8, a, B) == np.float32(1.0) / (a / np.float32(448.0))
    assert bench.quant_scale(B.AR_QUANT_NVFP4, a, B) == np.float32(2688.0) / a
    assert bench.quant_scale(B.AR_QUANT_NVFP4, 0.0, B) == np.float32(1.0)
    assert bench.quant_scale(B.AR_QUANT_FP8, a, B) == oracle.fp8_inv_scale(a)
    assert bench.quant_scale(B.AR_QUANT_NVFP4, a, B) == oracle.nvfp4_global_scale(a)
