"""The seeded input recipe: the target workloads carry the stated shapes,
element types, eps and output patterns; generation is deterministic; the drawn
values have the stated distributions (partials N(0, p_std) with a heavy tail
where stated, residual N(0, 1), gamma N(1, 0.1), plain-sum inputs U(-1, 1))."""
import ast
import os

import numpy as np
import torch

from allreduce_residual_rmsnorm_gb300 import workloads as W


def test_target_workloads_are_the_stated_configurations():
    got = {w.name: (w.R, w.T, w.H, w.dtype, w.pattern, w.eps, w.p_std, w.heavy_frac)
           for w in W.FUSED}
    assert got == {
        "r2_t16_h512_res_norm": (2, 16, 512, "bf16", W.RES_NORM, 1e-6, 1.0, 0.0),
        "r8_t128_h4096_res_norm": (8, 128, 4096, "bf16", W.RES_NORM, 1e-5, 0.5, 0.0),
        "r4_t2048_h8192_res_norm_fp8": (4, 2048, 8192, "bf16", W.RES_NORM_FP8, 1e-6, 1.0, 0.0),
        "r8_t8192_h7168_res_nvfp4": (8, 8192, 7168, "bf16", W.RES_QUANT_NVFP4, 1e-6, 1.0, 0.01),
    }
    assert W.NVFP4_PREFILL.heavy_std == 20.0
    assert [s.N for s in W.SUMS] == [1024 * 4 ** k for k in range(10)] + [1_000_003]
    assert all(s.R == 8 and s.dtype == "fp16" for s in W.SUMS)


def test_generation_is_deterministic_and_seeded():
    w = W.TINY
    a, b = W.make_fused_inputs(w), W.make_fused_inputs(w)
    for x, y in ((a.partials, b.partials), (a.residual, b.residual), (a.gamma, b.gamma)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    c = W.make_fused_inputs(w.with_(seed=1))
    assert not torch.equal(a.partials, c.partials)
    s1 = W.make_sum_inputs(W.SumWorkload("s", R=3, N=1000))
    s2 = W.make_sum_inputs(W.SumWorkload("s", R=3, N=1000))
    assert torch.equal(s1.view(torch.int16), s2.view(torch.int16))


def test_drawn_values_have_the_stated_distributions():
    w = W.FusedWorkload("dist", R=2, T=512, H=1024, heavy_frac=0.01, heavy_std=20.0,
                        pattern=W.RES_NORM)
    inp = W.make_fused_inputs(w)
    p = inp.partials.float().numpy().ravel()
    n = p.size
    # heavy tail: P(|x| > 6) = 0.01 * P(|N(0, 20)| > 6) = 0.01 * 0.764, the
    # N(0, 1) part contributes ~2e-9
    frac = np.mean(np.abs(p) > 6)
    assert abs(frac - 0.00764) < 5 * np.sqrt(0.00764 / n)
    assert abs(p.var() - (0.99 + 0.01 * 400)) < 0.25
    x = inp.residual.float().numpy()
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    g = inp.gamma.float().numpy()
    assert abs(g.mean() - 1) < 0.02 and abs(g.std() - 0.1) < 0.01
    d = W.make_fused_inputs(W.DECODE.with_(T=64)).partials.float().numpy()
    assert abs(d.std() - 0.5) < 0.01
    s = W.make_sum_inputs(W.SumWorkload("s", R=8, N=100_000)).float().numpy()
    assert s.min() >= -1 and s.max() <= 1 and abs(s.mean()) < 0.01


def test_generator_module_holds_none_of_the_method():
    # the module both sides share imports neither the oracle nor the library
    path = W.__file__
    tree = ast.parse(open(path).read(), path)
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom):
            mods.add((node.module or "").split(".")[0] if node.level == 0 else "." + (node.module or ""))
    assert mods <= {"__future__", "dataclasses", "torch", "numpy", "typing", "math"}, mods
    assert os.path.basename(path) == "workloads.py"
