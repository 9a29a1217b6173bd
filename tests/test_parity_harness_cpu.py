"""The comparison rules of the GPU parity tests have teeth: outputs with a
planted error (one bit of residual_out, a norm_out element outside the
tolerance, a quantised code two steps away or too many one step away, a NaN)
are reported or rejected, while the oracle's own outputs pass."""
import numpy as np
import pytest
import torch

import parity as PY
from allreduce_residual_rmsnorm_gb300 import workloads as W


def expected(pattern, dtype="bf16"):
    w = W.FusedWorkload(f"harness_{pattern}_{dtype}", R=3, T=64, H=512, dtype=dtype,
                        pattern=pattern, seed=3)
    exp = PY.oracle_expected(w, W.make_fused_inputs(w))
    got = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in exp.items()}
    return w, exp, got


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_oracle_outputs_pass_with_no_mismatch(dtype):
    for pattern in (W.RES_NORM, W.RES_NORM_FP8, W.RES_NORM_NVFP4):
        w, exp, got = expected(pattern, dtype)
        stats = PY.check_all(w, got, exp)
        assert all(v == 0 for k, v in stats.items() if k != "errors"), stats
        assert all(e["max_abs_err"] == 0.0 and e["max_rel_err"] == 0.0
                   for e in stats["errors"].values()), stats


def test_one_residual_bit_is_counted():
    w, exp, got = expected(W.RES_NORM)
    got["residual"][5, 17] ^= 1                       # one unit in the last place
    assert PY.check_all(w, got, exp)["residual_mismatch"] == 1


def test_norm_outside_tolerance_is_rejected():
    w, exp, got = expected(W.RES_NORM)
    n = PY.to_float(got["norm"], "bf16")
    n[3, 100] += 0.5
    got["norm"] = W.bits(torch.from_numpy(n).to(torch.bfloat16))
    with pytest.raises(AssertionError, match="norm_out"):
        PY.check_all(w, got, exp)


def test_nan_in_an_output_is_rejected():
    w, exp, got = expected(W.RES_NORM)
    got["residual"][0, 0] = 0x7FC0                    # bf16 quiet NaN
    with pytest.raises(AssertionError, match="residual_out"):
        PY.check_all(w, got, exp)


def test_fp8_code_two_steps_away_is_rejected():
    w, exp, got = expected(W.RES_NORM_FP8)
    c = int(got["quant"][1, 1])
    mag = c & 0x7F
    got["quant"][1, 1] = (c & 0x80) | (mag + 2 if mag <= 0x7C else mag - 2)
    with pytest.raises(AssertionError, match="fp8 codes"):
        PY.check_all(w, got, exp)


def test_too_many_codes_one_step_away_are_rejected():
    w, exp, got = expected(W.RES_NORM_FP8)
    q = got["quant"].reshape(-1)
    n = int(0.002 * q.size) + 1                      # 0.2 % of the codes
    idx = np.arange(n) * 7
    mag = q[idx] & 0x7F
    q[idx] = (q[idx] & 0x80) | np.where(mag < 0x7E, mag + 1, mag - 1)
    with pytest.raises(AssertionError, match="codes differ"):
        PY.check_all(w, got, exp)


def test_few_codes_one_step_away_are_counted():
    w, exp, got = expected(W.RES_NORM_FP8)
    q = got["quant"].reshape(-1)
    idx = np.array([10, 2000, 30000])
    mag = q[idx] & 0x7F
    q[idx] = (q[idx] & 0x80) | np.where(mag < 0x7E, mag + 1, mag - 1)
    assert PY.check_all(w, got, exp)["fp8_off"] == 3


def test_signed_zero_codes_are_equal():
    a = np.array([0x00, 0x80, 0x08, 0x88], np.uint8)
    assert PY.e4m3_step(a, a[[1, 0, 1, 0]]).tolist() == [0, 0, 8, 8]
    assert PY.e2m1_step(np.array([0x0, 0x8]), np.array([0x8, 0x0])).tolist() == [0, 0]


def test_swapped_nvfp4_nibbles_are_rejected():
    w, exp, got = expected(W.RES_NORM_NVFP4)
    q = got["quant"].reshape(-1)
    lo, hi = q & 0xF, q >> 4
    d = PY.e2m1_step(lo, hi)
    idx = np.nonzero(d >= 2)[0][:64]                  # pairs whose halves differ by 2+ steps
    assert idx.size
    q[idx] = (lo[idx] << 4) | hi[idx]
    with pytest.raises(AssertionError, match="nvfp4 codes"):
        PY.check_all(w, got, exp)


def test_a_wrong_block_scale_is_rejected():
    w, exp, got = expected(W.RES_NORM_NVFP4)
    s = got["sf"].reshape(-1)
    k = int(np.argmax((s & 0x7F) > 0x10))
    s[k] = (s[k] & 0x80) | ((s[k] & 0x7F) - 8)       # one binade lower
    with pytest.raises(AssertionError, match="nvfp4 scales"):
        PY.check_all(w, got, exp)
