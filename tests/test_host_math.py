"""Host-compiled checks of the kernels' own arithmetic helpers (no GPU)."""
import os
import subprocess

from allreduce_residual_rmsnorm_gb300 import build as BUILD

HERE = os.path.dirname(os.path.abspath(__file__))


def _df_check(tmp_path, plant: int):
    exe = tmp_path / f"df_check_{plant}"
    subprocess.check_call([BUILD.nvcc(), "-O2", "-std=c++17", "-I", BUILD.INCLUDE, "-I", BUILD.CSRC,
                           f"-DAR_DF_CHECK_PLANT={plant}",
                           os.path.join(HERE, "host_df_check.cu"), "-o", str(exe)])
    return subprocess.run([str(exe)], capture_output=True, text=True)


def test_double_float_sum_of_squares_is_correctly_rounded(tmp_path):
    r = _df_check(tmp_path, 0)
    assert r.returncode == 0, r.stdout + r.stderr


def test_double_float_check_rejects_a_plain_fp32_sum(tmp_path):
    """The same check with the TwoSum errors dropped must fail most trials."""
    r = _df_check(tmp_path, 1)
    assert r.returncode != 0
    bad = int(r.stdout.strip().split()[0].split("/")[0])
    assert bad > 800, r.stdout


# ---- the packed 16-bit residual add: rnd16(fp32(a + b)) == rnd16(a + b)
#
# The kernels form y = rnd(f(a) + f(x)) with one packed bf16x2 / f16x2 add,
# i.e. a single correct rounding of the exact sum, while the operation adds in
# fp32 and rounds that to the element type.  The two agree because when the
# exact sum is not an fp32 value the smaller addend sits far below the larger
# one's last 16-bit bit.  Checked here with exact rational arithmetic.

from fractions import Fraction  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

FORMATS = {  # name: (mantissa bits, min normal exponent, max exponent)
    "bf16": (7, -126, 127),
    "fp16": (10, -14, 15),
}


def _round_exact(x: Fraction, fmt: str) -> float:
    """Correct round-to-nearest-even of a rational to the 16-bit format
    (as a Python float; overflow to +-inf)."""
    mbits, emin, emax = FORMATS[fmt]
    if x == 0:
        return 0.0
    sgn = -1 if x < 0 else 1
    ax = abs(x)
    e = ax.numerator.bit_length() - ax.denominator.bit_length()
    if Fraction(2) ** e > ax:
        e -= 1
    e = max(e, emin)                       # subnormals share the smallest quantum
    q = Fraction(2) ** (e - mbits)
    n = ax / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = fl * q
    if v >= Fraction(2) ** (emax + 1):
        return sgn * float("inf")
    return sgn * float(v)


def _pairs(fmt, n, rng):
    """Random finite 16-bit values, plus pairs built to sit near ties."""
    dt = torch.bfloat16 if fmt == "bf16" else torch.float16
    bits = rng.integers(0, 1 << 16, size=(n, 2), dtype=np.int64).astype(np.int16)
    v = torch.from_numpy(bits).view(dt).float().numpy()
    v = v[np.isfinite(v).all(axis=1)]
    # same-exponent pairs (ties), near-cancellation, and tiny second addends
    a = torch.from_numpy((rng.standard_normal(n) * 4).astype(np.float32)).to(dt).float().numpy()
    k = rng.integers(0, 40, size=n)
    tiny = torch.from_numpy((a * np.ldexp(1.0, -k) * (1 + rng.standard_normal(n) / 64))
                            .astype(np.float32)).to(dt).float().numpy()
    near = torch.from_numpy((-a * (1 + rng.standard_normal(n) / 256)).astype(np.float32)).to(dt).float().numpy()
    return np.concatenate([v, np.stack([a, tiny], 1), np.stack([a, near], 1)])


def _via_fp32(a, b, fmt):
    s = (a.astype(np.float32) + b.astype(np.float32)).astype(np.float32)
    if fmt == "bf16":
        return torch.from_numpy(s).to(torch.bfloat16).float().numpy()
    with np.errstate(over="ignore"):          # sums beyond 65504 round to inf
        return s.astype(np.float16).astype(np.float32)


def test_packed_16bit_add_equals_fp32_add_then_round():
    rng = np.random.default_rng(7)
    for fmt in FORMATS:
        p = _pairs(fmt, 6000, rng)
        got = _via_fp32(p[:, 0], p[:, 1], fmt)
        for (a, b), g in zip(p, got):
            want = _round_exact(Fraction(float(a)) + Fraction(float(b)), fmt)
            assert g == want or (g == 0 and want == 0), (fmt, a, b, g, want)


def test_exact_rounding_helper_on_known_ties():
    # 1 + 2^-8 is a bf16 tie between 1 and 1 + 2^-7: rounds to even (1)
    assert _round_exact(Fraction(1) + Fraction(1, 256), "bf16") == 1.0
    assert _round_exact(Fraction(1) + Fraction(3, 256), "bf16") == 1.0 + 2 ** -6
    # fp16: 2048 + 1 ties to 2048, 2048 + 3 to 2052
    assert _round_exact(Fraction(2049), "fp16") == 2048.0
    assert _round_exact(Fraction(2051), "fp16") == 2052.0
    assert _round_exact(Fraction(70000), "fp16") == float("inf")
