"""Pins for the oracle's fused epilogue, quantisers, R-way sum and workspace
arithmetic.  Every expected value here comes from something other than the
oracle's own formula: a closed form, a special case that reduces to a library
routine (torch bf16 arithmetic, torch rms_norm), exact rational arithmetic on
tiny inputs, an invariant, or a worked value stated in the test.

Sources of the definitions (page title, function):
  TensorRT-LLM allReduceFusionKernels.cu: allreduce_sum (fp32 rank-order
    accumulation, one rounding), add128 / fused_op (residual add in the element
    type), rms_norm (acc / hidden_dim + eps, then x * s * gamma),
    is_neg_zero / push loop of allreduce_fusion_kernel_oneshot_lamport
    (-0.0 sentinel per 32-bit word), Workspace (region sizes).
  mscclpp allreduce.cu: vectorSum (plain element-wise R-way sum).
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from allreduce_residual_rmsnorm_gb300 import workloads as W

BF16 = oracle.BF16
FP16 = oracle.FP16
bits = W.bits


def bf(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def ulp_diff_bf16(a_bits, b_bits):
    """Distance in bf16 ulps between two arrays of bf16 bit patterns (finite)."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7fff), b & 0x7fff)
    return np.abs(key(a_bits) - key(b_bits))


def run(partials, residual, gamma, eps, dtype=BF16, acc=0):
    return oracle.fused(dtype, bits(partials), bits(residual), bits(gamma), eps, threads=2, acc=acc)


# -------------------------------------------------- residual path (steps 1-2)

@pytest.mark.parametrize("R", [1, 2, 3, 4, 8, 16])
def test_identical_partials_sum_equals_R_times_x(R):
    # R copies of x: every partial fp32 sum k*x has at most 12 significant
    # bits, so the rank sum is exactly R*x and the only rounding is the final
    # one -- the same as torch's single fp32 -> bf16 conversion of R*x.
    g = torch.Generator().manual_seed(R)
    T, H = 5, 72
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    res = torch.randn(T, H, generator=g).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    partials = x.unsqueeze(0).expand(R, T, H).contiguous()
    out, _, _ = run(partials, res, gamma, 1e-6)
    a = (x.float() * R).to(torch.bfloat16)
    expect = a + res        # torch CPU bf16 add: fp32 add, one RNE rounding
    assert np.array_equal(out, bits(expect))


def test_zero_partials_leave_residual_unchanged_and_norm_is_textbook():
    g = torch.Generator().manual_seed(7)
    R, T, H = 4, 6, 256
    res = torch.randn(T, H, generator=g).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    partials = torch.zeros(R, T, H, dtype=torch.bfloat16)
    out, nrm, _ = run(partials, res, gamma, 1e-6)
    assert np.array_equal(out, bits(res))
    ref = F.rms_norm(res.float(), (H,), gamma.float(), 1e-6).to(torch.bfloat16)
    d = ulp_diff_bf16(nrm, bits(ref))
    assert d.max() <= 1 and (d > 0).mean() < 0.01


@pytest.mark.parametrize("dtype", [BF16, FP16])
def test_single_rank_is_textbook_residual_rmsnorm(dtype):
    tdt = torch.bfloat16 if dtype == BF16 else torch.float16
    g = torch.Generator().manual_seed(11)
    T, H = 8, 512
    p = torch.randn(1, T, H, generator=g).to(tdt)
    res = torch.randn(T, H, generator=g).to(tdt)
    gamma = (1 + 0.1 * torch.randn(H, generator=g)).to(tdt)
    out, nrm, _ = run(p, res, gamma, 1e-6, dtype)
    y = p[0] + res          # torch CPU half/bf16 add: one rounding of the fp32 sum
    assert np.array_equal(out, bits(y))
    ref = F.rms_norm(y.float(), (H,), gamma.float(), 1e-6).to(tdt)
    if dtype == BF16:
        d = ulp_diff_bf16(nrm, bits(ref))
    else:
        d = np.abs(nrm.astype(np.int32) - bits(ref).astype(np.int32))
    assert d.max() <= 1 and (d > 0).mean() < 0.01


def test_rank_order_fp32_accumulation_worked_value():
    # Partials 2^24, 1, -2^24 (all exact in bf16).  In fp32, rank order:
    # 2^24 + 1 = 16777217 is not representable and rounds (tie, to even) to
    # 2^24; adding -2^24 gives 0.  Any other order, or fp64, gives 1.
    P = torch.zeros(3, 1, 8, dtype=torch.bfloat16)
    P[0] = bf(2.0 ** 24)
    P[1] = bf(1.0)
    P[2] = bf(-(2.0 ** 24))
    res = bf(np.full((1, 8), 0.5))
    gamma = bf(np.ones(8))
    out, _, _ = run(P, res, gamma, 1e-6)
    assert np.array_equal(out, bits(res))                 # y = 0 + 0.5


def test_rank_sum_is_rounded_before_residual_add_worked_value():
    # s = 1 + 2^-8 is exactly half way between bf16 neighbours 1 and 1 + 2^-7:
    # ties-to-even gives a = 1.  Then 1 + 2^-8 again rounds to 1.
    # Adding the residual to the unrounded sum would give 1 + 2^-7 exactly.
    P = torch.zeros(2, 1, 8, dtype=torch.bfloat16)
    P[0] = bf(1.0)
    P[1] = bf(2.0 ** -8)
    res = bf(np.full((1, 8), 2.0 ** -8))
    gamma = bf(np.ones(8))
    out, _, _ = run(P, res, gamma, 1e-6)
    assert np.array_equal(out, bits(bf(np.ones((1, 8)))))


# ------------------------------------- element-type accumulation (variant)

def test_element_type_accumulation_worked_value():
    # Partials 1, 2^-8, 2^-8.  fp32 accumulation: 1 + 2^-8 + 2^-8 = 1 + 2^-7
    # exactly, one rounding keeps it.  bf16 accumulation: 1 + 2^-8 is a tie
    # between bf16 neighbours 1 and 1 + 2^-7 and rounds to even (1), twice.
    P = torch.zeros(3, 1, 8, dtype=torch.bfloat16)
    P[0] = bf(1.0)
    P[1] = bf(2.0 ** -8)
    P[2] = bf(2.0 ** -8)
    res = torch.zeros(1, 8, dtype=torch.bfloat16)
    gamma = bf(np.ones(8))
    out32, _, _ = run(P, res, gamma, 1e-6, acc=0)
    out16, _, _ = run(P, res, gamma, 1e-6, acc=1)
    assert np.all(out32 == bits(bf(1.0 + 2.0 ** -7)).item())
    assert np.all(out16 == bits(bf(1.0)).item())


@pytest.mark.parametrize("dtype", [BF16, FP16])
def test_element_type_accumulation_is_chained_library_adds(dtype):
    # torch CPU adds of two bf16 / fp16 tensors round once per addition: the
    # chained sum p0 + p1 + ... is the element-type accumulation
    tdt = torch.bfloat16 if dtype == BF16 else torch.float16
    g = torch.Generator().manual_seed(31)
    R, T, H = 6, 4, 256
    P = torch.randn(R, T, H, generator=g).to(tdt)
    res = torch.randn(T, H, generator=g).to(tdt)
    gamma = (1 + 0.1 * torch.randn(H, generator=g)).to(tdt)
    a = P[0].clone()
    for r in range(1, R):
        a = a + P[r]
    out, _, _ = run(P, res, gamma, 1e-6, dtype, acc=1)
    assert np.array_equal(out, bits(a + res))


def test_vector_sum_element_type_accumulation():
    g = torch.Generator().manual_seed(2)
    x = (torch.rand(8, 5003, generator=g) * 2 - 1).to(torch.float16)
    a = x[0].clone()
    for r in range(1, 8):
        a = a + x[r]
    assert np.array_equal(oracle.vector_sum(FP16, bits(x), threads=2, acc=1), bits(a))


@pytest.mark.parametrize("dtype", [BF16, FP16])
def test_vector_sum_element_type_special_values_are_chained_library_adds(dtype):
    # signed zeros, subnormals, ties, the largest finite values, infinities and
    # NaN: the per-add rounding (with overflow to infinity, -0 + -0 = -0 and
    # +0 + -0 = +0) follows torch's chained 16-bit adds; NaN only in position
    tdt = torch.bfloat16 if dtype == BF16 else torch.float16
    fin = torch.finfo(tdt)
    pool = torch.tensor([0.0, -0.0, fin.smallest_normal, fin.smallest_normal / 4, -fin.tiny / 8,
                         1.0, 1.0 + fin.eps, fin.eps / 2, -fin.eps / 2, fin.max, -fin.max,
                         fin.max / 2, float("inf"), float("-inf"), float("nan"), 0.75],
                        dtype=torch.float32).to(tdt)
    g = torch.Generator().manual_seed(5)
    R, N = 5, 6000
    x = pool[torch.randint(0, len(pool), (R, N), generator=g)]
    a = x[0].clone()
    for r in range(1, R):
        a = a + x[r]
    got = oracle.vector_sum(dtype, bits(x), threads=2, acc=1)
    nan = torch.isnan(a).numpy()
    assert nan.any() and torch.isinf(a).any()
    got_t = torch.from_numpy(got.view(np.int16)).view(tdt)
    assert np.array_equal(torch.isnan(got_t).numpy(), nan)
    assert np.array_equal(got[~nan], bits(a)[~nan])


# ----------------------------------------------------- RMSNorm (steps 3-5)

@pytest.mark.parametrize("H,c", [(8, 1.0), (512, -0.25), (7168, 4.0), (4096, -2.0 ** -6)])
def test_constant_power_of_two_row_normalises_to_signed_gamma_exactly(H, c):
    # y_h = c = +-2^k and eps = 0: ss = H c^2, ss / H = c^2, sqrt = |c|, all
    # exact, so rstd = 1/|c| exactly and (c * rstd) * gamma = sign(c) * gamma.
    g = torch.Generator().manual_seed(H)
    gamma = (1 + 0.3 * torch.randn(H, generator=g)).to(torch.bfloat16)
    P = torch.zeros(2, 1, H, dtype=torch.bfloat16)
    res = bf(np.full((1, H), c))
    _, nrm, rstd = run(P, res, gamma, 0.0)
    assert rstd[0] == np.float32(1.0 / abs(c))
    expect = gamma if c > 0 else -gamma
    assert np.array_equal(nrm[0], bits(expect))


def test_constant_row_with_eps_closed_form():
    # rstd = 1 / sqrt(c^2 + eps): for c = 1 and eps = 0.5625 that is exactly
    # 1 / 1.25 = 0.8 (rounded once to fp32), n = rnd((c*0.8f)*gamma).
    H = 64
    gamma = bf(np.linspace(-2, 2, H))
    P = torch.zeros(1, 1, H, dtype=torch.bfloat16)
    res = bf(np.ones((1, H)))
    _, nrm, rstd = run(P, res, gamma, 0.5625)
    assert rstd[0] == np.float32(0.8)
    expect = (torch.full((H,), float(np.float32(0.8))) * gamma.float()).to(torch.bfloat16)
    assert np.array_equal(nrm[0], bits(expect))


def test_exact_rational_brute_force_tiny():
    # Dyadic inputs (multiples of 1/16 in [-4, 4]) keep every fp32 rank sum and
    # residual add exact, so y is one rounding of an exact rational.  ss, the
    # mean, eps and the inverse square root are then done exactly / in fp64.
    rng = np.random.default_rng(5)
    for trial in range(20):
        R = int(rng.integers(1, 5))
        T = int(rng.integers(1, 4))
        H = 8 * int(rng.integers(1, 5))
        P = rng.integers(-64, 65, (R, T, H)) / 16.0
        X = rng.integers(-64, 65, (T, H)) / 16.0
        G = rng.integers(8, 24, H) / 16.0
        eps = 1e-3
        Pt, Xt, Gt = bf(P), bf(X), bf(G)
        assert np.array_equal(Pt.float().numpy(), P) and np.array_equal(Xt.float().numpy(), X)
        out, nrm, _ = run(Pt, Xt, Gt, eps)
        for t in range(T):
            s = [sum(Fraction(float(P[r, t, h])) for r in range(R)) for h in range(H)]
            a = [float(bf(float(v))) for v in s]          # exact rational -> one rounding
            y = [float(bf(ai + float(X[t, h]))) for h, ai in enumerate(a)]
            assert np.array_equal(out[t], bits(bf(y)))
            ss = sum(Fraction(v) ** 2 for v in y)
            rstd = 1.0 / math.sqrt(float(ss / H) + eps)
            n = bf([yi * rstd * float(G[h]) for h, yi in enumerate(y)])
            d = ulp_diff_bf16(nrm[t], bits(n))
            assert d.max() <= 1, (trial, t)


# Exact rational arithmetic with explicit round-to-nearest-even, for pins that
# must see every fp32 rounding of the normalisation in the pages' order.
F32_BITS, F16_BITS, BF16_BITS = 23, 10, 7


def _rnd(q, mbits):
    """q rounded to nearest (ties to even) with `mbits` fraction bits (normal range)."""
    if q == 0:
        return Fraction(0)
    sgn = -1 if q < 0 else 1
    a = abs(Fraction(q))
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    quantum = Fraction(2) ** (e - mbits)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sgn * fl * quantum


def _sqrt_rnd32(q):
    """Correctly rounded fp32 square root of a positive rational."""
    q = Fraction(q)
    e = (q.numerator.bit_length() - q.denominator.bit_length()) // 2
    while Fraction(4) ** e > q:
        e -= 1
    while Fraction(4) ** (e + 1) <= q:
        e += 1
    quantum = Fraction(2) ** (e - F32_BITS)
    n = q / (quantum * quantum)                  # sqrt(n) in [2^23, 2^24)
    fl = math.isqrt(n.numerator // n.denominator)
    mid = Fraction(2 * fl + 1, 2) ** 2
    if n > mid or (n == mid and fl % 2 == 1):
        fl += 1
    return fl * quantum


def _exact_row(P, x, g, eps, mbits):
    """One row in the pages' order, every step rounded as stated: fp32 rank
    sum, rounded to D; fp32 residual add, rounded to D; sum of squares exact,
    rounded to fp32 once; mean = ss / H; + eps; sqrt; 1 / sqrt (each fp32);
    n = ((y * rstd) * gamma) left to right in fp32, rounded to D."""
    H = len(x)
    eps32 = _rnd(Fraction(eps), F32_BITS)
    y = []
    for h in range(H):
        s = Fraction(float(P[0][h]))
        for r in range(1, len(P)):
            s = _rnd(s + Fraction(float(P[r][h])), F32_BITS)
        a = _rnd(s, mbits)
        y.append(_rnd(_rnd(a + Fraction(float(x[h])), F32_BITS), mbits))
    ss32 = _rnd(sum(v * v for v in y), F32_BITS)
    ms = _rnd(ss32 / H, F32_BITS)
    v = _rnd(ms + eps32, F32_BITS)
    rstd = _rnd(1 / _sqrt_rnd32(v), F32_BITS)
    n = [_rnd(_rnd(_rnd(yh * rstd, F32_BITS) * Fraction(float(g[h])), F32_BITS), mbits)
         for h, yh in enumerate(y)]
    return y, rstd, n


@pytest.mark.parametrize("dtype", [BF16, FP16])
def test_rows_follow_the_pages_rounding_order_exactly(dtype):
    # Random rows (hidden sizes that are not powers of two, so dividing by H
    # rounds): residual_out, the fp32 rstd and norm_out equal the exact
    # step-by-step evaluation bit for bit.
    tdt = torch.bfloat16 if dtype == BF16 else torch.float16
    mbits = BF16_BITS if dtype == BF16 else F16_BITS
    g = torch.Generator().manual_seed(21 + dtype)
    for R, H, eps in ((1, 24, 1e-6), (2, 40, 1e-5), (3, 56, 0.01), (2, 200, 0.3), (4, 96, 1e-6)):
        T = 3
        P = torch.randn(R, T, H, generator=g).to(tdt)
        X = torch.randn(T, H, generator=g).to(tdt)
        G = (1 + 0.3 * torch.randn(H, generator=g)).to(tdt)
        res, nrm, rstd = run(P, X, G, eps, dtype)
        for t in range(T):
            y, r32, n = _exact_row(P[:, t].float().numpy(), X[t].float().numpy(),
                                   G.float().numpy(), eps, mbits)
            assert np.array_equal(res[t], bits(torch.tensor([float(v) for v in y]).to(tdt)))
            assert Fraction(float(rstd[t])) == r32, (R, H, t)
            assert np.array_equal(nrm[t], bits(torch.tensor([float(v) for v in n]).to(tdt)))


def test_normalisation_multiplies_rstd_before_gamma():
    # A constant fp16 row where the two product orders round to different
    # fp16 values: y = 1.8515625 (all 8 elements), eps = 0.0399933..., gamma_0
    # = 0.35888671875.  (y * rstd) * gamma gives 0.356689453125; (y * gamma)
    # * rstd would give 0.3569335... (one fp16 step higher).
    c, eps, g0 = 1.8515625, 0.03999330475926399, 0.35888671875
    H = 8
    P = torch.zeros(1, 1, H, dtype=torch.float16)
    X = torch.full((1, H), c, dtype=torch.float16)
    G = torch.ones(H, dtype=torch.float16)
    G[0] = g0
    _, nrm, _ = run(P, X, G, eps, FP16)
    _, rstd, n = _exact_row(P[:, 0].float().numpy(), X[0].float().numpy(), G.float().numpy(),
                            eps, F16_BITS)
    other = _rnd(_rnd(_rnd(Fraction(c) * Fraction(g0), F32_BITS) * rstd, F32_BITS), F16_BITS)
    assert n[0] == Fraction(0.356689453125) and other != n[0]
    assert nrm[0][0] == bits(torch.tensor([0.356689453125], dtype=torch.float16))[0]


def test_norm_invariant_locates_eps_and_mean():
    # mean_h (n_h / gamma_h)^2 = ms / (ms + eps) up to bf16 rounding; a large
    # eps makes the factor far from 1 so a misplaced eps or a wrong divisor
    # for the mean shows up.
    g = torch.Generator().manual_seed(3)
    R, T, H = 3, 4, 1024
    P = torch.randn(R, T, H, generator=g).to(torch.bfloat16)
    X = torch.randn(T, H, generator=g).to(torch.bfloat16)
    G = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    eps = 2.0
    out, nrm, _ = run(P, X, G, eps)
    y = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).double()
    n = torch.from_numpy(nrm.view(np.int16)).view(torch.bfloat16).double()
    ms = (y ** 2).mean(dim=1)
    lhs = ((n / G.double()) ** 2).mean(dim=1)
    rhs = ms / (ms + eps)
    assert torch.allclose(lhs, rhs, rtol=6e-3)


# ------------------------------------------------------- sentinel (staging)

def test_lamport_flip_only_touches_negative_zero_words():
    # little-endian pairs: (lo=+0, hi=-0) is the word 0x80000000 -> rewritten;
    # (lo=-0, hi=+0) is 0x00008000 -> kept; other words kept.
    a = np.array([0x0000, 0x8000, 0x8000, 0x0000, 0x8000, 0x8000, 0x3f80, 0x8000],
                 dtype=np.uint16)
    got = oracle.lamport_flip(a)
    assert list(got) == [0x0000, 0x0000, 0x8000, 0x0000, 0x8000, 0x8000, 0x3f80, 0x8000]


# ---------------------------------------------------------- FP8 per-tensor

def _norm_of_random(T=16, H=256, seed=9):
    g = torch.Generator().manual_seed(seed)
    P = torch.randn(4, T, H, generator=g).to(torch.bfloat16)
    X = torch.randn(T, H, generator=g).to(torch.bfloat16)
    G = (1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    _, nrm, _ = run(P, X, G, 1e-6)
    return nrm


def test_fp8_multiplier_is_the_reciprocal_of_the_rounded_scale():
    # The configuration supplies scale = amax / 448 and the kernel multiplies
    # by its inverse: two fp32 roundings, rnd(1 / rnd(amax / 448)), which for
    # some amax differs from the single rounding of 448 / amax.
    amaxes = torch.linspace(0.01, 300.0, 3001).to(torch.bfloat16).float().unique().numpy()
    differs = 0
    for a in amaxes:
        want = _rnd(1 / _rnd(Fraction(float(a)) / 448, F32_BITS), F32_BITS)
        assert Fraction(float(oracle.fp8_inv_scale(float(a)))) == want, a
        differs += want != _rnd(Fraction(448) / Fraction(float(a)), F32_BITS)
    assert differs > 0
    assert oracle.fp8_inv_scale(0.0) == 1.0


def test_fp8_amax_element_maps_to_448_and_roundtrip_bound():
    nrm = _norm_of_random()
    amax = oracle.amax(BF16, nrm)
    n = torch.from_numpy(nrm.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert amax == np.abs(n).max()
    inv = oracle.fp8_inv_scale(amax)
    q = oracle.quant_fp8(BF16, nrm, inv)
    at_max = np.abs(n) == amax
    assert np.all((q[at_max] & 0x7f) == 0x7e)
    scale = np.float32(amax / 448.0)
    dq = oracle.e4m3_decode(q) * scale
    normal = np.abs(n) * inv >= 2.0 ** -6
    assert np.all(np.abs(dq - n)[normal] <= 2.0 ** -4 * np.abs(n)[normal] * (1 + 1e-6))
    assert np.all(np.abs(dq - n)[~normal] <= 2.0 ** -10 * scale * (1 + 1e-6))
    # sign and monotonicity
    assert np.all(np.signbit(n[n != 0]) == ((q[n != 0] & 0x80) != 0))


@pytest.mark.parametrize("dtype", [BF16, FP16])
def test_amax_is_the_largest_magnitude_on_either_side(dtype):
    # the per-tensor scale must cover the most negative element too
    tdt = torch.bfloat16 if dtype == BF16 else torch.float16
    x = torch.tensor([[0.5, -3.5, 2.0, -0.0], [1.25, 0.0, -1.0, 3.0]], dtype=tdt)
    assert oracle.amax(dtype, bits(x)) == 3.5
    assert oracle.amax(dtype, bits(-x)) == 3.5
    assert oracle.amax(dtype, bits(torch.zeros(3, 8, dtype=tdt))) == 0.0


# ------------------------------------------------------------------ NVFP4

def test_scales_of_an_all_zero_tensor_are_finite():
    # an all-zero tensor (amax = 0) must not produce an infinite multiplier
    assert oracle.fp8_inv_scale(0.0) == 1.0
    assert oracle.nvfp4_global_scale(0.0) == 1.0
    z = np.zeros((2, 32), np.uint16)
    assert np.all(oracle.quant_fp8(BF16, z, oracle.fp8_inv_scale(0.0)) == 0)
    q, s = oracle.quant_nvfp4(BF16, z, oracle.nvfp4_global_scale(0.0))
    assert np.all(q == 0) and np.all(s == 0)


def test_nvfp4_zero_block_and_max_element():
    H = 64
    n = np.zeros((2, H), np.uint16)
    vals = np.linspace(-3, 5, 16)
    n[0, 16:32] = bits(bf(vals))
    n[1, 48:64] = bits(bf(-vals))
    gs = oracle.nvfp4_global_scale(5.0)
    q, s = oracle.quant_nvfp4(BF16, n, gs)
    # all-zero blocks: scale 0 and every code 0
    assert s[0, 0] == 0 and s[0, 2] == 0 and s[1, 0] == 0
    assert np.all(q[0, 0:8] == 0) and np.all(q[1, 0:16] == 0)
    # the element holding the block maximum encodes to +-6 (code 7 / 15)
    codes0 = np.stack([q[0, 8:16] & 0xf, q[0, 8:16] >> 4], 1).ravel()
    assert codes0[15] == 0x7
    codes1 = np.stack([q[1, 24:32] & 0xf, q[1, 24:32] >> 4], 1).ravel()
    assert codes1[15] == 0xf


@pytest.mark.parametrize("dtype", [BF16, FP16])
def test_nvfp4_global_scale_puts_the_amax_block_on_the_largest_scale(dtype):
    # The stated global-scale convention (the tensor amax maps onto 448 x 6,
    # the largest E4M3 block scale times the largest E2M1 value) is a reading,
    # not on the pages; this holds the oracle to it: the block holding the
    # amax gets scale byte 0x7E (448) and its largest element the code +-6.
    nrm = _norm_of_random(seed=17) if dtype == BF16 else bits(
        torch.from_numpy(_norm_of_random(seed=17).view(np.int16)).view(torch.bfloat16)
        .float().to(torch.float16))
    tdt = torch.bfloat16 if dtype == BF16 else torch.float16
    n = torch.from_numpy(nrm.view(np.int16)).view(tdt).float().numpy()
    amax = oracle.amax(dtype, nrm)
    q, sf = oracle.quant_nvfp4(dtype, nrm, oracle.nvfp4_global_scale(amax))
    t, h = np.argwhere(np.abs(n) == amax)[0]
    assert sf[t, h // 16] == 0x7E
    code = (q[t, h // 2] >> (4 * (h % 2))) & 0xF
    assert code == (0xF if n[t, h] < 0 else 0x7)
    # no block scale exceeds it
    assert sf.max() <= 0x7E


def test_nvfp4_nibble_order_convention():
    # Stated convention: element 2k in the low nibble of byte k.
    n = np.zeros((1, 16), np.uint16)
    n[0, 0] = bits(bf(6.0)).item()       # first element large, second zero
    gs = oracle.nvfp4_global_scale(6.0)
    q, _ = oracle.quant_nvfp4(BF16, n, gs)
    assert q[0, 0] == 0x07


def test_nvfp4_roundtrip_bound_random():
    nrm = _norm_of_random(T=32, H=512, seed=21)
    amax = oracle.amax(BF16, nrm)
    gs = oracle.nvfp4_global_scale(amax)
    q, s = oracle.quant_nvfp4(BF16, nrm, gs)
    n = torch.from_numpy(nrm.view(np.int16)).view(torch.bfloat16).float().numpy()
    codes = np.stack([q & 0xf, q >> 4], -1).reshape(n.shape)
    dec = oracle.e4m3_decode(s)                                   # [T, H/16]
    dq = oracle.e2m1_decode(codes) * np.repeat(dec, 16, axis=1) / gs
    err = np.abs(dq - n)
    bmax = np.repeat(np.abs(n).reshape(n.shape[0], -1, 16).max(-1), 16, axis=1)
    bound = np.repeat(dec, 16, axis=1) / gs + bmax * 2.0 ** -4
    assert np.all(err <= bound * (1 + 1e-5))
    # every block's maximum element encodes to +-6
    blk = np.abs(n).reshape(n.shape[0], -1, 16)
    cblk = codes.reshape(n.shape[0], -1, 16) & 0x7
    arg = blk.argmax(-1)
    top = np.take_along_axis(cblk, arg[..., None], -1)[..., 0]
    nz = blk.max(-1) > 0
    assert np.all(top[nz] == 7)


# ------------------------------------------------------------- R-way sum

def test_vector_sum_closed_form_and_fp64():
    R, N = 8, 4099
    ins = np.full((R, N), bits(torch.tensor([0.125], dtype=torch.float16)).item(), np.uint16)
    out = oracle.vector_sum(FP16, ins, threads=2)
    assert np.all(out == bits(torch.tensor([1.0], dtype=torch.float16)).item())   # 8 * 0.125
    g = torch.Generator().manual_seed(0)
    x = (torch.rand(R, N, generator=g) * 2 - 1).to(torch.float16)
    out = oracle.vector_sum(FP16, bits(x), threads=2)
    ref = x.double().sum(0).to(torch.float16)    # fp64 sum, one rounding (fp64->fp16)
    mism = np.count_nonzero(out != bits(ref))
    assert mism <= N // 1000, mism


# ------------------------------------------------------ workspace / state

def test_workspace_sizes_match_page_formula_golden():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "workspace_sizes.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert rows
    for R, maxT, H, elem, oneshot, flags, buf, flg, slot, lam in rows:
        got = oracle.workspace_sizes(int(R), int(maxT), int(H), int(elem), int(oneshot), int(flags))
        assert got == (int(buf), int(flg), int(slot), int(lam))


def test_lamport_state_cycles():
    flag, clear = 0, 0
    seen = []
    for k in range(7):
        flag, clear, rd, cl = oracle.lamport_step(flag, clear, 2, 16, 512)
        seen.append((rd, cl, flag))
        assert clear == 2 * 16 * 512
    assert seen[:4] == [(0, 2, 1), (1, 0, 2), (2, 1, 0), (0, 2, 1)]


# ------------------------------------------------- NVFP4 scale tile layout

@pytest.mark.parametrize("T,KB", [(1, 1), (128, 4), (200, 28), (257, 448), (300, 5)])
def test_swizzled_scales_are_a_tile_permutation(T, KB):
    # every (row, block) lands on its own byte; whole 128 x 4 tiles are
    # contiguous 512-byte ranges; the padded buffer holds exactly the tiles
    lin = np.arange(T * KB, dtype=np.int64)
    out = oracle.swizzle_scales(np.ones((T, KB), np.uint8))
    Tp, KBp = (T + 127) // 128 * 128, (KB + 3) // 4 * 4
    assert out.size == Tp * KBp
    # a distinct 24-bit tag per cell, carried in three byte planes
    planes = [oracle.swizzle_scales(((lin >> (8 * i)) & 0xff).astype(np.uint8).reshape(T, KB))
              for i in range(3)]
    present = oracle.swizzle_scales(np.ones((T, KB), np.uint8))
    tags = sum(p.astype(np.int64) << (8 * i) for i, p in enumerate(planes))
    assert present.sum() == T * KB
    assert np.array_equal(np.sort(tags[present == 1]), lin)
    # tile (rb, kb) of the linear matrix occupies bytes [512 t, 512 t + 512)
    ktiles = KBp // 4
    for rb in range((T + 127) // 128):
        for kt in range(ktiles):
            t = rb * ktiles + kt
            rows = np.arange(rb * 128, min(T, rb * 128 + 128))
            cols = np.arange(kt * 4, min(KB, kt * 4 + 4))
            if rows.size == 0 or cols.size == 0:
                continue
            cell = (rows[:, None] * KB + cols[None, :]).ravel()
            got = tags[t * 512:(t + 1) * 512][present[t * 512:(t + 1) * 512] == 1]
            assert np.array_equal(np.sort(got), np.sort(cell))


def test_swizzled_scales_worked_positions():
    # within a tile: row 0 block 0 -> 0, row 1 -> 16, row 32 -> 4, row 96 block 3 -> 15,
    # row 31 block 2 -> 31*16 + 2; next tile along the blocks starts at 512
    ids = np.zeros((128, 8), np.uint8)
    ids[0, 0], ids[1, 0], ids[32, 0], ids[96, 3], ids[31, 2], ids[0, 4] = 1, 2, 3, 4, 5, 6
    out = oracle.swizzle_scales(ids)
    assert (out[0], out[16], out[4], out[15], out[31 * 16 + 2], out[512]) == (1, 2, 3, 4, 5, 6)


# ------------------------------------------------------ fp32 element type

def run32(partials, residual, gamma, eps):
    return oracle.fused_f32(partials.numpy(), residual.numpy(), gamma.numpy(), eps, threads=2)


@pytest.mark.parametrize("R", [1, 2, 4, 8, 16])
def test_f32_identical_partials_power_of_two_ranks(R):
    # k * x is exact in fp32 for k <= R (powers of two and small multiples of
    # a value with a short significand): x drawn with 16 significant bits
    g = torch.Generator().manual_seed(R)
    x = (torch.randn(4, 64, generator=g) * 1024).round() / 1024
    res = torch.randn(4, 64, generator=g)
    gamma = 1 + 0.1 * torch.randn(64, generator=g)
    out, _, _ = run32(x.unsqueeze(0).expand(R, 4, 64).contiguous(), res, gamma, 1e-6)
    assert np.array_equal(out, (x * R + res).numpy())        # torch fp32: one rounding


def test_f32_zero_partials_and_textbook_rmsnorm():
    g = torch.Generator().manual_seed(8)
    res = torch.randn(6, 512, generator=g)
    gamma = 1 + 0.1 * torch.randn(512, generator=g)
    out, nrm, _ = run32(torch.zeros(3, 6, 512), res, gamma, 1e-5)
    assert np.array_equal(out, res.numpy())
    ref = F.rms_norm(res.double(), (512,), gamma.double(), 1e-5).float().numpy()
    assert np.allclose(nrm, ref, rtol=2e-6, atol=1e-7)


def test_f32_rank_order_worked_value():
    P = torch.zeros(3, 1, 8)
    P[0], P[1], P[2] = 2.0 ** 24, 1.0, -(2.0 ** 24)
    out, _, _ = run32(P, torch.full((1, 8), 0.5), torch.ones(8), 1e-6)
    assert np.all(out == np.float32(0.5))                    # (2^24 + 1) rounds to 2^24


def test_f32_constant_power_of_two_row():
    g = torch.Generator().manual_seed(9)
    gamma = 1 + 0.3 * torch.randn(4096, generator=g)
    _, nrm, rstd = run32(torch.zeros(2, 1, 4096), torch.full((1, 4096), -0.125), gamma, 0.0)
    assert rstd[0] == np.float32(8.0)
    assert np.array_equal(nrm[0], (-gamma).numpy())


def test_f32_quantisers_match_the_16_bit_ones_on_representable_values():
    # n values that are exact bf16 numbers give the same codes through the
    # fp32 and the bf16 entry points
    g = torch.Generator().manual_seed(10)
    n16 = (torch.randn(8, 256, generator=g) * 3).to(torch.bfloat16)
    n32 = n16.float().numpy()
    assert np.array_equal(oracle.quant_fp8_f32(n32, 17.5), oracle.quant_fp8(BF16, bits(n16), 17.5))
    q32, s32 = oracle.quant_nvfp4_f32(n32, 300.0)
    q16, s16 = oracle.quant_nvfp4(BF16, bits(n16), 300.0)
    assert np.array_equal(q32, q16) and np.array_equal(s32, s16)
    assert oracle.amax_f32(n32) == oracle.amax(BF16, bits(n16))
    # the largest magnitude may sit on the negative side
    assert oracle.amax_f32(np.array([[0.5, -3.5, 2.0, -0.0]], np.float32)) == 3.5


def test_f32_vector_sum():
    x = torch.full((8, 1001), 0.125)
    assert np.all(oracle.vector_sum_f32(x.numpy()) == 1.0)
    g = torch.Generator().manual_seed(4)
    y = torch.rand(4, 999, generator=g) * 2 - 1
    ref = ((y[0] + y[1]) + y[2]) + y[3]                      # torch fp32, rank order
    assert np.array_equal(oracle.vector_sum_f32(y.numpy()), ref.numpy())


def test_f32_constant_row_with_eps_closed_form():
    # y = 0.75 everywhere, eps = 0.4375: mean square + eps = 1 exactly, so
    # rstd = 1 and norm_out = 0.75 * gamma exactly
    g = torch.Generator().manual_seed(12)
    gamma = 1 + 0.2 * torch.randn(1024, generator=g)
    P = torch.zeros(4, 3, 1024)
    P[1] = 0.5
    out, nrm, rstd = run32(P, torch.full((3, 1024), 0.25), gamma, 0.4375)
    assert np.all(out == np.float32(0.75)) and np.all(rstd == np.float32(1.0))
    assert np.array_equal(nrm, (0.75 * gamma).expand(3, 1024).numpy())


def test_f32_rows_follow_the_pages_rounding_order_exactly():
    # fp32 elements: every rounding of the row is an fp32 rounding and none is
    # hidden by a final 16-bit one, so residual_out, rstd and norm_out are
    # compared bit for bit with the exact step-by-step evaluation
    g = torch.Generator().manual_seed(31)
    for R, H, eps in ((1, 24, 1e-6), (2, 40, 1e-5), (3, 200, 0.25), (4, 56, 1e-6)):
        T = 3
        P = torch.randn(R, T, H, generator=g)
        X = torch.randn(T, H, generator=g)
        G = 1 + 0.3 * torch.randn(H, generator=g)
        res, nrm, rstd = run32(P, X, G, eps)
        for t in range(T):
            y, r32, n = _exact_row(P[:, t].numpy(), X[t].numpy(), G.numpy(), eps, F32_BITS)
            assert [Fraction(float(v)) for v in res[t]] == y, (R, H, t)
            assert Fraction(float(rstd[t])) == r32, (R, H, t)
            assert [Fraction(float(v)) for v in nrm[t]] == n, (R, H, t)


def test_f32_norm_is_rmsnorm_of_residual_out():
    # with nonzero partials the normalised row is the textbook RMSNorm of the
    # updated residual (computed here in fp64 by torch)
    g = torch.Generator().manual_seed(13)
    P = torch.randn(4, 5, 768, generator=g)
    res = torch.randn(5, 768, generator=g)
    gamma = 1 + 0.1 * torch.randn(768, generator=g)
    out, nrm, _ = run32(P, res, gamma, 1e-6)
    ref = F.rms_norm(torch.from_numpy(out).double(), (768,), gamma.double(), 1e-6).float().numpy()
    assert np.allclose(nrm, ref, rtol=2e-6, atol=1e-7)
