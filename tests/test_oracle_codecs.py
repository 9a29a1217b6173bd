"""Pins for the oracle's element codecs (bf16, fp16, E4M3, E2M1).

Each codec is checked against something other than itself: a library
conversion (torch / numpy), a brute-force nearest-value search over the
format's value table, or values fixed by the format definitions
(OCP 8-bit floating point E4M3 "fn"; OCP microscaling E2M1).
"""
import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


def _interesting_f32(n=20000):
    # random magnitudes over a wide exponent range, both signs, plus exact
    # ties of the 16-bit formats and boundaries
    e = RNG.uniform(-30, 20, n)
    v = (RNG.choice([-1.0, 1.0], n) * np.exp2(e)).astype(np.float32)
    ties = []
    for k in range(-20, 16):
        base = np.float32(2.0 ** k)
        ties += [base * (1 + 2 ** -8), base * (1 + 3 * 2 ** -8), base * (1 + 2 ** -11),
                 base * (1 + 3 * 2 ** -11), base * (1 + 5 * 2 ** -9)]
    special = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 65536.0, 2 ** -24, 2 ** -25,
               3 * 2 ** -25, 2 ** -14, 2 ** -15 * 1.5, 1e-45, 3.4e38, -3.4e38, 448.0, 464.0, 480.0]
    return np.concatenate([v, np.array(ties + special, dtype=np.float32)]).astype(np.float32)


def test_bf16_round_matches_torch():
    x = _interesting_f32()
    ours = oracle.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_decode_matches_torch():
    codes = np.arange(0, 65536, 7, dtype=np.uint16)
    codes = codes[(codes & 0x7f80) != 0x7f80]          # finite only
    ours = oracle.bf16_to_f32(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_f16_round_matches_numpy():
    x = _interesting_f32()
    ours = oracle.f16_round(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_decode_matches_numpy():
    codes = np.arange(0, 65536, dtype=np.uint16)
    codes = codes[(codes & 0x7c00) != 0x7c00]
    ours = oracle.f16_to_f32(codes)
    ref = codes.view(np.float16).astype(np.float32)
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------ E4M3 --

# Values fixed by the E4M3 ("fn") format definition: bias 7, 3 mantissa bits,
# no infinities, S.1111.111 is NaN.
E4M3_FACTS = {
    0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
    0x3c: 1.5, 0x40: 2.0, 0x77: 240.0, 0x7e: 448.0, 0x80: -0.0, 0xfe: -448.0,
}


def test_e4m3_decode_facts():
    for c, v in E4M3_FACTS.items():
        got = float(oracle.e4m3_decode([c])[0])
        assert got == v and np.signbit(got) == np.signbit(v), hex(c)
    assert np.isnan(oracle.e4m3_decode([0x7f])[0]) and np.isnan(oracle.e4m3_decode([0xff])[0])


def test_e4m3_decode_matches_torch():
    codes = np.array([c for c in range(256) if c & 0x7f != 0x7f], dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def _brute_nearest(x, table, max_code):
    """Nearest entry of a non-negative value table (index = code), ties to the
    code with an even last mantissa bit (even code), magnitudes beyond the
    largest finite value saturate.  Sign is carried separately."""
    ax = np.abs(x).astype(np.float64)
    d = np.abs(ax[:, None] - table[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = cand & ((np.arange(table.size)[None, :] & 1) == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    pick = np.where(ax >= table[max_code], max_code, pick)
    return pick


def test_e4m3_encode_brute_force_all_bf16_inputs():
    # every finite bf16 value times a few multipliers: covers every binade,
    # every tie, the subnormal band and saturation
    b = np.arange(0, 65536, dtype=np.uint32)
    b = b[((b >> 7) & 0xff) != 0xff]
    base = (b << 16).view(np.float32)
    for mult in (1.0, 0.5, 448.0 / 7.0, 2.0 ** -9):
        with np.errstate(over="ignore"):
            x = (base * np.float32(mult)).astype(np.float32)
        x = x[np.isfinite(x)]
        table = np.array([E4M3_positive(c) for c in range(0x7f)], dtype=np.float64)
        pick = _brute_nearest(x, table, 0x7e)
        expect = (pick | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)
        got = oracle.e4m3_encode(x)
        bad = np.nonzero(got != expect)[0]
        assert bad.size == 0, (mult, x[bad[:5]], got[bad[:5]], expect[bad[:5]])


def E4M3_positive(c):
    # table built from torch's decoder (a library routine), positive codes
    return float(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float())


def test_e4m3_encode_matches_torch_below_saturation():
    x = _interesting_f32()
    x = x[np.abs(x) < 448.0]
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_ties_to_even_examples():
    # midpoints between neighbouring codes: 1 + 1/16 (between 1 and 1.125) ->
    # 1.0 (even mantissa); 1 + 3/16 -> 1.25; 2^-10 (half the smallest
    # subnormal) -> 0; 3 * 2^-10 -> 2 * 2^-9; 232 (between 224 and 240) -> 224
    got = oracle.e4m3_encode([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 232.0])
    assert list(got) == [0x38, 0x3a, 0x00, 0x02, 0x76]


def test_e4m3_saturates_and_keeps_nan():
    got = oracle.e4m3_encode([448.0, 449.0, 464.0, 480.0, 1e30, np.inf, -np.inf, -500.0])
    assert list(got) == [0x7e, 0x7e, 0x7e, 0x7e, 0x7e, 0x7e, 0xfe, 0xfe]
    assert oracle.e4m3_encode([np.nan])[0] & 0x7f == 0x7f


# ------------------------------------------------------------------ E2M1 --

# The E2M1 value set fixed by the format (1 sign, 2 exponent bits with bias 1,
# 1 mantissa bit): codes 0..7.
E2M1_TABLE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def test_e2m1_decode_table():
    got = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    assert np.array_equal(got[:8], E2M1_TABLE.astype(np.float32))
    assert np.array_equal(got[8:], -E2M1_TABLE.astype(np.float32))
    assert np.signbit(got[8])


def test_e2m1_encode_brute_force():
    x = np.concatenate([
        np.linspace(-8, 8, 64001, dtype=np.float32),
        np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 6.0, 7.0, 1e30,
                  1e-30, -0.0, 0.0], dtype=np.float32),
        _interesting_f32(5000),
    ]).astype(np.float32)
    pick = _brute_nearest(x, E2M1_TABLE, 7)
    expect = (pick | np.where(np.signbit(x), 0x8, 0)).astype(np.uint8)
    got = oracle.e2m1_encode(x)
    bad = np.nonzero(got != expect)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], expect[bad[:5]])


def test_e2m1_ties_to_even_examples():
    # midpoints: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2.0, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    got = oracle.e2m1_encode([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert list(got) == [0x0, 0x2, 0x2, 0x4, 0x4, 0x6, 0x6]


@pytest.mark.parametrize("v,code", [(6.0, 0x7), (100.0, 0x7), (-6.5, 0xf), (-0.0, 0x8)])
def test_e2m1_saturation_and_sign(v, code):
    assert oracle.e2m1_encode([v])[0] == code
