"""Pins of the oracle's number formats and matrix-vector products to what the pages and
the mathematics fix (kimi-k3-in-c, section 4 "Reduction one" and section 5)."""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))


def e2m1_closed_form(code):
    """E2M1 from its bit fields: sign, 2 exponent bits (bias 1), 1 mantissa bit; the
    exponent-0 codes are subnormal (0.m x 2^0)."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = (m * 0.5) if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return -mag if s else mag


def test_e2m1_matches_printed_table():
    want = GOLD["e2m1_lut"]["values"]
    got = [oracle.e2m1(c) for c in range(16)]
    assert got == want
    # signed zero is kept (code 8 is -0.0)
    assert math.copysign(1.0, oracle.e2m1(8)) == -1.0


def test_e2m1_matches_bitfield_definition():
    for c in range(16):
        assert oracle.e2m1(c) == e2m1_closed_form(c)


def test_e8m0_closed_form_all_bytes():
    for b in range(256):
        want = 0.0 if b == 255 else math.ldexp(1.0, b - 127)
        assert oracle.e8m0(b) == want
    assert oracle.e8m0(127) == 1.0
    # byte 0 is 2^-127: a float subnormal, kept (no flush to zero)
    assert np.float32(oracle.e8m0(0)) == np.float32(2.0 ** -127) and oracle.e8m0(0) > 0


def test_bf16_widening_is_a_shift_and_rounding_is_nearest_even():
    bits = np.array([0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x4049], dtype=np.uint16)
    f = oracle.bf16_to_f32(bits)
    assert f[0] == 1.0 and f[1] == -1.0
    assert f[4] == np.float32(3.140625)
    # round trip of every representable value
    assert (oracle.f32_to_bf16(f) == bits).all()
    # ties to even: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> 1 (even mantissa)
    assert oracle.f32_to_bf16(np.float32(1.0 + 2.0 ** -8))[()] == 0x3F80
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6 -> the even one, 1 + 2^-6
    assert oracle.f32_to_bf16(np.float32(1.0 + 3 * 2.0 ** -8))[()] == 0x3F82
    assert oracle.f32_to_bf16(np.float32(1.0 + 2.0 ** -8 + 2.0 ** -20))[()] == 0x3F81


def test_nibble_order_low_nibble_is_even_column():
    # one row of 32 columns: byte k holds columns 2k (low nibble) and 2k+1 (high nibble)
    packed = np.zeros((1, 16), dtype=np.uint8)
    packed[0, 0] = 0x71      # col 0 <- code 1 (0.5), col 1 <- code 7 (6.0)
    packed[0, 3] = 0x9E      # col 6 <- code 14 (-4.0), col 7 <- code 9 (-0.5)
    scales = np.array([[127]], dtype=np.uint8)
    w = oracle.dequant_mxfp4(packed, scales, 1, 32)
    assert w[0, 0] == 0.5 and w[0, 1] == 6.0 and w[0, 6] == -4.0 and w[0, 7] == -0.5
    # through the product: x = e_1 picks column 1
    x = np.zeros(32, dtype=np.float32)
    x[1] = 1.0
    assert oracle.mxfp4_gemv(packed, scales, 1, 32, x)[0] == 6.0


def swapped_nibble_dequant(packed, scales, rows, cols):
    """A planted mistake (high nibble read as the even column), used only to show that
    the position tests catch it."""
    sw = ((packed & 0x0F) << 4) | (packed >> 4)
    return oracle.dequant_mxfp4(sw.astype(np.uint8), scales, rows, cols)


def test_swapped_nibbles_have_same_statistics_but_fail_the_position_pin():
    rng = np.random.default_rng(0)
    packed = rng.integers(0, 256, (4, 64), dtype=np.uint8)
    scales = rng.integers(120, 130, (4, 4), dtype=np.uint8)
    good = oracle.dequant_mxfp4(packed, scales, 4, 128)
    bad = swapped_nibble_dequant(packed, scales, 4, 128)
    assert sorted(good.ravel().tolist()) == sorted(bad.ravel().tolist())  # same multiset
    assert not np.array_equal(good, bad)                                # wrong positions


def test_dequant_exhaustive_code_by_scale():
    # every (code, scale byte) pair once: 16 codes x 256 scale bytes
    rows, cols = 256, 32
    packed = np.zeros((rows, 16), dtype=np.uint8)
    codes = np.arange(32) % 16
    packed[:] = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    scales = np.arange(256, dtype=np.uint8).reshape(256, 1)
    w = oracle.dequant_mxfp4(packed, scales, rows, cols)
    for s in range(256):
        for c in range(32):
            with np.errstate(over="ignore"):  # scale 254 with |code| >= 2 is beyond float
                want = np.float32(e2m1_closed_form(c % 16) * (0.0 if s == 255 else 2.0 ** (s - 127)))
            assert w[s, c] == want or (want == 0 and w[s, c] == 0)


def brute_mxfp4(packed, scales, rows, cols, x):
    """Textbook: dequantise to a double matrix with the closed forms, then matvec."""
    W = np.zeros((rows, cols))
    for r in range(rows):
        for c in range(cols):
            b = int(packed[r, c // 2])
            code = (b >> 4) if (c & 1) else (b & 15)
            s = int(scales[r, c // 32])
            W[r, c] = e2m1_closed_form(code) * (0.0 if s == 255 else 2.0 ** (s - 127))
    return W @ x.astype(np.float64)


@pytest.mark.parametrize("cols", [32, 96, 50])
def test_mxfp4_gemv_brute_force(cols):
    rng = np.random.default_rng(cols)
    rows = 7
    packed = rng.integers(0, 256, (rows, (cols + 1) // 2), dtype=np.uint8)
    scales = rng.integers(118, 132, (rows, (cols + 31) // 32), dtype=np.uint8)
    scales[2, 0] = 255  # a NaN scale: its group contributes nothing
    x = rng.standard_normal(cols).astype(np.float32)
    got = oracle.mxfp4_gemv(packed, scales, rows, cols, x)
    want = brute_mxfp4(packed, scales, rows, cols, x)
    # double accumulation of exact products, one rounding to float: within 1 ulp
    assert np.all(np.abs(got - want) <= np.spacing(np.abs(want).astype(np.float32)) + 1e-30)


def test_mxfp4_gemv_basis_vectors_return_columns():
    rng = np.random.default_rng(5)
    rows, cols = 5, 64
    packed = rng.integers(0, 256, (rows, 32), dtype=np.uint8)
    scales = rng.integers(100, 140, (rows, 2), dtype=np.uint8)
    W = oracle.dequant_mxfp4(packed, scales, rows, cols)
    for k in (0, 1, 31, 32, 63):
        x = np.zeros(cols, dtype=np.float32)
        x[k] = 1.0
        assert np.array_equal(oracle.mxfp4_gemv(packed, scales, rows, cols, x), W[:, k])


def test_mxfp4_gemv_equal_scales_factor_out():
    rng = np.random.default_rng(6)
    rows, cols = 4, 96
    packed = rng.integers(0, 256, (rows, 48), dtype=np.uint8)
    x = rng.standard_normal(cols).astype(np.float32)
    y127 = oracle.mxfp4_gemv(packed, np.full((rows, 3), 127, np.uint8), rows, cols, x)
    y130 = oracle.mxfp4_gemv(packed, np.full((rows, 3), 130, np.uint8), rows, cols, x)
    assert np.array_equal(y130, y127 * np.float32(8.0))


def test_bf16_gemv_matches_textbook_double():
    rng = np.random.default_rng(7)
    W = oracle.f32_to_bf16(rng.standard_normal((6, 40)).astype(np.float32))
    x = rng.standard_normal(40).astype(np.float32)
    want = oracle.bf16_to_f32(W).astype(np.float64) @ x.astype(np.float64)
    got = oracle.bf16_gemv(W, x)
    assert np.all(np.abs(got - want) <= np.spacing(np.abs(want).astype(np.float32)))


def test_rmsnorm_closed_forms():
    x = np.full(8, 3.0, dtype=np.float32)
    # mean(x^2) = 9: out = 3 / sqrt(9 + eps)
    out = oracle.rmsnorm(x, eps=1e-5)
    assert np.allclose(out, 3.0 / math.sqrt(9.0 + 1e-5), rtol=1e-7)
    # epsilon inside the root: a zero vector stays zero and finite
    assert np.array_equal(oracle.rmsnorm(np.zeros(4, np.float32)), np.zeros(4, np.float32))
    # scale invariance (up to eps)
    v = np.random.default_rng(8).standard_normal(64).astype(np.float32)
    assert np.allclose(oracle.rmsnorm(v, eps=0.0), oracle.rmsnorm(v * 4, eps=0.0), rtol=1e-6)
    # weight multiplies
    w = np.arange(64, dtype=np.float32)
    assert np.allclose(oracle.rmsnorm(v, w, eps=0.0), oracle.rmsnorm(v, eps=0.0) * w, rtol=1e-6)
