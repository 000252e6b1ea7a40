"""Pins of the oracle's fp16 conversion, group quantisation, packing and
dequantisation against things other than the oracle itself: numpy's IEEE
binary16 conversion (a library routine), closed-form grids, the round-half-
even rule on exact half-way points, degenerate groups and the error bound.

Format reading (the pages name INT2/INT4-style quantisation families in the
"VeriCache Guide" section "The Uniform Compressor Interface" but give no bit
format): asymmetric, 32-channel groups of one token, fp16 scale = fp16((max -
min) / (2^b - 1)), fp16 zero = fp16(min), codes rint((x - zero) / scale)
clamped to [0, 2^b - 1], packed little-endian, b bits per code.
"""
import os

import numpy as np
import pytest

import oracle
from synth import bf16_bits, bf16_to_f32


# ---------------------------------------------------------------- fp16

def _check_f16_against_numpy(u):
    f = u.view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    got = oracle.f32_to_f16(f)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    g = got[nan]
    assert np.all(((g & 0x7C00) == 0x7C00) & ((g & 0x3FF) != 0))


def test_f32_to_f16_all_high_halves_vs_numpy():
    """Every sign / exponent / top-7-mantissa pattern (all 2^16 high halves)
    combined with the low halves that sit on and around every rounding
    boundary (normal numbers round at bit 12, with bit 13 as the tie-break
    parity; subnormal boundaries lie in the high half) plus random ones,
    against numpy's round-to-nearest-even cast."""
    rng = np.random.default_rng(0)
    lows = [0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x2FFF, 0x3000,
            0x3001, 0x7FFF, 0x8000, 0x8001, 0xEFFF, 0xF000, 0xF001, 0xFFFF]
    lows += [int(v) for v in rng.integers(0, 1 << 16, 16)]
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    for lo in lows:
        _check_f16_against_numpy(hi | np.uint32(lo))


@pytest.mark.skipif(not os.environ.get("VC_EXHAUSTIVE"), reason="set VC_EXHAUSTIVE=1 (about a minute)")
def test_f32_to_f16_exhaustive_vs_numpy():
    """All 2^32 fp32 bit patterns."""
    step = 1 << 24
    for s in range(0, 1 << 32, step):
        _check_f16_against_numpy(np.arange(s, s + step, dtype=np.uint32))


def test_f16_to_f32_exhaustive_vs_numpy():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = oracle.f16_to_f32(h)
    nan = np.isnan(ref)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert np.all(np.isnan(got[nan]))


# ---------------------------------------------------------------- groups

@pytest.mark.parametrize("bits", [2, 3, 4])
def test_exact_grid_round_trip(bits):
    """x = mn + k * s with s a power of two: codes are k, dequant is exact."""
    q = (1 << bits) - 1
    s = 2.0 ** -3
    mn = -1.0
    k = np.arange(32) % (q + 1)
    k[0], k[1] = 0, q                      # make min and max present
    x = (mn + k * s).astype(np.float32)
    codes, sh, zh = oracle.quantize_group(x, bits)
    assert oracle.f16_to_f32(np.array([sh]))[0] == np.float32(s)
    assert oracle.f16_to_f32(np.array([zh]))[0] == np.float32(mn)
    assert np.array_equal(codes, k.astype(np.uint8))
    xr = oracle.dequant_row(codes, np.array([sh]), np.array([zh]))
    assert np.array_equal(xr, x.astype(np.float64))


def test_half_way_points_round_to_even():
    """x = mn + (k + 1/2) s falls exactly half-way: rint must pick the even
    neighbour (round-half-away would pick k + 1 every time)."""
    bits, s, mn = 4, 2.0 ** -3, -1.0
    k = np.arange(32) % 15
    x = (mn + (k + 0.5) * s).astype(np.float32)
    x[0], x[1] = mn, mn + 15 * s           # pin min/max so that s stays 1/8
    codes, _, _ = oracle.quantize_group(x, bits)
    want = np.where(k % 2 == 0, k, k + 1).astype(np.uint8)
    want[0], want[1] = 0, 15
    assert np.array_equal(codes, want)


def test_constant_group():
    x = np.full(32, 0.75, np.float32)
    codes, sh, zh = oracle.quantize_group(x, 2)
    assert sh == 0 and np.all(codes == 0)
    assert oracle.f16_to_f32(np.array([zh]))[0] == np.float32(0.75)
    assert np.all(oracle.dequant_row(codes, np.array([sh]), np.array([zh])) == 0.75)


def test_negative_zero_minimum_is_stored_as_plus_zero():
    x = np.abs(np.linspace(0.0, 1.0, 32, dtype=np.float32))
    x[0] = -0.0
    _, _, zh = oracle.quantize_group(x, 4)
    assert zh == 0x0000


def test_subnormal_scale_clamps_codes():
    """A tiny range whose scale rounds DOWN to the smallest fp16 subnormal:
    the maximum's quotient exceeds 2^b - 1 and must clamp to it.
    mn = 2^-20 (exact in bf16 and fp16), mx = mn + 35 * 2^-27.
    s_dot = 35 * 2^-27 / 3 ~= 1.458 * 2^-24 -> fp16 2^-24;
    (mx - mn) / 2^-24 = 35 / 8 = 4.375 -> rint 4 -> clamp 3."""
    mn = 2.0 ** -20
    mx = mn + 35 * 2.0 ** -27
    x = np.full(32, mn, np.float32)
    x[5] = mx
    assert np.array_equal(bf16_to_f32(bf16_bits(x)), x)     # representable in bf16
    codes, sh, zh = oracle.quantize_group(x, 2)
    assert sh == 0x0001 and oracle.f16_to_f32(np.array([zh]))[0] == np.float32(mn)
    assert codes[5] == 3 and np.all(np.delete(codes, 5) == 0)


def test_zero_rounded_above_minimum_clamps_at_zero():
    """mn too small for fp16 precision: fp16(mn) > mn, so (mn - z) / s < 0 and
    the code must clamp to 0, not wrap."""
    mn = float(bf16_to_f32(bf16_bits(np.array([1.0e-6], np.float32)))[0])
    z = float(oracle.f16_to_f32(oracle.f32_to_f16(np.array([mn], np.float32)))[0])
    assert z > mn
    x = np.full(32, 0.5, np.float32)
    x[3] = mn
    codes, _, zh = oracle.quantize_group(x, 4)
    assert codes[3] == 0 and oracle.f16_to_f32(np.array([zh]))[0] == np.float32(z)


def test_saturation_of_large_scale():
    x = np.zeros(32, np.float32)
    x[0], x[1] = -1.0e6, 1.0e6      # range 2e6 / 3 > 65504
    codes, sh, zh = oracle.quantize_group(x, 2)
    assert sh == 0x7BFF and zh == 0xFBFF          # +65504, -65504
    assert codes.max() <= 3


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_error_bound_random_rows(bits):
    """|x - x_hat| <= s/2 + |z - mn| + (2^b - 1) |s - s_dot| + tiny, per
    element, on bf16 N(0,1) rows with x10 outliers."""
    rng = np.random.default_rng(7)
    q = (1 << bits) - 1
    for _ in range(200):
        x = rng.standard_normal(128).astype(np.float32)
        x[rng.integers(0, 128, 3)] *= 10
        xb = bf16_bits(x)
        xf = bf16_to_f32(xb).astype(np.float64)
        codes, s16, z16 = oracle.quantize_row(xb, bits)
        assert codes.max() <= q
        xr = oracle.dequant_row(codes, s16, z16)
        s = oracle.f16_to_f32(s16).astype(np.float64)
        z = oracle.f16_to_f32(z16).astype(np.float64)
        g = xf.reshape(4, 32)
        mn, mx = g.min(1), g.max(1)
        sdot = (mx - mn) / q
        bound = s / 2 + np.abs(z - mn) + q * np.abs(s - sdot) + 1e-6 * np.abs(g).max(1)
        err = np.abs(xr - xf).reshape(4, 32).max(1)
        assert np.all(err <= bound)
        # the stored parameters describe the group: z ~ mn, z + q s ~ mx
        assert np.all(np.abs(z - mn) <= 2.0 ** -10 * np.abs(mn) + 2.0 ** -24)


# ---------------------------------------------------------------- packing

def test_pack_known_patterns():
    c = np.zeros(32, np.uint8)
    c[:4] = [1, 2, 3, 0]
    p = oracle.pack_codes(c, 2)
    assert p[0] == 0x39 and np.all(p[1:] == 0)
    c = np.zeros(32, np.uint8)
    c[:8] = np.arange(8)
    p = oracle.pack_codes(c, 3)       # sum_i i << 3i = 0xFAC688
    assert list(p[:3]) == [0x88, 0xC6, 0xFA] and np.all(p[3:] == 0)
    c = np.zeros(32, np.uint8)
    c[:2] = [0xA, 0x5]
    p = oracle.pack_codes(c, 4)
    assert p[0] == 0x5A
    c[:] = 1
    assert np.all(oracle.pack_codes(c, 2) == 0x55)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pack_unpack_identity(bits):
    rng = np.random.default_rng(bits)
    for d in (32, 64, 128, 256):
        c = rng.integers(0, 1 << bits, d).astype(np.uint8)
        p = oracle.pack_codes(c, bits)
        assert p.size == d * bits // 8
        assert np.array_equal(oracle.unpack_codes(p, d, bits), c)
        # bit-level definition: code i = bits [b i, b i + b) of the LE string
        allbits = np.unpackbits(p, bitorder="little")
        for i in (0, 1, d // 2, d - 1):
            v = sum(int(allbits[bits * i + k]) << k for k in range(bits))
            assert v == c[i]


def test_compress_bits16_is_a_gather():
    rng = np.random.default_rng(3)
    k = rng.integers(0, 1 << 16, (50, 2, 32)).astype(np.uint16)
    v = rng.integers(0, 1 << 16, (50, 2, 32)).astype(np.uint16)
    kept = np.array([0, 3, 4, 17, 49], np.int32)
    out = oracle.compress(k, v, kept, 16)
    assert np.array_equal(out["k16"], k[kept]) and np.array_equal(out["v16"], v[kept])
    with pytest.raises(ValueError):
        oracle.compress(k, v, np.array([50], np.int32), 16)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_compress_rows_match_row_quantiser(bits):
    rng = np.random.default_rng(11)
    k = bf16_bits(rng.standard_normal((40, 2, 64)).astype(np.float32))
    v = bf16_bits(rng.standard_normal((40, 2, 64)).astype(np.float32))
    kept = np.array([1, 5, 6, 39], np.int32)
    out = oracle.compress(k, v, kept, bits)
    for j, t in enumerate(kept):
        for h in range(2):
            c, s, z = oracle.quantize_row(v[t, h], bits)
            assert np.array_equal(out["v_packed"][j, h], oracle.pack_codes(c, bits))
            assert np.array_equal(out["v_scales"][j, h], s) and np.array_equal(out["v_zeros"][j, h], z)
