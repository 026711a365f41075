"""Pins for the oracle's MXFP8 quantiser (E4M3 elements, one E8M0 scale per
1x32 block along the row).

The pages only name the format and its quantise op (project summary
"Mixture-of-Kittens (MoK)", core-concepts table, MXFP8 row); the public
definition is OCP Microscaling Formats v1.0 with OFP8 E4M3. Pins: the
element rule against a brute-force nearest search over every decoded E4M3
value (ties to the even code, saturation at 448), published E4M3 code
points, the scale exponent against numpy's floor(log2(.)), exact round trips
and the half-quantum error bound.
"""
import numpy as np
import pytest

import oracle


def _decoded_table():
    codes = np.arange(0x7F)  # non-negative finite codes 0x00..0x7E
    e, m = codes >> 3, codes & 7
    val = np.where(e == 0, m * 2.0 ** -9, (8 + m) * 2.0 ** (e - 10.0))
    return codes, val


def _brute_encode(v):
    codes, val = _decoded_table()
    a = min(abs(v), 448.0)
    d = np.abs(val - a)
    best = np.flatnonzero(d == d.min())
    code = int(codes[best[0]]) if len(best) == 1 else int(codes[best][codes[best] % 2 == 0][0])
    return code | (0x80 if np.signbit(v) else 0)


def test_published_code_points():
    assert oracle.e4m3_encode(1.0) == 0x38
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(240.0) == 0x77
    assert oracle.e4m3_encode(2.0 ** -6) == 0x08   # smallest normal
    assert oracle.e4m3_encode(2.0 ** -9) == 0x01   # smallest subnormal
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-2.0) == 0xC0
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert np.isnan(oracle.e4m3_decode(0x7F))
    assert oracle.e4m3_encode(1e9) == 0x7E      # saturating
    assert oracle.e4m3_encode(464.0) == 0x7E    # would round toward 480 = NaN code


def test_element_rule_matches_brute_force_on_every_bf16_value():
    bits = np.arange(0, 0x10000, dtype=np.uint32)
    f32 = (bits << 16).view(np.float32)
    vals = f32[np.isfinite(f32)].astype(np.float64)
    vals = vals[np.abs(vals) <= 1024.0]
    for v in vals:
        assert oracle.e4m3_encode(v) == _brute_encode(v), v


def test_midpoints_round_to_even():
    _, val = _decoded_table()
    for lo, hi in zip(val[:-1], val[1:]):
        mid = (lo + hi) / 2
        assert oracle.e4m3_encode(mid) == _brute_encode(mid)
        assert oracle.e4m3_encode(mid) % 2 == 0


def _bf16_bits(a):
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _f(bits):
    return oracle.bf16_bits_to_f64(bits)


def test_scale_exponent_rule():
    rng = np.random.default_rng(0)
    src = _bf16_bits(rng.standard_normal((64, 256)) * np.exp(rng.uniform(-30, 30, (64, 1))))
    q, s = oracle.mxfp8_quantize(src)
    amax = np.abs(_f(src)).reshape(64, 8, 32).max(axis=2)
    expect = np.clip(np.floor(np.log2(amax)) - 8 + 127, 0, 254)
    np.testing.assert_array_equal(s, expect.astype(np.uint8))


def test_zero_block_and_powers_of_two():
    src = np.zeros((2, 64), np.float32)
    src[1, 32:] = 2.0 ** np.arange(-5, 27)
    q, s = oracle.mxfp8_quantize(_bf16_bits(src))
    assert s[0, 0] == 0 and s[0, 1] == 0 and s[1, 0] == 0 and np.all(q[0] == 0)
    assert s[1, 1] == 26 - 8 + 127
    # 2^26 / 2^18 = 2^8 = 256 -> E4M3 code for 256 (exponent field 15, mantissa 0)
    assert q[1, 63] == (15 << 3)


def test_exactly_representable_blocks_round_trip():
    rng = np.random.default_rng(3)
    _, val = _decoded_table()
    for trial in range(20):
        shift = int(rng.integers(-20, 20))
        block = rng.choice(val[val <= 448.0], 32) * rng.choice([-1, 1], 32)
        block[0] = 448.0  # pins amax so the scale is 2^shift
        src = _bf16_bits(block * 2.0 ** shift)
        assert np.all(_f(src) == block * 2.0 ** shift)  # bf16-exact (3 mantissa bits)
        q, s = oracle.mxfp8_quantize(src.reshape(1, 32))
        deq = np.array([oracle.e4m3_decode(c) for c in q[0]]) * 2.0 ** (int(s[0, 0]) - 127)
        np.testing.assert_array_equal(deq, _f(src))


def test_quantisation_error_bound():
    rng = np.random.default_rng(4)
    src = _bf16_bits(rng.standard_normal((16, 128)))
    q, s = oracle.mxfp8_quantize(src)
    v = _f(src).reshape(16, 4, 32)
    scale = 2.0 ** (s.astype(np.float64) - 127)
    deq = np.vectorize(oracle.e4m3_decode)(q).reshape(16, 4, 32) * scale[:, :, None]
    # half an E4M3 quantum at the element's binade (relative 2^-4), or half the
    # subnormal quantum 2^-10 * scale; the floor rule can put a block's largest
    # elements above 448 * scale, where they saturate to exactly 448 * scale
    sc = scale[:, :, None]
    bound = np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10 * sc)
    sat = np.abs(v) > 448.0 * sc
    assert np.all(np.abs(deq - v)[~sat] <= bound[~sat])
    np.testing.assert_array_equal(np.abs(deq[sat]), (448.0 * np.broadcast_to(sc, v.shape))[sat])


def test_rejects_ragged_columns():
    with pytest.raises(oracle.OracleError):
        oracle.mxfp8_quantize(np.zeros((2, 48), np.uint16))
