"""Pins of the oracle's FP8 KV layout: e4m3 coding (OCP FP8 e4m3: 1 sign, 4
exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN)
and the per-row scaled split of a KV row ("DeepSeek-V4 CSA/HCA walkthrough",
section 2.3 step 4 and section 5.3: FP8 for the non-RoPE part, the RoPE part
kept wider).

Decoded values are checked against values worked out by hand from the bit
fields, rounding against midpoints and neighbours, the bf16 rounding against
torch's own cast, and the quantiser against its defining properties (the row
maximum lands on the largest code, the error stays within half a code step).
"""
import numpy as np
import pytest
import torch

import oracle


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x30, 0.5), (0x38, 1.0), (0x3F, 1.875), (0x40, 2.0), (0x52, 10.0), (0x7E, 448.0),
    (0x80, -0.0), (0xB8, -1.0), (0xFE, -448.0)])
def test_decode_by_hand(code, value):
    got = oracle.e4m3_decode(np.array([code], np.uint8))[0]
    assert got == value and np.signbit(got) == np.signbit(value)


def test_nan_codes():
    assert np.all(np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))))


def test_positive_codes_increase():
    v = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)
    assert v[-1] == 448.0


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)


def test_midpoints_round_to_the_even_code():
    v = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (v[:-1] + v[1:]) / 2
    got = oracle.e4m3_encode(mids)
    for i, c in enumerate(got):
        assert c == (i if i % 2 == 0 else i + 1), (i, hex(c))
    assert np.array_equal(oracle.e4m3_encode(-mids), got | 0x80)


def test_nearest_code_elsewhere():
    v = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    x = np.random.default_rng(0).uniform(0, 448, 20000)
    got = oracle.e4m3_decode(oracle.e4m3_encode(x))
    best = v[np.argmin(np.abs(x[:, None] - v[None, :]), axis=1)]
    assert np.array_equal(got, best)


def test_saturation_and_signed_zero():
    got = oracle.e4m3_encode(np.array([448.0, 449.0, 480.0, 1e9, -500.0, -0.0, -1e-9]))
    assert [int(c) for c in got] == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x80]


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(1).standard_normal(10000).astype(np.float32) * 100
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(oracle.bf16_round(x), want)


def test_quantised_rows():
    rng = np.random.default_rng(2)
    kv = (rng.standard_normal((50, 128)) * rng.uniform(0.01, 30, (50, 1))).astype(np.float32)
    codes, rope, scale = oracle.quantize_kv_fp8(kv, 64)
    assert codes.shape == (50, 64) and rope.shape == (50, 64) and scale.shape == (50,)
    amax = np.abs(kv[:, :64]).max(axis=1)
    # the row maximum maps onto +-448
    at = np.abs(kv[:, :64]).argmax(axis=1)
    assert np.all((codes[np.arange(50), at] & 0x7F) == 0x7E)
    np.testing.assert_allclose(scale, amax / 448.0, rtol=1e-6)
    deq = oracle.dequantize_kv_fp8(codes, rope, scale)
    # within half a code step: 2^-4 relative for normal codes, scale * 2^-10 near zero
    err = np.abs(deq[:, :64] - kv[:, :64])
    bound = np.maximum(np.abs(kv[:, :64]) * 2.0 ** -4, scale[:, None] * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(err <= bound)
    assert np.array_equal(deq[:, 64:], torch.from_numpy(kv[:, 64:]).to(torch.bfloat16).double().numpy())


def test_zero_row_part():
    kv = np.zeros((2, 8), np.float32)
    kv[1, 4:] = 3.0
    codes, rope, scale = oracle.quantize_kv_fp8(kv, 4)
    assert np.all(scale == 1.0) and np.all(codes == 0)
    assert np.array_equal(oracle.dequantize_kv_fp8(codes, rope, scale), kv.astype(np.float64))
