"""Pins for the oracle's E4M3 codec.  The why-be.why-be.co.kr (wr_id 35533)
page fixes the format (E4M3 for every tensor); the bit layout, rounding and
saturation follow the E4M3FN reading."""
import ctypes
import math

import numpy as np
import pytest
import torch


def test_decode_matches_torch_float8_e4m3fn(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_codes = {0x7F, 0xFF}
    for c in range(256):
        if c in nan_codes:
            assert math.isnan(ours[c]) and math.isnan(ref[c])
        else:
            assert ours[c] == ref[c], (c, ours[c], ref[c])
            assert math.copysign(1.0, ours[c]) == math.copysign(1.0, ref[c])


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6),
    (0x38, 1.0), (0x39, 1.125), (0x3F, 1.875), (0x40, 2.0), (0x7E, 448.0),
    (0x7D, 416.0), (0xFE, -448.0), (0xB8, -1.0), (0x70, 128.0), (0x78, 256.0),
])
def test_decode_hand_values(orc, code, value):
    assert orc.e4m3_decode(np.array([code]))[0] == value


def test_negative_zero_code(orc):
    v = orc.e4m3_decode(np.array([0x80]))[0]
    assert v == 0.0 and math.copysign(1.0, v) < 0
    assert orc.e4m3_encode(np.array([-0.0], np.float32))[0] == 0x80


def test_round_trip_every_finite_code(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = orc.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(orc.e4m3_encode(vals), codes)


@pytest.mark.parametrize("x,code", [
    (2.0 ** -10, 0x00),               # half of the smallest subnormal: tie -> even (0)
    (3 * 2.0 ** -10, 0x02),           # 1.5 quanta: tie -> even (2)
    (5 * 2.0 ** -10, 0x02),           # 2.5 quanta: tie -> even (2)
    (1.0625, 0x38),                   # halfway 1.0 / 1.125: even mantissa 0
    (1.1875, 0x3A),                   # halfway 1.125 / 1.25: even mantissa 2
    (464.0, 0x7E),                    # halfway 448 / (480): even -> 448
    (465.0, 0x7E),                    # past the midpoint: saturates to 448
    (1e30, 0x7E), (-1e30, 0xFE),
    (float("inf"), 0x7E), (float("-inf"), 0xFE),
    (-2.0 ** -11, 0x80),              # rounds to zero, keeps its sign
    (0.0009765625 * 1.0000001, 0x01),
])
def test_encode_edges(orc, x, code):
    assert orc.e4m3_encode(np.array([x], np.float32))[0] == code


def test_pin_table_matches_decode(orc, pin_lib):
    for c in range(127):
        assert pin_lib.table_value(c) == orc.e4m3_decode(np.array([c]))[0]


def test_encode_exhaustive_all_fp32(orc, pin_lib):
    """All 2^32 fp32 bit patterns: oracle encoder == independent nearest search."""
    chunk = 1 << 26
    for start in range(0, 1 << 32, chunk):
        q = orc.e4m3_encode_bits(start, chunk)
        first = ctypes.c_int64(-1)
        bad = pin_lib.check_chunk(start, chunk, q.ctypes.data_as(ctypes.c_void_p), ctypes.byref(first))
        assert bad == 0, "mismatch at fp32 bits 0x%08x" % (start + first.value)


def test_encode_matches_torch_in_range(orc):
    """torch's float8_e4m3fn cast is RNE but not saturating: above the 448/480
    midpoint (464) it returns NaN, so compare only up to 464."""
    g = torch.Generator().manual_seed(7)
    bits = torch.randint(0, 1 << 31, (1 << 22,), generator=g, dtype=torch.int64)
    x = bits.to(torch.int32).view(torch.float32)
    x = torch.cat([x, -x])
    x = x[torch.isfinite(x) & (x.abs() <= 464)]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = orc.e4m3_encode(x.numpy())
    assert np.array_equal(ours, ref)
