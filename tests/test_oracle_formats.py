"""Pins for the oracle's NVFP4 format code (CPU only).

Each test ties oracle.formats to something other than itself: the formats'
closed forms, torch's float8_e4m3fn cast, independent scalar encoders written
from a different formulation (threshold table, quantum-and-round), and
invariants of block quantization.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "format_closed_forms.json")


def test_closed_forms_match_golden():
    g = json.load(open(GOLDEN))
    assert list(F.e2m1_decode(np.arange(8))) == g["e2m1_magnitudes_by_code"]
    assert list(F.e2m1_decode(np.arange(8, 16))) == [-v for v in g["e2m1_magnitudes_by_code"]]
    for code, v in g["e4m3_landmarks"].items():
        assert F.e4m3_value(int(code, 16)) == v, code
    assert np.nanmax(F.E4M3_TABLE) == g["e4m3_max"]
    assert math.isnan(F.e4m3_value(0x7F)) and math.isnan(F.e4m3_value(0xFF))
    assert float(F.GLOBAL_SCALE_DIVISOR) == g["global_scale_divisor"] == g["e2m1_max"] * g["e4m3_max"]


def test_e4m3_table_against_torch_float8():
    # torch's float8_e4m3fn decode is an independent implementation of the format.
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(t) & np.isnan(F.E4M3_TABLE)
    assert np.all(both_nan | (t == F.E4M3_TABLE))


def test_round_trip_all_codes():
    c = np.arange(16, dtype=np.uint8)
    assert np.array_equal(F.e2m1_encode(F.e2m1_decode(c).astype(np.float32)), c)
    c8 = np.arange(0x7F, dtype=np.uint8)
    assert np.array_equal(F.e4m3_encode(F.e4m3_decode(c8).astype(np.float32)), c8)


def _e2m1_threshold(y: float) -> int:
    """Independent E2M1 encoder from the round-to-nearest-even threshold table."""
    v = abs(y)
    if v <= 0.25:
        m = 0
    elif v < 0.75:
        m = 1
    elif v <= 1.25:
        m = 2
    elif v < 1.75:
        m = 3
    elif v <= 2.5:
        m = 4
    elif v < 3.5:
        m = 5
    elif v <= 5.0:
        m = 6
    else:
        m = 7
    return m | (8 if math.copysign(1.0, y) < 0 else 0)


def test_e2m1_encode_all_bf16_inputs_vs_threshold_table():
    bits = np.arange(65536, dtype=np.uint32) << 16
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    for scale in (1.0, 0.37, 3.1):
        y = (vals * np.float32(scale)).astype(np.float32)
        y = y[np.isfinite(y)]
        got = F.e2m1_encode(y)
        ref = np.array([_e2m1_threshold(float(v)) for v in y], dtype=np.uint8)
        assert np.array_equal(got, ref)


def test_e2m1_ties_to_even_and_saturation():
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    assert list(F.e2m1_encode(mids)) == [0, 2, 2, 4, 4, 6, 6]
    assert list(F.e2m1_encode(-mids)) == [8, 10, 10, 12, 12, 14, 14]
    assert list(F.e2m1_encode(np.array([6.0, 7.0, 1e30], np.float32))) == [7, 7, 7]
    # negative values that round to zero keep their sign (code 0x8)
    assert list(F.e2m1_encode(np.array([-0.1, -0.0, 0.0, 0.1], np.float32))) == [8, 8, 0, 0]


def _e4m3_formula(v: float) -> int:
    """Independent E4M3 encoder: quantum q = 2^(floor(log2 v) - 3) for v >= 2^-6
    (2^-9 below), n = round-half-even(v / q) in exact rational arithmetic, a
    carry to 16 bumps the exponent, saturation at 448; the code is assembled
    from (exponent, mantissa) bits."""
    if v >= 448.0:
        return 0x7E
    fv = Fraction(v)
    if fv < Fraction(1, 64):
        n = round(fv * 512)            # subnormal quantum 2^-9; n == 8 is the first normal
        return n
    e = 0
    while Fraction(2) ** (e + 1) <= fv:
        e += 1
    while Fraction(2) ** e > fv:
        e -= 1
    n = round(fv / Fraction(2) ** (e - 3))   # 8 <= n <= 16, halves to even
    if n == 16:
        e, n = e + 1, 8
    code = ((e + 7) << 3) | (n - 8)
    return min(code, 0x7E)


def test_e4m3_encode_vs_formula_and_torch():
    rng = np.random.default_rng(0)
    # every midpoint between neighbouring codes, one ulp either side, plus a dense random sample
    vals = F.E4M3_TABLE[:0x7F]
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    below = np.nextafter(mids, np.float32(0))
    above = np.nextafter(mids, np.float32(1e9))
    samp = rng.uniform(0, 448, 4000).astype(np.float32)
    small = (rng.uniform(0, 0.03, 2000)).astype(np.float32)
    x = np.concatenate([mids, below, above, samp, small, vals.astype(np.float32)])
    got = F.e4m3_encode(x)
    ref = np.array([_e4m3_formula(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # torch's cast rounds to nearest even below the overflow point
    tt = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, tt)


def test_e4m3_exhaustive_bit_patterns_vs_torch():
    # every 7th float32 bit pattern in [0, 448]
    top = np.array([448.0], np.float32).view(np.uint32)[0]
    bits = np.arange(0, top + 1, 7, dtype=np.uint32)
    x = bits.view(np.float32)
    got = F.e4m3_encode(x)
    tt = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, tt)


def test_e4m3_saturates():
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3e38, np.inf], np.float32)
    assert np.all(F.e4m3_encode(x) == 0x7E)


def test_encoders_monotone():
    x = np.sort(np.random.default_rng(1).uniform(0, 500, 10000).astype(np.float32))
    assert np.all(np.diff(F.e4m3_encode(x).astype(int)) >= 0)
    y = np.sort(np.random.default_rng(2).uniform(0, 8, 10000).astype(np.float32))
    assert np.all(np.diff(F.e2m1_encode(y).astype(int)) >= 0)


def test_global_scale():
    assert F.global_scale(0.0) == np.float32(1.0)
    assert F.global_scale(2688.0) == np.float32(1.0)
    a = np.float32(3.7)
    assert F.global_scale(a) == np.float32(a / np.float32(2688.0))


def test_quantize_block_holding_tensor_amax():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    gs = F.global_scale(np.max(np.abs(x)))
    codes, sb = F.quantize_rows(x, gs)
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sb[r, c // 16] == 0x7E
    q = F.unpack_codes(codes)[r, c]
    assert (q & 7) == 7 and (q >> 3) == (1 if x[r, c] < 0 else 0)


def test_quantize_reproduces_exact_inputs():
    rng = np.random.default_rng(4)
    rows, K = 32, 128
    q = rng.integers(0, 16, (rows, K)).astype(np.uint8)
    q[:, ::16] = rng.choice([7, 15], (rows, K // 16))      # every block holds a +-6
    sb = rng.integers(1, 0x7F, (rows, K // 16)).astype(np.uint8)
    gs = np.float32(2.0 ** -5)                              # power of two keeps products exact
    x = (F.e2m1_decode(q) * np.repeat(F.e4m3_decode(sb), 16, axis=1) * float(gs)).astype(np.float32)
    assert np.array_equal(x.astype(np.float64), F.e2m1_decode(q) * np.repeat(F.e4m3_decode(sb), 16, axis=1) * float(gs))
    codes, s2 = F.quantize_rows(x, gs)
    assert np.array_equal(s2, sb)
    got = F.unpack_codes(codes)
    # +0 and -0 both decode to zero; compare values for zeros, codes otherwise
    nz = (q & 7) != 0
    assert np.array_equal(got[nz], q[nz])
    assert np.all((got[~nz] & 7) == 0)


def test_quantize_error_bound():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((128, 512)) * rng.uniform(0.01, 10, (128, 1))).astype(np.float32)
    gs = F.global_scale(np.max(np.abs(x)))
    codes, sb = F.quantize_rows(x, gs)
    deq = F.dequantize_rows(codes, sb) * float(gs)
    unit = np.repeat(F.e4m3_decode(sb), 16, axis=1) * float(gs)
    # largest gap on the E2M1 grid is 2 (between 4 and 6): error <= 1 unit, plus float32 slack
    assert np.all(np.abs(deq - x) <= unit * 1.0 + 1e-6 * np.abs(x) + 1e-30)
    # and for values below 2 units the gap is 0.5: error <= 0.25 unit
    small = np.abs(x) < 1.75 * unit
    assert np.all((np.abs(deq - x) <= 0.25 * unit * (1 + 1e-6) + 1e-30)[small])


def test_quantize_zero_blocks():
    x = np.zeros((2, 32), np.float32)
    x[1] = -0.0
    codes, sb = F.quantize_rows(x, np.float32(1.0))
    assert np.all(sb == 0)
    assert np.all(codes[0] == 0)
    assert np.all(codes[1] == 0x88)


def test_nibble_order_low_first():
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = 6.0
    x[0, 1] = 1.0
    codes, sb = F.quantize_rows(x, np.float32(1.0))
    q = F.unpack_codes(codes)
    assert q[0, 0] == 7 and q[0, 1] == 2 and codes[0, 0] == (7 | (2 << 4))


@pytest.mark.parametrize("rows,K", [(1, 16), (3, 64), (17, 256)])
def test_packing_shapes(rows, K):
    x = np.random.default_rng(6).standard_normal((rows, K)).astype(np.float32)
    codes, sb = F.quantize_rows(x, np.float32(0.01))
    assert codes.shape == (rows, K // 2) and sb.shape == (rows, K // 16)
    assert np.array_equal(F.unpack_codes(codes).reshape(rows, K // 2, 2)[..., 0], codes & 0xF)
