"""NVFP4 number formats and block quantization, written from their definitions.

Format facts used (from the pages):
  * weights and activations are FP4 (E2M1) with FP8 block scales -- FlashInfer
    issue #2723, "Model" table ("FP4 weights with FP8 block scales");
  * the block-scaled MMA operands are E2M1 x E2M1 with unsigned E4M3 scales,
    four scales per 64-element MMA K step, i.e. one scale per 16 elements --
    unsloth report, SASS paragraph under "Why it matters" (E2M1.E2M1.UE4M3.4X);
  * the per-block amax is taken in FP32 -- FlashInfer issue #2723, "What We
    Tried", item 2 "FP32 Amax Computation";
  * activations are quantized BF16 -> FP4 per token -- FlashInfer issue #2723,
    "Why 39 vs 49 tok/s?".
The pages give no rounding rule and no global-scale formula.  Readings taken
here: round-to-nearest-even with saturation for both encoders; the FP32
per-tensor global scale is a decode scale gs = amax / (6 * 448), so a block
scale is E4M3(amax_block / (6 * gs)).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32

# E2M1: sign bit 3, two exponent bits, one mantissa bit; magnitudes by code & 7.
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_MAX = 6.0
E4M3_MAX = 448.0
GLOBAL_SCALE_DIVISOR = F32(6.0 * 448.0)  # 2688: E2M1 max times E4M3 max
BLOCK = 16


def e4m3_value(code: int) -> float:
    """Value of an E4M3 (fn) byte: sign, 4 exponent bits (bias 7), 3 mantissa bits.

    Exponent field 0 is subnormal (m * 2^-9); 0x7F / 0xFF are NaN; there is no
    infinity, so the largest finite magnitude is 0x7E = 1.75 * 2^8 = 448.
    """
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    mag = m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
# Non-negative finite codes 0x00..0x7E are strictly increasing in value.
_E4M3_POS_VALUES = E4M3_TABLE[:0x7F]


def e2m1_decode(codes) -> np.ndarray:
    """E2M1 4-bit codes -> float64 values (sign-magnitude)."""
    c = np.asarray(codes).astype(np.int64)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where((c >> 3) & 1, -mag, mag)


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 bytes -> float64 values."""
    return E4M3_TABLE[np.asarray(codes).astype(np.int64)]


def _nearest_even(v: np.ndarray, values: np.ndarray) -> np.ndarray:
    """Index of the nearest entry of the increasing table ``values`` to each v >= 0.

    An exact tie between two neighbours goes to the even index (the code whose
    last mantissa bit is 0): round-to-nearest-even.  Values beyond the last
    entry map to the last entry (saturation).  Inside the table's range the
    differences are taken in float64, where they are exact for float32 inputs.
    """
    v = np.asarray(v, dtype=np.float64)
    n = len(values)
    hi_raw = np.searchsorted(values, v, side="left")      # values[hi-1] < v <= values[hi]
    hi = np.clip(hi_raw, 0, n - 1)
    lo = np.clip(hi - 1, 0, n - 1)
    d_lo = np.abs(v - values[lo])
    d_hi = np.abs(values[hi] - v)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(hi_raw >= n, n - 1, np.where(pick_hi, hi, lo))


def e2m1_encode(y) -> np.ndarray:
    """float32 -> E2M1 code: nearest magnitude, ties to the even code, saturating
    at 6; the sign bit is copied from y, so negative values that round to zero
    give code 0x8 (reading: the pages are silent on signed zero)."""
    y = np.asarray(y, dtype=F32)
    idx = _nearest_even(np.abs(y), E2M1_MAGNITUDES)
    return (idx | (np.signbit(y).astype(np.int64) << 3)).astype(np.uint8)


def e4m3_encode(v) -> np.ndarray:
    """float32 v >= 0 -> unsigned E4M3 byte: nearest finite value, ties to even,
    saturating at 448 (what a satfinite conversion does; +inf also gives 448)."""
    v = np.asarray(v, dtype=F32)
    if np.any(v < 0) or np.any(np.isnan(v)):
        raise ValueError("e4m3_encode expects non-negative, non-NaN inputs")
    return _nearest_even(v, _E4M3_POS_VALUES).astype(np.uint8)


def global_scale(amax) -> np.float32:
    """FP32 decode global scale of a tensor: amax / 2688 (one FP32 division), or 1
    for an all-zero tensor (reading: the pages give no formula)."""
    a = F32(amax)
    return F32(1.0) if a == 0 else F32(a / GLOBAL_SCALE_DIVISOR)


def quantize_rows(x, gs):
    """Quantize float32 rows [rows, K] to NVFP4 along K.

    gs: FP32 global decode scale, a scalar or one value per row.
    Per 16-element block, every step one IEEE float32 operation:
        amax = max |x_i|
        sb   = E4M3(amax / (6 * gs))
        r    = 0 if dec(sb) * gs == 0 else 1 / (dec(sb) * gs)
        q_i  = E2M1(x_i * r)
    Returns (codes uint8 [rows, K/2] with element 2j in the low nibble of byte j,
    scales uint8 [rows, K/16]).
    """
    x = np.asarray(x, dtype=F32)
    rows, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 16")
    gs = np.broadcast_to(np.asarray(gs, dtype=F32).reshape(-1, 1), (rows, 1)).astype(F32)
    blocks = x.reshape(rows, K // BLOCK, BLOCK)
    amax = np.max(np.abs(blocks), axis=2)                            # [rows, K/16], exact
    t1 = (F32(6.0) * gs).astype(F32)                                 # [rows, 1]
    with np.errstate(over="ignore"):
        t2 = (amax / t1).astype(F32)                                 # may overflow to +inf
    sb = e4m3_encode(t2)
    t3 = (e4m3_decode(sb).astype(F32) * gs).astype(F32)
    with np.errstate(divide="ignore"):
        r = np.where(t3 == 0, F32(0.0), (F32(1.0) / t3)).astype(F32)
    q = e2m1_encode((blocks * r[:, :, None]).astype(F32)).reshape(rows, K)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return codes, sb


def unpack_codes(codes) -> np.ndarray:
    """uint8 [rows, K/2] -> 4-bit codes [rows, K] (low nibble first)."""
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = c & 0xF
    out[..., 1::2] = c >> 4
    return out


def dequantize_rows(codes, scales) -> np.ndarray:
    """NVFP4 rows without the global scale: e2m1(q) * e4m3(sb), float64 (exact)."""
    q = e2m1_decode(unpack_codes(codes))
    s = e4m3_decode(scales)
    return q * np.repeat(s, BLOCK, axis=-1)
