"""Test-side helpers: build/load the CUDA library and undo its internal layouts.

The layouts undone here (scale atoms, grouped tiles, the prepared w13 row
order) are stated in include/nvfp4moe.h; these helpers restate them in numpy
so the parity tests can compare canonical [rows, K/16] views with the oracle.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def ensure_built():
    from nvfp4_moe_grouped_router_gb300 import build
    return build.build()


TILE_BYTES = 18432
TILE_CODE_BYTES = 16384


def atom_index(r128, b4):
    return (r128 % 32) * 16 + (r128 // 32) * 4 + b4


def row_tiles(rows: int, offsets=None, tile_offsets=None):
    """(tile, r) of every row of a TILED_GROUPED operand (one group when offsets is None)."""
    p = np.arange(rows)
    if offsets is None:
        return p // 128, p % 128
    offsets = np.asarray(offsets, dtype=np.int64)
    tile_offsets = np.asarray(tile_offsets, dtype=np.int64)
    g = np.searchsorted(offsets, p, side="right") - 1
    local = p - offsets[g]
    return tile_offsets[g] + local // 128, local % 128


def tiled_index(tile, r, K):
    """Byte offsets of every code byte [rows, K/2] and scale byte [rows, K/16] of a
    TILED_GROUPED operand: 18432-byte chunk (tile, kt) = [codes][atoms]."""
    nkt = (K + 255) // 256
    tile = np.asarray(tile, dtype=np.int64)[:, None]
    r = np.asarray(r, dtype=np.int64)[:, None]
    b = np.arange(K // 2)[None, :]
    kt, bb = b // 128, b % 128
    code = (tile * nkt + kt) * TILE_BYTES + r * 128 + (((bb // 16) ^ (r % 8)) * 16) + bb % 16
    kb = np.arange(K // 16)[None, :]
    kt2, kk, s = kb // 16, (kb % 16) // 4, kb % 4
    sf = (tile * nkt + kt2) * TILE_BYTES + TILE_CODE_BYTES + kk * 512 + atom_index(r % 128, s)
    return code, sf


def tiled_unpack(buf, K, tile, r):
    """TILED_GROUPED bytes -> (codes [rows, K/2], scales [rows, K/16]) for rows at (tile, r)."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    code, sf = tiled_index(tile, r, K)
    return buf[code], buf[sf]


def weight_index(rows: int, K: int, group_rows: int):
    """Byte offsets of every code byte [rows, K/2] and scale byte [rows, K/16] in
    the TILED (weight) layout: groups of group_rows rows; within a group, tiles
    2p and 2p + 1 share 36864-byte units [codes 2p][codes 2p+1][atoms 2p]
    [atoms 2p+1] per K tile; an odd last tile has 18432-byte units."""
    nkt = (K + 255) // 256
    row = np.arange(rows, dtype=np.int64)
    g, rl = row // group_rows, row % group_rows
    ntg = (group_rows + 127) // 128
    tile = rl // 128
    pair, half = tile // 2, tile % 2
    paired = 2 * pair + 1 < ntg
    r = (rl % 128)[:, None]

    def unit(kt):
        return ((g * ntg + 2 * pair)[:, None] * nkt + kt * np.where(paired, 2, 1)[:, None]) * TILE_BYTES

    b = np.arange(K // 2)[None, :]
    kt, bb = b // 128, b % 128
    codes = unit(kt) + np.where(paired, half * TILE_CODE_BYTES, 0)[:, None]
    code = codes + r * 128 + (((bb // 16) ^ (r % 8)) * 16) + bb % 16
    kb = np.arange(K // 16)[None, :]
    kt2, kk, s = kb // 16, (kb % 16) // 4, kb % 4
    atoms = unit(kt2) + np.where(paired, 2 * TILE_CODE_BYTES + half * 2048, TILE_CODE_BYTES)[:, None]
    sf = atoms + kk * 512 + atom_index(r, s)
    return code, sf


def weight_unpack(buf, K, rows, group_rows):
    """TILED (weight) bytes -> (codes [rows, K/2], scales [rows, K/16])."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    code, sf = weight_index(rows, K, group_rows)
    return buf[code], buf[sf]


def weight_pack(codes, scales, K, group_rows, nbytes):
    """Inverse of weight_unpack; bytes not covered stay 0."""
    out = np.zeros(nbytes, np.uint8)
    code, sf = weight_index(codes.shape[0], K, group_rows)
    out[code] = codes
    out[sf] = scales
    return out


def tiled_pack(codes, scales, K, tile, r, nbytes):
    """Inverse of tiled_unpack; bytes not covered stay 0."""
    out = np.zeros(nbytes, np.uint8)
    code, sf = tiled_index(tile, r, K)
    out[code] = codes
    out[sf] = scales
    return out


def w13_prepared_rows(I: int) -> np.ndarray:
    """Canonical row of each prepared w13 row: blocks of 16 gate rows then 16 up rows."""
    r = np.arange(2 * I)
    c, within = r // 32, r % 32
    return np.where(within < 16, 16 * c + within, I + 16 * c + within - 16)


def rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    return float(np.max(np.abs(got - ref)) / rms) if ref.size and rms > 0 else float(np.max(np.abs(got - ref), initial=0))


# ----------------------------------------------------------------------------- independent quantizer
# A second statement of NVFP4 block quantization, written from the threshold
# table (E2M1) and the quantum-and-round formula (E4M3) rather than the
# oracle's nearest-value search.  The tests use it to check that a GPU
# intermediate (the requantized h) is a valid quantization of the GPU's own
# values without feeding GPU data into the oracle.
def e2m1_threshold_encode(y):
    y = np.asarray(y, dtype=np.float32)
    v = np.abs(y)
    m = np.select([v <= 0.25, v < 0.75, v <= 1.25, v < 1.75, v <= 2.5, v < 3.5, v <= 5.0], [0, 1, 2, 3, 4, 5, 6], 7)
    return (m | (np.signbit(y).astype(np.int64) << 3)).astype(np.uint8)


def e4m3_formula_encode(v):
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros(v.shape, np.int64)
    sat = v >= 448.0
    sub = v < 2.0 ** -6
    out[sub] = np.rint(v[sub] * 512.0).astype(np.int64)
    nrm = ~sat & ~sub
    mant, ex = np.frexp(v[nrm])                 # v = mant * 2^ex, mant in [0.5, 1)
    e = ex - 1                                  # floor(log2 v)
    n = np.rint(v[nrm] / np.ldexp(1.0, e - 3)).astype(np.int64)
    carry = n == 16
    e = np.where(carry, e + 1, e)
    n = np.where(carry, 8, n)
    out[nrm] = np.minimum(((e + 7) << 3) | (n - 8), 0x7E)
    out[sat] = 0x7E
    return out.astype(np.uint8)


def e4m3_formula_decode(b):
    b = np.asarray(b, dtype=np.int64)
    e, m = (b >> 3) & 0xF, b & 7
    return np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * np.ldexp(1.0, e - 7))


def quantize_rows_check(x, gs):
    f32 = np.float32
    x = np.asarray(x, dtype=f32)
    rows, K = x.shape
    gs = np.broadcast_to(np.asarray(gs, dtype=f32).reshape(-1, 1), (rows, 1)).astype(f32)
    b = x.reshape(rows, K // 16, 16)
    amax = np.abs(b).max(axis=2)
    with np.errstate(over="ignore", divide="ignore", invalid="ignore"):
        t2 = (amax / (f32(6.0) * gs).astype(f32)).astype(f32)
        sb = e4m3_formula_encode(t2)
        t3 = (e4m3_formula_decode(sb).astype(f32) * gs).astype(f32)
        r = np.where(t3 == 0, f32(0), f32(1.0) / t3).astype(f32)
        q = e2m1_threshold_encode((b * r[:, :, None]).astype(f32)).reshape(rows, K)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8), sb


def dequant_check(codes, scales):
    """Dequantized NVFP4 rows without the global scale, from the formulas above."""
    c = np.asarray(codes, dtype=np.uint8)
    q = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), np.int64)
    q[..., 0::2] = c & 0xF
    q[..., 1::2] = c >> 4
    mag = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])[q & 7]
    val = np.where(q & 8, -mag, mag)
    return val * np.repeat(e4m3_formula_decode(scales), 16, axis=-1)
