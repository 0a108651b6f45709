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


def atom_index(r128, b4):
    return (r128 % 32) * 16 + (r128 // 32) * 4 + b4


def unswizzle_mma(sf: np.ndarray, rows: int, K: int) -> np.ndarray:
    """NVF_SF_MMA bytes -> [rows, K/16]."""
    sf = np.asarray(sf, dtype=np.uint8).reshape(-1)
    r = np.arange(rows)[:, None]
    kb = np.arange(K // 16)[None, :]
    off = ((r // 128) * (K // 64) + kb // 4) * 512 + atom_index(r % 128, kb % 4)
    return sf[off]


def unswizzle_grouped(sf: np.ndarray, offsets, tile_offsets, K: int) -> np.ndarray:
    """NVF_SF_GROUPED bytes -> [offsets[-1], K/16] for the rows of every group."""
    sf = np.asarray(sf, dtype=np.uint8).reshape(-1)
    offsets = np.asarray(offsets, dtype=np.int64)
    tile_offsets = np.asarray(tile_offsets, dtype=np.int64)
    R = int(offsets[-1])
    out = np.zeros((R, K // 16), np.uint8)
    kb = np.arange(K // 16)[None, :]
    for g in range(len(offsets) - 1):
        lo, hi = offsets[g], offsets[g + 1]
        if hi == lo:
            continue
        local = np.arange(hi - lo)[:, None]
        tile = tile_offsets[g] + local // 128
        off = (tile * (K // 64) + kb // 4) * 512 + atom_index(local % 128, kb % 4)
        out[lo:hi] = sf[off]
    return out


def grouped_from_rowmajor(scales: np.ndarray, offsets, tile_offsets, K: int, nbytes: int) -> np.ndarray:
    """[R, K/16] -> NVF_SF_GROUPED bytes (inverse of unswizzle_grouped; other bytes 0)."""
    out = np.zeros(nbytes, np.uint8)
    offsets = np.asarray(offsets, dtype=np.int64)
    tile_offsets = np.asarray(tile_offsets, dtype=np.int64)
    kb = np.arange(K // 16)[None, :]
    for g in range(len(offsets) - 1):
        lo, hi = offsets[g], offsets[g + 1]
        if hi == lo:
            continue
        local = np.arange(hi - lo)[:, None]
        tile = tile_offsets[g] + local // 128
        off = (tile * (K // 64) + kb // 4) * 512 + atom_index(local % 128, kb % 4)
        out[off] = scales[lo:hi]
    return out


def mma_from_rowmajor(scales: np.ndarray, rows: int, K: int) -> np.ndarray:
    out = np.zeros((rows + 127) // 128 * 128 * (K // 16), np.uint8)
    r = np.arange(rows)[:, None]
    kb = np.arange(K // 16)[None, :]
    off = ((r // 128) * (K // 64) + kb // 4) * 512 + atom_index(r % 128, kb % 4)
    out[off] = scales
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
