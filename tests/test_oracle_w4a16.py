"""Pins of the oracle's weight-only (W4A16) product (CPU).

An exact small case, a per-element math.fsum brute force, and consistency
with the W4A4 grouped GEMM: activations that lie exactly on the NVFP4 grid
(e2m1 x e4m3 x gs) give the same product through both definitions."""
import math

import numpy as np

from oracle import formats as F
from oracle import moe as M


def _pack(q):
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def test_exact_case():
    # weights: codes 2 (1.0) and 6 (4.0), scale 0x38 (1.0), gs 0.5; activations small integers
    K, N = 32, 2
    q = np.zeros((N, K), np.uint8)
    q[0, :] = 2
    q[1, ::2] = 6
    w_c, w_s = _pack(q), np.full((N, K // 16), 0x38, np.uint8)
    a = np.arange(K, dtype=np.float64)[None, :]
    d = M.w4a16_matmul(a, w_c, w_s, np.float32(0.5))
    assert d[0, 0] == 0.5 * a.sum() and d[0, 1] == 0.5 * 4.0 * a[0, ::2].sum()


def test_brute_force_against_fsum():
    rng = np.random.default_rng(0)
    K, N, R = 64, 5, 3
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w_c, w_s, gs = M.quantize_expert_weights(w)
    a = rng.standard_normal((R, K)).astype(np.float32).astype(np.float64)
    dw = F.dequantize_rows(w_c, w_s)
    d = M.w4a16_matmul(a, w_c, w_s, gs)
    for r in range(R):
        for n in range(N):
            exact = float(np.float32(gs)) * math.fsum(float(a[r, k]) * float(dw[n, k]) for k in range(K))
            assert abs(d[r, n] - exact) <= 1e-15 * abs(exact) + 1e-300


def test_consistent_with_w4a4_on_grid_activations():
    rng = np.random.default_rng(1)
    K, N, sizes = 128, 8, [3, 0, 5]
    G = len(sizes)
    offs = np.concatenate([[0], np.cumsum(sizes)])
    R = int(offs[-1])
    x = rng.standard_normal((R, K)).astype(np.float32)
    gs_a = F.global_scale(np.abs(x).max())
    a_c, a_s = F.quantize_rows(x, gs_a)
    a_grid = F.dequantize_rows(a_c, a_s) * np.float64(gs_a)      # exactly representable activations
    w = (rng.standard_normal((G, N, K)) * 0.02).astype(np.float32)
    qw = [M.quantize_expert_weights(w[g]) for g in range(G)]
    w_c = np.stack([q[0] for q in qw])
    w_s = np.stack([q[1] for q in qw])
    gs_w = np.array([q[2] for q in qw], np.float32)
    w4a16 = M.grouped_w4a16(a_grid, offs, w_c, w_s, gs_w)
    w4a4 = M.grouped_gemm(a_c, a_s, offs, np.full(G, gs_a, np.float32), w_c, w_s, gs_w)
    # the two scale the same exact sum by gs_w (W4A16) and by gs_a * gs_w rounded to FP32 (W4A4)
    for e in range(G):
        lo, hi = offs[e], offs[e + 1]
        if hi > lo:
            s_exact = M.block_scaled_matmul(a_c[lo:hi], a_s[lo:hi], w_c[e], w_s[e])
            assert np.allclose(w4a16[lo:hi], np.float64(gs_w[e]) * np.float64(gs_a) * s_exact, rtol=1e-14, atol=0)
            assert np.allclose(w4a4[lo:hi], np.float64(M.alpha(gs_a, gs_w[e])) * s_exact, rtol=0, atol=0)
