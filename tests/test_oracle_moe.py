"""Pins for the oracle's routing, permutation, GEMM, epilogue and combine (CPU only).

Each check ties oracle.moe to an independent formulation: brute-force sorts in
pure Python, exact rational arithmetic for block-scaled products, scipy's
softmax, algebraic identities of SiLU, reductions of the combine to a plain
unpermute or a dense mixture, and an end-to-end per-token walk on the tiny
layer that uses no permutation arrays and its own scalar encoders.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

from oracle import formats as F
from oracle import moe as M
from synth import CONFIGS, expert_weights, make_inputs


# ----------------------------------------------------------------------------- routing
def _route_brute(lp_row, k):
    E = len(lp_row)
    order = sorted(range(E), key=lambda e: (-float(lp_row[e]), e))[:k]
    m = float(lp_row[order[0]])
    p = [math.exp(float(lp_row[e]) - m) for e in order]
    s = math.fsum(p)
    return order, [v / s for v in p]


@pytest.mark.parametrize("T,E,k", [(16, 8, 2), (7, 33, 5), (5, 128, 8), (3, 513, 10)])
def test_route_vs_brute_force(T, E, k):
    rng = np.random.default_rng(T * E + k)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.5).astype(np.float32)
    ids, w = M.route(logits, bias, k, True)
    lp = (logits + bias).astype(np.float32)
    for t in range(T):
        order, wt = _route_brute(lp[t], k)
        assert list(ids[t]) == order
        assert np.allclose(w[t], wt, rtol=1e-14, atol=0)
        assert len(set(ids[t])) == k
        assert abs(w[t].sum() - 1) < 1e-12


def test_route_forced_ties():
    logits = np.zeros((4, 16), np.float32)
    ids, w = M.route(logits, None, 5, True)
    assert np.all(ids == np.arange(5)) and np.allclose(w, 0.2)
    logits[:, 3] = 1.0
    logits[:, 9] = 1.0
    ids, _ = M.route(logits, None, 3, True)
    assert np.all(ids == [3, 9, 0])


def test_route_not_renormalised_is_full_softmax():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((6, 20)).astype(np.float32)
    ids, w = M.route(logits, None, 4, False)
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(full, ids.astype(np.int64), 1), rtol=1e-12)


def test_zipf_bias_skews_routing():
    cfg = CONFIGS["skewed"].scaled(T=512)
    x, logits, bias = make_inputs(cfg, seed=0)
    ids, _ = M.route(logits.numpy(), bias.numpy(), cfg.k, True)
    counts = np.bincount(ids.reshape(-1), minlength=cfg.E)
    assert counts[0] > counts[50] > 0 and (counts == 0).sum() > 50


# ----------------------------------------------------------------------------- permutation
@pytest.mark.parametrize("shared", [False, True])
def test_permute_vs_brute_force(shared):
    rng = np.random.default_rng(11)
    T, E, k = 37, 12, 3
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, p2s, s2p = M.permute(ids, E, shared)
    flat = list(ids.reshape(-1)) + ([E] * T if shared else [])
    E_tot = E + int(shared)
    # brute force: walk experts in order, append assignments in index order
    ref = [a for e in range(E_tot) for a in range(len(flat)) if flat[a] == e]
    assert list(p2s) == ref
    assert sorted(p2s) == list(range(len(flat)))
    assert np.all(s2p[p2s] == np.arange(len(flat)))
    assert list(counts) == [flat.count(e) for e in range(E_tot)]
    assert offsets[0] == 0 and offsets[-1] == len(flat)
    if shared:
        assert list(p2s[T * k:]) == list(range(T * k, T * k + T))
        assert list(M.assignment_token(p2s[T * k:], T, k)) == list(range(T))


def test_tile_offsets():
    counts = [0, 1, 127, 128, 129, 8065]
    to = M.tile_offsets(counts)
    ref = [0]
    for c in counts:
        ref.append(ref[-1] + -(-c // 128))
    assert list(to) == ref


# ----------------------------------------------------------------------------- GEMM
def _exact_dot(qa, sa, qb, sb):
    acc = Fraction(0)
    for i in range(len(qa)):
        va = Fraction(F.e2m1_decode(qa[i]).item()) * Fraction(F.e4m3_decode(sa[i // 16]).item())
        vb = Fraction(F.e2m1_decode(qb[i]).item()) * Fraction(F.e4m3_decode(sb[i // 16]).item())
        acc += va * vb
    return acc


def test_block_scaled_matmul_exact_rational():
    rng = np.random.default_rng(12)
    m, n, K = 5, 4, 128
    qa = rng.integers(0, 16, (m, K)).astype(np.uint8)
    qb = rng.integers(0, 16, (n, K)).astype(np.uint8)
    sa = rng.integers(0, 0x7F, (m, K // 16)).astype(np.uint8)
    sb = rng.integers(0, 0x7F, (n, K // 16)).astype(np.uint8)
    pack = lambda q: (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    S = M.block_scaled_matmul(pack(qa), sa, pack(qb), sb)
    for i in range(m):
        for j in range(n):
            exact = _exact_dot(qa[i], sa[i], qb[j], sb[j])
            assert abs(Fraction(S[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)


def test_grouped_gemm_groups_and_alpha():
    rng = np.random.default_rng(13)
    K, N = 64, 8
    sizes = [0, 1, 3, 0, 5]
    offsets = np.concatenate([[0], np.cumsum(sizes)])
    R, G = offsets[-1], len(sizes)
    a = rng.standard_normal((R, K)).astype(np.float32)
    ac, asc = F.quantize_rows(a, np.float32(0.01))
    w = rng.standard_normal((G, N, K)).astype(np.float32)
    wc = np.stack([F.quantize_rows(w[g], np.float32(0.02))[0] for g in range(G)])
    ws = np.stack([F.quantize_rows(w[g], np.float32(0.02))[1] for g in range(G)])
    gs_a = np.full(G, 0.01, np.float32)
    gs_w = np.full(G, 0.02, np.float32)
    D = M.grouped_gemm(ac, asc, offsets, gs_a, wc, ws, gs_w)
    for g in range(G):
        for p in range(offsets[g], offsets[g + 1]):
            da = F.dequantize_rows(ac[p:p + 1], asc[p:p + 1])[0] * float(np.float32(0.01))
            dw = F.dequantize_rows(wc[g], ws[g]) * float(np.float32(0.02))
            # alpha is rounded to float32 once; compare with a relative bound
            assert np.allclose(D[p], dw @ da, rtol=1e-6, atol=1e-12)


# ----------------------------------------------------------------------------- epilogue, combine
def test_swiglu_identities():
    g = np.linspace(-20, 20, 401)
    c = np.stack([g, np.ones_like(g)], 1)
    h = M.swiglu(c, 1)[:, 0]
    hn = M.swiglu(np.stack([-g, np.ones_like(g)], 1), 1)[:, 0]  # silu(-g) * 1
    assert h[200] == 0.0
    assert np.allclose(h - hn, g, rtol=1e-13, atol=1e-13)       # silu(g) - silu(-g) = g
    assert np.allclose(h, g * scipy.special.expit(g), rtol=1e-13, atol=1e-300)
    z = M.swiglu(np.stack([g, np.zeros_like(g)], 1), 1)
    assert np.all(z == 0)


def test_combine_k1_is_unpermute():
    rng = np.random.default_rng(14)
    T, E, H = 9, 4, 6
    ids = rng.integers(0, E, (T, 1)).astype(np.int32)
    _, _, p2s, s2p = M.permute(ids, E, False)
    y = rng.standard_normal((T, H))
    yp = y[p2s]                                  # rows in permuted order
    out = M.combine(yp, np.ones((T, 1)), s2p, T, 1, False)
    assert np.array_equal(out, y)


def test_combine_k_equals_E_is_dense_mixture():
    rng = np.random.default_rng(15)
    T, E, H = 5, 6, 3
    logits = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = M.route(logits, None, E, True)
    _, _, p2s, s2p = M.permute(ids, E, False)
    ye = rng.standard_normal((E, T, H))         # expert e applied to token t
    tok = M.assignment_token(p2s, T, E)
    y = np.stack([ye[ids.reshape(-1)[a], tok[i]] for i, a in enumerate(p2s)])
    out = M.combine(y, w, s2p, T, E, False)
    dense = np.einsum("te,eth->th", scipy.special.softmax(logits.astype(np.float64), 1), ye)
    assert np.allclose(out, dense, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- end to end
def _scalar_quant_block(vals, gs):
    """Independent scalar NVFP4 block quantizer (threshold-table E2M1, formula E4M3)."""
    from tests.test_oracle_formats import _e2m1_threshold, _e4m3_formula
    f32 = np.float32
    amax = max(abs(f32(v)) for v in vals)
    t2 = f32(amax) / (f32(6.0) * f32(gs))
    sb = _e4m3_formula(float(t2))
    d = f32(F.e4m3_value(sb))
    t3 = f32(d * f32(gs))
    r = f32(0.0) if t3 == 0 else f32(f32(1.0) / t3)
    return [_e2m1_threshold(float(f32(f32(v) * r))) for v in vals], sb


def _scalar_quant_row(row, gs):
    codes, scales = [], []
    for b in range(0, len(row), 16):
        q, s = _scalar_quant_block(row[b:b + 16], gs)
        codes += q
        scales.append(s)
    return codes, scales


def _deq(codes, scales):
    return [F.E2M1_MAGNITUDES[c & 7] * (-1 if c & 8 else 1) * F.e4m3_value(scales[i // 16])
            for i, c in enumerate(codes)]


def _weights_for(cfg, seed=0):
    cache = {}

    def get(e):
        if e not in cache:
            w13, w2 = expert_weights(cfg, e, seed)
            c13, s13, g13 = M.quantize_expert_weights(w13.numpy())
            c2, s2, g2 = M.quantize_expert_weights(w2.numpy())
            cache[e] = (c13, s13, g13, c2, s2, g2)
        return cache[e]
    return get


def test_tiny_layer_per_token_walk():
    """Walk each token through its k experts directly: no permutation arrays,
    scalar encoders, math.fsum dot products."""
    cfg = CONFIGS["tiny"]
    x, logits, bias = make_inputs(cfg, seed=0)
    xf = x.to(torch.float32).numpy()
    wts = _weights_for(cfg)
    gs_a1 = np.full(cfg.E, F.global_scale(np.max(np.abs(xf))), np.float32)
    gs_a2 = np.full(cfg.E, np.float32(0.004), np.float32)
    ref = M.moe_forward(xf, logits.numpy(), None, cfg.k, True, False, wts, gs_a1, gs_a2)
    lp = logits.numpy()
    I, H = cfg.I, cfg.H
    for t in range(cfg.T):
        order, wt = _route_brute(lp[t], cfg.k)
        acc = np.zeros(H)
        xc, xs = _scalar_quant_row(xf[t], gs_a1[0])
        dx = _deq(xc, xs)
        for j, e in enumerate(order):
            c13, s13, g13, c2, s2, g2 = wts(e)
            a1 = float(np.float32(gs_a1[e] * g13))
            W13 = F.dequantize_rows(c13, s13)
            c1 = [a1 * math.fsum(dx[i] * W13[n, i] for i in range(H)) for n in range(2 * I)]
            h = [np.float32(c1[n] / (1 + math.exp(-c1[n])) * c1[I + n]) for n in range(I)]
            hc, hs = _scalar_quant_row(h, gs_a2[e])
            p = ref["src_to_perm"][t * cfg.k + j]
            assert list(F.unpack_codes(ref["a1_codes"][p])) == xc
            assert list(ref["a1_scales"][p]) == xs
            assert np.allclose(ref["h"][p], h, rtol=1e-6, atol=1e-9)
            assert list(F.unpack_codes(ref["a2_codes"][p])) == hc
            assert list(ref["a2_scales"][p]) == hs
            dh = _deq(hc, hs)
            W2 = F.dequantize_rows(c2, s2)
            a2 = float(np.float32(gs_a2[e] * g2))
            y = [a2 * math.fsum(dh[i] * W2[n, i] for i in range(I)) for n in range(H)]
            assert np.allclose(ref["y"][p], y, rtol=1e-12, atol=1e-15)
            acc += wt[j] * np.array(y)
        assert np.allclose(ref["out"][t], acc, rtol=1e-10, atol=1e-13)


def test_single_expert_is_plain_swiglu_mlp():
    """E = 1, k = 1: the layer is an NVFP4 SwiGLU MLP, written here as dense math."""
    rng = np.random.default_rng(16)
    T, H, I = 6, 64, 32
    x = rng.standard_normal((T, H)).astype(np.float32)
    w13 = (rng.standard_normal((2 * I, H)) * 0.02).astype(np.float32)
    w2 = (rng.standard_normal((H, I)) * 0.02).astype(np.float32)
    q = (M.quantize_expert_weights(w13), M.quantize_expert_weights(w2))
    wts = lambda e: (*q[0], *q[1])
    gs1 = np.array([F.global_scale(np.abs(x).max())], np.float32)
    gs2 = np.array([np.float32(0.001)], np.float32)
    ref = M.moe_forward(x, np.zeros((T, 1), np.float32), None, 1, True, False, wts, gs1, gs2)
    xc, xs = F.quantize_rows(x, gs1[0])
    dx = F.dequantize_rows(xc, xs) * float(gs1[0])
    dw13 = F.dequantize_rows(q[0][0], q[0][1]) * float(q[0][2])
    c1 = dx @ dw13.T
    hh = (c1[:, :I] * scipy.special.expit(c1[:, :I]) * c1[:, I:]).astype(np.float32)
    hc, hs = F.quantize_rows(hh, gs2[0])
    out = (F.dequantize_rows(hc, hs) * float(gs2[0])) @ (F.dequantize_rows(q[1][0], q[1][1]) * float(q[1][2])).T
    assert np.allclose(ref["out"], out, rtol=1e-5, atol=1e-7)
