"""Plain CPU definition of the NVFP4 MoE expert computation, step by step.

Steps (the data-parallel path the source pages keep returning to): top-k
routing, permutation of tokens by expert, NVFP4 activation quantization, a
grouped block-scaled FP4 GEMM for gate_up, SiLU(gate) * up with
requantization, a grouped FP4 GEMM for down, and a weighted top-k combine.

Citations:
  * top-k routing with many routed experts plus one shared expert, k per
    token -- FlashInfer issue #2723, "Model" table (512 routed + 1 shared,
    10 routed per token);
  * per-expert problem sizes and offsets for the grouped GEMM -- vLLM PR
    #29242, review of nvfp4_blockwise_moe_kernel.cu (error text listing
    num_experts, M, N, K) and the commit "Fix get_cutlass_moe_mm_data not
    compiling";
  * per-expert alpha applied in the GEMM epilogue with beta = 0 -- vLLM PR
    #29242, review of nvfp4_blockwise_moe_kernel.cu (alpha_ptr_array, dAlpha,
    beta = 0.0f);
  * the grouped GEMM is the MoE expert computation -- FlashInfer issue #2723,
    "The Problem".
Readings where the pages are silent (each listed in the design notes):
  * selection on FP32 logit + bias, descending, ties to the lower expert id;
    weights are a softmax over the k selected logits (renormalised) or over
    all E logits (not renormalised);
  * the permutation is a stable sort of the assignments a = t*k + j by expert;
    the shared expert (id E, weight 1) takes T more rows a = T*k + t at the end;
  * w13 rows [0, I) are gate, [I, 2I) are up; h = silu(gate) * up;
  * alpha_e = gs_act[e] * gs_w[e] (one FP32 multiply);
  * GEMM sums are exact products accumulated in float64.
"""
from __future__ import annotations

import numpy as np

from . import formats as F

F32 = np.float32
TILE_M = 128


# ----------------------------------------------------------------------------- router gate
def router_logits(x, w_gate):
    """Router gate, the step before routing: logits[t, j] = sum_h x[t, h] *
    w_gate[j, h] for bf16 activations x [T, H] and bf16 gate rows w_gate
    [n, H] (given here as their exact float values).  Every product of two bf16
    values is exact in float64 and the sum is taken in float64, then rounded
    once to float32 (the logits' type).  The pages name the routed experts the
    gate scores (FlashInfer issue #2723, "Model" table: 512 routed + 1 shared,
    10 per token) but give no gate formula; reading: a plain linear gate
    without bias, one row per routed expert, plus optionally one row whose
    logit gates the shared expert (shared_gate)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w_gate, dtype=np.float64)
    return (x @ w.T).astype(F32)


def shared_gate(gate_logit):
    """Weight of the shared expert's output: sigmoid of its gate logit, float64.
    Reading (the pages give no formula): sigmoid(z) = 1 / (1 + exp(-z))."""
    z = np.asarray(gate_logit, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


# ----------------------------------------------------------------------------- routing
def route(logits, bias, k: int, renormalize: bool = True):
    """Top-k selection and softmax weights.

    l'_e = logit_e + bias_e in FP32; the k largest l' in descending order, ties
    to the lower e; p_j = exp(l'_j - l'_max) in float64; w_j = p_j / sum(p).
    Returns ids int32 [T,k] and weights float64 [T,k].
    """
    lp = np.asarray(logits, dtype=F32)
    if bias is not None:
        lp = (lp + np.asarray(bias, dtype=F32)[None, :]).astype(F32)
    T, E = lp.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    # Stable sort of -l' keeps equal values in increasing expert order.
    order = np.argsort(-lp, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(lp, order, axis=1).astype(np.float64)
    m = sel[:, :1]
    p = np.exp(sel - m)
    if renormalize:
        denom = p.sum(axis=1, keepdims=True)
    else:
        denom = np.exp(lp.astype(np.float64) - m).sum(axis=1, keepdims=True)
    return order.astype(np.int32), p / denom


def permute(ids, E: int, shared: bool = False):
    """Stable permutation of assignments by expert.

    counts_e = #{a : e_a = e}; offsets = exclusive prefix (length E' + 1);
    perm_to_src[p] = a for the p-th assignment in (expert, a) order;
    src_to_perm = its inverse.  With a shared expert its T rows follow all
    routed rows in token order.
    """
    ids = np.asarray(ids, dtype=np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)
    if shared:
        flat = np.concatenate([flat, np.full(T, E, dtype=np.int64)])
    E_tot = E + (1 if shared else 0)
    counts = np.bincount(flat, minlength=E_tot).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    perm_to_src = np.argsort(flat, kind="stable").astype(np.int64)
    src_to_perm = np.empty_like(perm_to_src)
    src_to_perm[perm_to_src] = np.arange(len(flat))
    return counts, offsets, perm_to_src, src_to_perm


def assignment_token(a, T: int, k: int):
    """Token of assignment a: a // k for routed rows, a - T*k for shared rows."""
    a = np.asarray(a, dtype=np.int64)
    return np.where(a < T * k, a // k, a - T * k)


def tile_offsets(counts):
    """Exclusive prefix of ceil(m_e / 128): the 128-row M tiles of each expert."""
    tiles = (np.asarray(counts, dtype=np.int64) + TILE_M - 1) // TILE_M
    return np.concatenate([[0], np.cumsum(tiles)]).astype(np.int64)


# ----------------------------------------------------------------------------- GEMMs
def block_scaled_matmul(a_codes, a_scales, b_codes, b_scales) -> np.ndarray:
    """S = dA @ dB^T, float64, over dequantized operands without global scales.

    Every product dA * dB is exact (each factor has at most 5 significant bits);
    the float64 sum is the reference accumulation.
    """
    return F.dequantize_rows(a_codes, a_scales) @ F.dequantize_rows(b_codes, b_scales).T


def alpha(gs_a, gs_w) -> np.float32:
    """Per-expert epilogue scale alpha = gs_act * gs_w, one FP32 multiply."""
    return F32(F32(gs_a) * F32(gs_w))


def grouped_gemm(a_codes, a_scales, offsets, gs_a, w_codes, w_scales, gs_w):
    """D[p] = alpha_e * (A[p] . W_e^T) for rows p of group e (float64 result).

    a_codes [R, K/2], a_scales [R, K/16]; w_codes [G, N, K/2], w_scales [G, N, K/16];
    offsets [G+1]; gs_a, gs_w [G].
    """
    G, N = w_codes.shape[0], w_codes.shape[1]
    R = a_codes.shape[0]
    out = np.zeros((R, N), dtype=np.float64)
    for e in range(G):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        s = block_scaled_matmul(a_codes[lo:hi], a_scales[lo:hi], w_codes[e], w_scales[e])
        out[lo:hi] = np.float64(alpha(gs_a[e], gs_w[e])) * s
    return out


def w4a16_matmul(a, w_codes, w_scales, gs_w):
    """Weight-only NVFP4 product (the W4A16 decode alternative the pages compare
    against, e.g. Marlin W4A16 in FlashInfer issue #2723, "Speed Comparison",
    and the W4A16 columns of the unsloth report's per-GEMM table):
    D = gs_w * (A . dW^T) with A the bf16 activations (as exact float values,
    no quantization) and dW = e2m1 * e4m3 of the weight blocks.  Every product
    is exact in float64 and the sum is float64."""
    a = np.asarray(a, dtype=np.float64)
    return np.float64(F32(gs_w)) * (a @ F.dequantize_rows(w_codes, w_scales).T)


def grouped_w4a16(a, offsets, w_codes, w_scales, gs_w):
    """D[p] = w4a16_matmul(A[p], W_e) for the rows p of group e (float64)."""
    G, N = w_codes.shape[0], w_codes.shape[1]
    out = np.zeros((np.asarray(a).shape[0], N), dtype=np.float64)
    for e in range(G):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            out[lo:hi] = w4a16_matmul(np.asarray(a)[lo:hi], w_codes[e], w_scales[e], gs_w[e])
    return out


def swiglu(c1, I: int) -> np.ndarray:
    """h = silu(g) * u = g / (1 + exp(-g)) * u, float64, for g = C1[:, :I], u = C1[:, I:]."""
    c1 = np.asarray(c1, dtype=np.float64)
    g, u = c1[:, :I], c1[:, I:2 * I]
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def combine(y, weights, src_to_perm, T: int, k: int, shared: bool, shared_weight=None):
    """out[t] = sum_j w[t,j] * y[src_to_perm[t*k+j]] (+ g[t] * y of the shared row), float64.
    g[t] = 1 without a shared-expert gate, else shared_weight[t]."""
    y = np.asarray(y, dtype=np.float64)
    w = np.asarray(weights, dtype=np.float64)
    rows = np.asarray(src_to_perm[: T * k]).reshape(T, k)
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for j in range(k):                       # slot order
        out += w[:, j:j + 1] * y[rows[:, j]]
    if shared:
        ys = y[np.asarray(src_to_perm[T * k: T * k + T])]
        out += ys if shared_weight is None else np.asarray(shared_weight, np.float64)[:, None] * ys
    return out


# ----------------------------------------------------------------------------- weights
def quantize_expert_weights(w_fp32):
    """Per-expert weight prep: gs = amax/2688, then NVFP4 rows along K (the input dim)."""
    w = np.asarray(w_fp32, dtype=F32)
    gs = F.global_scale(np.max(np.abs(w)))
    codes, scales = F.quantize_rows(w, gs)
    return codes, scales, gs


# ----------------------------------------------------------------------------- layer
def moe_forward(x, logits, bias, k, renormalize, shared, weights, gs_a1, gs_a2, experts=None, shared_gate_logit=None):
    """Whole layer, returning every intermediate.

    x        : float32 [T, H] (the bf16 activations, exactly converted)
    weights  : callable e -> (w13_codes, w13_scales, gs_w13, w2_codes, w2_scales, gs_w2)
               for e in 0..E'-1 (canonical row order: gate rows then up rows)
    gs_a1/2  : float32 [E'] static activation global scales
    experts  : optional set of experts to evaluate; rows of other experts are
               left as NaN (for sampled checks of large layers).
    shared_gate_logit : optional float32 [T]: the shared expert's output is
               scaled by shared_gate(logit) instead of 1.
    """
    x = np.asarray(x, dtype=F32)
    T, H = x.shape
    E = np.asarray(logits).shape[1]
    ids, w = route(logits, bias, k, renormalize)
    counts, offsets, p2s, s2p = permute(ids, E, shared)
    E_tot = E + (1 if shared else 0)
    R = len(p2s)
    tok = assignment_token(p2s, T, k)
    a1_codes = np.zeros((R, H // 2), np.uint8)
    a1_scales = np.zeros((R, H // 16), np.uint8)
    out = dict(ids=ids, weights=w, counts=counts, offsets=offsets, perm_to_src=p2s,
               src_to_perm=s2p, perm_token=tok, a1_codes=a1_codes, a1_scales=a1_scales)
    I = None
    y = h = a2_codes = a2_scales = c1 = None
    for e in range(E_tot):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo or (experts is not None and e not in experts):
            continue
        w13c, w13s, gw13, w2c, w2s, gw2 = weights(e)
        if I is None:
            I = w13c.shape[0] // 2
            c1 = np.full((R, 2 * I), np.nan)
            h = np.full((R, I), np.nan, dtype=F32)
            a2_codes = np.zeros((R, I // 2), np.uint8)
            a2_scales = np.zeros((R, I // 16), np.uint8)
            y = np.full((R, H), np.nan)
        ac, asc = F.quantize_rows(x[tok[lo:hi]], gs_a1[e])
        a1_codes[lo:hi], a1_scales[lo:hi] = ac, asc
        c1[lo:hi] = np.float64(alpha(gs_a1[e], gw13)) * block_scaled_matmul(ac, asc, w13c, w13s)
        he = swiglu(c1[lo:hi], I).astype(F32)
        h[lo:hi] = he
        qc, qs = F.quantize_rows(he, gs_a2[e])
        a2_codes[lo:hi], a2_scales[lo:hi] = qc, qs
        y[lo:hi] = np.float64(alpha(gs_a2[e], gw2)) * block_scaled_matmul(qc, qs, w2c, w2s)
    out.update(c1=c1, h=h, a2_codes=a2_codes, a2_scales=a2_scales, y=y)
    sw = None if shared_gate_logit is None else shared_gate(shared_gate_logit)
    out["out"] = combine(y, w, s2p, T, k, shared, sw) if y is not None else None
    return out
