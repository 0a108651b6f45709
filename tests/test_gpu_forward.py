"""End-to-end GPU parity of nvfp4_moe_forward against the oracle.

Bit-exact against the oracle: routing ids, offsets, permutation, A1 codes
and scales, and the prepared codes, scales and global scales of every expert
the oracle evaluates.  Within 5e-3 * rms(oracle): routing weights (1e-6
relative), h, y and out (FP32 output; BF16 output adds one BF16 rounding).

A2 (the requantized h) is compared bit-exactly against the quantization of
the GPU's own h (an independent checker, not the oracle).  Against the
oracle's own A2 it may differ where h sits on a rounding boundary (GPU and
oracle sum GEMM1 in different orders): such code flips must be rare
(<= 1e-4 of the codes), each at most one E2M1 step, and each flipped block
scale at most one E4M3 code.  y and out are then held to the strict bound
against the oracle's down GEMM and combine applied to the GPU's own A2, and,
as an extra check, against the oracle's own y and out with the flips' exact
effect added.  Large layers are checked on sampled tokens: the oracle
evaluates only the experts those tokens visit.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import moe as M
from synth import CONFIGS, expert_weights, make_inputs
from tests import oracle_pool
from tests.nvf_testutil import (ROOT, dequant_check, ensure_built, quantize_rows_check, rel_err, row_tiles,
                                 tiled_unpack, w13_prepared_rows, weight_index)

pytestmark = pytest.mark.gpu
TOL = 5e-3
SCALES = json.load(open(os.path.join(ROOT, "tests", "golden", "activation_scales.json")))
_PREPARED = {}


@pytest.fixture(scope="module")
def nvf():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as m
    return m


class Layer:
    """A synthetic layer.  Weights are drawn on `wdev` ("cpu": the CPU generator,
    uploaded; "cuda": torch's CUDA generator) and prepared by the library; the
    oracle quantizes its own copy of every expert it needs."""

    def __init__(self, nvf, cfg, seed=0, parent=None, wdev="cpu"):
        self.nvf, self.cfg, self.seed, self.wdev = nvf, cfg, seed, wdev
        # activations and logits from the CPU generator (the recipe the stored
        # activation scales were calibrated on), uploaded
        x, logits, bias = make_inputs(cfg, seed, device="cpu")
        self.x, self.logits = x.cuda(), logits.cuda()
        self.bias = None if bias is None else bias.cuda()
        key = (cfg.H, cfg.I, cfg.E, cfg.shared, seed, wdev)
        if key not in _PREPARED:
            _PREPARED.clear()   # keep one weight set resident
            w = nvf.prepare_weights(cfg.E, cfg.H, cfg.I, cfg.shared,
                                    lambda e: expert_weights(cfg, e, seed, device=wdev))
            _PREPARED[key] = (w, {})
        self.wts, self.ocache = _PREPARED[key]
        sc = SCALES[parent or cfg.name]
        self.gs_a1 = np.full(cfg.E_total, sc["gs_a1"], np.float32)
        self.gs_a2 = np.full(cfg.E_total, sc["gs_a2"], np.float32)

    def need(self, experts):
        todo = [e for e in experts if e not in self.ocache]
        if not todo:
            return
        if self.wdev == "cpu":
            self.ocache.update(oracle_pool.quantize_generated(self.cfg, todo, self.seed))
        else:
            for i in range(0, len(todo), 16):
                pairs = {e: tuple(t.cpu().numpy() for t in expert_weights(self.cfg, e, self.seed, device="cuda"))
                         for e in todo[i:i + 16]}
                self.ocache.update(oracle_pool.quantize_arrays(pairs))

    def run(self, out_dtype=torch.float32, h_dump=True, ws=None):
        cfg, nvf = self.cfg, self.nvf
        L = nvf.workspace_layout(cfg.T, cfg.E, cfg.H, cfg.I, cfg.k, cfg.shared)
        if ws is None:
            ws = torch.zeros(max(L["total"], 256), dtype=torch.uint8, device="cuda")
        h = torch.full((L["R"], cfg.I), float("nan"), device="cuda") if h_dump else None
        out = nvf.moe_forward(self.wts, self.x, self.logits, cfg.k, torch.tensor(self.gs_a1, device="cuda"),
                              torch.tensor(self.gs_a2, device="cuda"), bias=self.bias,
                              renormalize=cfg.renormalize, out_dtype=out_dtype, h_dump=h, ws=ws)
        code, detail = nvf.device_status()
        assert code == 0, f"device error word {code} at {detail}"
        return out, ws, L, h


def _ws_view(ws, L, name, n, dtype):
    return ws[L[name]:L[name] + n * np.dtype(dtype).itemsize].cpu().numpy().view(dtype)


def check_layer(nvf, layer, out_dtype=torch.float32, tokens=None):
    cfg = layer.cfg
    out, ws, L, h_gpu = layer.run(out_dtype)
    R, Et = L["R"], cfg.E_total
    xf = layer.x.float().cpu().numpy()
    lg = layer.logits.cpu().numpy()
    bias = None if layer.bias is None else layer.bias.cpu().numpy()
    ids, _ = M.route(lg, bias, cfg.k, cfg.renormalize)
    if tokens is None:
        experts = sorted(set(ids.reshape(-1).tolist()) | ({cfg.E} if cfg.shared else set()))
    else:
        experts = sorted(set(ids[tokens].reshape(-1).tolist()) | ({cfg.E} if cfg.shared else set()))
    layer.need(experts)
    ref = M.moe_forward(xf, lg, bias, cfg.k, cfg.renormalize, cfg.shared, lambda e: layer.ocache[e],
                        layer.gs_a1, layer.gs_a2, experts=None if tokens is None else set(experts))
    offs = _ws_view(ws, L, "expert_offsets", Et + 1, np.int32)
    tiles = _ws_view(ws, L, "tile_offsets", Et + 1, np.int32)
    assert np.array_equal(_ws_view(ws, L, "topk_ids", cfg.T * cfg.k, np.int32).reshape(cfg.T, cfg.k), ref["ids"])
    assert np.allclose(_ws_view(ws, L, "topk_w", cfg.T * cfg.k, np.float32).reshape(cfg.T, cfg.k), ref["weights"],
                       rtol=1e-6, atol=1e-7)
    assert np.array_equal(offs, ref["offsets"])
    assert np.array_equal(_ws_view(ws, L, "perm_to_src", R, np.int32), ref["perm_to_src"])
    assert np.array_equal(_ws_view(ws, L, "src_to_perm", R, np.int32), ref["src_to_perm"])
    assert np.array_equal(_ws_view(ws, L, "perm_token", R, np.int32), ref["perm_token"])
    assert np.array_equal(tiles, M.tile_offsets(ref["counts"]))
    rows = np.zeros(R, bool)
    for e in experts:
        rows[offs[e]:offs[e + 1]] = True
    wsn = ws.cpu().numpy()
    tr = row_tiles(R, offs, tiles)
    a1c, a1s = tiled_unpack(wsn[L["a1"]:L["a2"]], cfg.H, *tr)
    a2c, a2s = tiled_unpack(wsn[L["a2"]:L["y"]], cfg.I, *tr)
    if out_dtype == torch.bfloat16:   # y is kept in the output's precision
        y = ws[L["y"]:L["y"] + R * cfg.H * 2].view(torch.bfloat16).float().cpu().numpy().reshape(R, cfg.H)
    else:
        y = _ws_view(ws, L, "y", R * cfg.H, np.float32).reshape(R, cfg.H)
    # one BF16 rounding of y (relative 2^-9, bounded here by 2^-8) when the output is BF16
    y_round = 2.0 ** -8 if out_dtype == torch.bfloat16 else 0.0
    h = h_gpu.cpu().numpy()
    assert np.array_equal(a1c[rows], ref["a1_codes"][rows])
    assert np.array_equal(a1s[rows], ref["a1_scales"][rows])
    # prepared weights of every expert the oracle evaluates equal the oracle's
    # quantization (w13 rows in the prepared order)
    check_prepared_weights(nvf, layer, experts)
    assert rel_err(h[rows], ref["h"][rows]) <= TOL
    # A2 is a valid requantization of the GPU's own h (independent checker, bit-exact)
    gs2_rows = np.repeat(layer.gs_a2, np.diff(offs))
    qc, qs = quantize_rows_check(h[rows], gs2_rows[rows])
    assert np.array_equal(a2c[rows], qc)
    assert np.array_equal(a2s[rows], qs)
    # Against the oracle's own A2 (from its float64 h): an h on a rounding
    # boundary may round either way.  Flips must be rare and one step each.
    g_codes, r_codes = F.unpack_codes(a2c[rows]), F.unpack_codes(ref["a2_codes"][rows])
    code_diff = g_codes != r_codes
    assert code_diff.mean() <= 1e-4, code_diff.mean()
    assert np.max(np.abs(e2m1_signed_index(g_codes) - e2m1_signed_index(r_codes)), initial=0) <= 1
    assert np.max(np.abs(a2s[rows].astype(np.int64) - ref["a2_scales"][rows].astype(np.int64)), initial=0) <= 1
    # y and out: the oracle's down GEMM (O10) and combine (O11) applied to the
    # GPU's own A2, strict 5e-3 * rms
    y_own = np.full((R, cfg.H), np.nan)
    for e in experts:
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        c2, s2, g2 = layer.ocache[e][3:]
        y_own[lo:hi] = np.float64(M.alpha(layer.gs_a2[e], g2)) * M.block_scaled_matmul(a2c[lo:hi], a2s[lo:hi], c2, s2)
    y_rms_own = np.sqrt(np.mean(y_own[rows] ** 2))
    assert np.all(np.abs(y[rows] - y_own[rows]) <= TOL * y_rms_own + y_round * np.abs(y_own[rows]))
    tsel = np.arange(cfg.T) if tokens is None else np.asarray(tokens)
    out_own = M.combine(y_own, ref["weights"], ref["src_to_perm"], cfg.T, cfg.k, cfg.shared)[tsel]
    o = out.float().cpu().numpy()[tsel]
    rms_own = np.sqrt(np.mean(out_own ** 2))
    bound = TOL * rms_own
    if out_dtype == torch.bfloat16:
        # one bf16 rounding of each y row the combine reads and one of the output
        mag = M.combine(np.abs(y_own), np.abs(ref["weights"]), ref["src_to_perm"], cfg.T, cfg.k, cfg.shared)[tsel]
        bound = bound + (mag + np.abs(out_own)) * 2.0 ** -8
    assert np.all(np.abs(o - out_own) <= bound)
    # Extra check against the oracle's own y and out: rows whose A2 matches are
    # within the bound; a row whose A2 flipped may differ further by exactly
    # what the flip explains, alpha2 * |W2| . |dA2 - dA2_oracle|.
    row_diff = np.zeros(R, bool)
    row_diff[rows] = code_diff.any(1) | (a2s[rows] != ref["a2_scales"][rows]).any(1)
    y_rms = np.sqrt(np.mean(ref["y"][rows] ** 2))
    explained = np.zeros((R, cfg.H))
    for p in np.nonzero(row_diff)[0]:
        e = int(np.searchsorted(offs, p, side="right") - 1)
        c2, s2, g2 = layer.ocache[e][3:]
        d = np.abs(dequant_check(a2c[p:p + 1], a2s[p:p + 1]) - dequant_check(ref["a2_codes"][p:p + 1],
                                                                             ref["a2_scales"][p:p + 1]))[0]
        alpha2 = float(np.float32(np.float32(layer.gs_a2[e]) * np.float32(g2)))
        explained[p] = alpha2 * (np.abs(dequant_check(c2, s2)) @ d)
    same = rows & ~row_diff
    yr = y_round * np.abs(ref["y"])
    assert np.all(np.abs(y[same] - ref["y"][same]) <= TOL * y_rms + yr[same])
    assert np.all(np.abs(y[rows] - ref["y"][rows]) <= TOL * y_rms + 1.001 * explained[rows] + yr[rows])
    s2p = ref["src_to_perm"]
    w = ref["weights"]
    ex_out = np.zeros((cfg.T, cfg.H))
    for t in tsel:
        for j in range(cfg.k):
            ex_out[t] += w[t, j] * explained[s2p[t * cfg.k + j]]
        if cfg.shared:
            ex_out[t] += explained[s2p[cfg.T * cfg.k + t]]
    r = ref["out"][tsel]
    slack = TOL * np.sqrt(np.mean(r ** 2)) + 1.001 * ex_out[tsel]
    if out_dtype == torch.bfloat16:
        mag = M.combine(np.abs(ref["y"]), np.abs(ref["weights"]), ref["src_to_perm"], cfg.T, cfg.k, cfg.shared)[tsel]
        slack = slack + (mag + np.abs(r)) * 2.0 ** -8
    assert np.all(np.abs(o - r) <= slack)
    return out


def e2m1_signed_index(codes):
    """Position of an E2M1 code on the signed value line (-6 .. 6 -> -7 .. 7;
    +0 and -0 share position 0): one E2M1 step is a difference of one."""
    c = np.asarray(codes).astype(np.int64)
    return np.where(c & 8, -(c & 7), c & 7)


def check_prepared_weights(nvf, layer, experts):
    """Codes, scales and global scales the library prepared for each expert
    equal the oracle's quantization of the same FP32 weights.  The tiled
    buffers are gathered into canonical [rows, K/2] / [rows, K/16] views on the
    device (index arrays from the layout stated in include/nvfp4moe.h)."""
    cfg = layer.cfg
    n13, n2 = nvf.tiled_bytes(2 * cfg.I, 0, cfg.H), nvf.tiled_bytes(cfg.H, 0, cfg.I)
    perm = w13_prepared_rows(cfg.I)
    i13 = [torch.from_numpy(a.astype(np.int64)).cuda() for a in weight_index(2 * cfg.I, cfg.H, 2 * cfg.I)]
    i2 = [torch.from_numpy(a.astype(np.int64)).cuda() for a in weight_index(cfg.H, cfg.I, cfg.H)]
    g13_all = layer.wts.gs_w13.cpu().numpy()
    g2_all = layer.wts.gs_w2.cpu().numpy()
    for e in experts:
        c13, s13, g13, c2, s2, g2 = layer.ocache[e]
        b13 = layer.wts.w13[e * n13:(e + 1) * n13]
        b2 = layer.wts.w2[e * n2:(e + 1) * n2]
        assert np.array_equal(b13[i13[0]].cpu().numpy(), c13[perm]), e
        assert np.array_equal(b13[i13[1]].cpu().numpy(), s13[perm]), e
        assert np.array_equal(b2[i2[0]].cpu().numpy(), c2), e
        assert np.array_equal(b2[i2[1]].cpu().numpy(), s2), e
        assert g13_all[e] == g13 and g2_all[e] == g2, e


def _sample_tokens(cfg, logits, bias, n=3):
    """The n-1 tokens whose experts hold the fewest rows, plus the last token
    (keeps the oracle's work small: it evaluates every row of those experts)."""
    ids, _ = M.route(logits.cpu().numpy(), None if bias is None else bias.cpu().numpy(), cfg.k, cfg.renormalize)
    pop = np.bincount(ids.reshape(-1), minlength=cfg.E)
    score = pop[ids].sum(1)
    return sorted(set(np.argsort(score, kind="stable")[:n - 1].tolist() + [cfg.T - 1]))


def test_tiny_layer(nvf):
    layer = Layer(nvf, CONFIGS["tiny"])
    check_layer(nvf, layer)
    check_layer(nvf, layer, torch.bfloat16)


@pytest.mark.parametrize("k,shared,T", [(1, False, 16), (8, False, 16), (8, True, 40), (2, True, 100)])
def test_routing_extremes(nvf, k, shared, T):
    """Top-1, top-E (every expert on every token), a shared expert beside
    top-E, and a batch between the small-group (<= 32 rows) and the
    large-batch (> 256 tokens) paths: the whole layer against the oracle."""
    cfg = CONFIGS["tiny"].scaled(k=k, shared=shared, T=T, name=f"tiny_k{k}_s{int(shared)}_t{T}")
    check_layer(nvf, Layer(nvf, cfg, parent="tiny"), torch.float32)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_layer(nvf, out_dtype):
    check_layer(nvf, Layer(nvf, CONFIGS["decode"]), out_dtype)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_prefill_layer_scaled(nvf, out_dtype):
    check_layer(nvf, Layer(nvf, CONFIGS["prefill"].scaled(T=512, name="prefill_T512"), parent="prefill"), out_dtype)


@pytest.mark.parametrize("parent,T", [("skewed", 384), ("large", 48)])
def test_scaled_layers_sampled(nvf, parent, T):
    cfg = CONFIGS[parent].scaled(T=T, name=f"{parent}_T{T}")
    layer = Layer(nvf, cfg, parent=parent, wdev="cuda")
    check_layer(nvf, layer, tokens=_sample_tokens(cfg, layer.logits, layer.bias))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefill", "large", "skewed"])
def test_full_size_sampled(nvf, name):
    """The bench's full-size layers: routing and permutation in full, everything
    else on sampled tokens (all rows of every expert they visit)."""
    cfg = CONFIGS[name]
    layer = Layer(nvf, cfg, wdev="cuda")
    check_layer(nvf, layer, tokens=_sample_tokens(cfg, layer.logits, layer.bias, n=2))


def test_stage_events_outside_a_graph(nvf):
    """Per-stage events given to a plain (not captured) forward are recorded and
    bracket the stages in order."""
    layer = Layer(nvf, CONFIGS["tiny"])
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record()      # torch creates the CUDA event on its first record
    torch.cuda.synchronize()
    cfg = layer.cfg
    out = nvf.moe_forward(layer.wts, layer.x, layer.logits, cfg.k, torch.tensor(layer.gs_a1, device="cuda"),
                          torch.tensor(layer.gs_a2, device="cuda"), stage_events=ev)
    torch.cuda.synchronize()
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(5)]
    assert all(t >= 0 for t in times) and sum(times) > 0
    ref = layer.run(h_dump=False)[0]
    assert torch.equal(out, ref)


def test_deterministic(nvf):
    layer = Layer(nvf, CONFIGS["tiny"].scaled(T=200, name="tiny_T200"), parent="tiny")
    a = layer.run()[0].cpu()
    b = layer.run()[0].cpu()
    assert torch.equal(a, b)


def test_empty_batch(nvf):
    cfg = CONFIGS["tiny"].scaled(T=0, name="tiny_T0")
    layer = Layer(nvf, cfg, parent="tiny")
    out = layer.run(h_dump=False)[0]
    assert out.shape == (0, cfg.H)
