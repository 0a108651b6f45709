"""Pins of the oracle's router gate and shared-expert gate (CPU).

router_logits is checked against an exact integer case, a brute-force
per-element sum with math.fsum, and the float32 rounding of the exact sum;
shared_gate against the sigmoid's closed-form values; the gated combine
reduces to the plain one when the gate is fully open and drops the shared
row when it is closed."""
import math

import numpy as np
import torch

from oracle import moe as M
from synth import CONFIGS, gate_weights, make_inputs


def test_exact_integer_case():
    # small integers are exact in bf16 and their dot products exact in float32
    x = np.array([[1, 2, 3, 4], [0, -1, 5, 2]], np.float32)
    w = np.array([[1, 0, -1, 2], [3, 3, 3, 3], [0, 0, 0, 1]], np.float32)
    expect = np.array([[6, 30, 4], [-1, 18, 2]], np.float32)
    assert np.array_equal(M.router_logits(x, w), expect)


def test_brute_force_against_fsum():
    cfg = CONFIGS["tiny"]
    x, _, _ = make_inputs(cfg, 0)
    w = gate_weights(cfg, 0, shared_gate=True)
    xf, wf = x.float().numpy(), w.float().numpy()
    got = M.router_logits(xf, wf)
    assert got.shape == (cfg.T, cfg.E + 1) and got.dtype == np.float32
    for t in range(cfg.T):
        for j in range(cfg.E + 1):
            exact = math.fsum(float(a) * float(b) for a, b in zip(xf[t], wf[j]))
            assert got[t, j] == np.float32(exact)          # one rounding of the exact sum


def test_gate_scale_matches_the_recipe():
    cfg = CONFIGS["decode"]
    x, _, _ = make_inputs(cfg, 0)
    lg = M.router_logits(x.float().numpy(), gate_weights(cfg, 0).float().numpy())
    assert 0.5 < lg.std() < 1.5        # like the N(0, 1) logits of the workload recipe


def test_shared_gate_closed_forms():
    assert M.shared_gate(0.0) == 0.5
    assert abs(M.shared_gate(math.log(3.0)) - 0.75) < 1e-15
    assert M.shared_gate(-1000.0) == 0.0 and M.shared_gate(1000.0) == 1.0


def test_gated_combine_reduces_to_the_plain_one():
    rng = np.random.default_rng(0)
    T, k, E, H = 6, 2, 4, 8
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    _, _, _, s2p = M.permute(ids, E, shared=True)
    y = rng.standard_normal((T * k + T, H))
    w = rng.random((T, k))
    plain = M.combine(y, w, s2p, T, k, True)
    assert np.allclose(M.combine(y, w, s2p, T, k, True, np.ones(T)), plain, rtol=0, atol=0)
    no_shared = M.combine(y, w, s2p, T, k, False)
    assert np.array_equal(M.combine(y, w, s2p, T, k, True, np.zeros(T)), no_shared)
    half = M.combine(y, w, s2p, T, k, True, np.full(T, 0.5))
    assert np.allclose(half, (plain + no_shared) / 2, rtol=1e-15, atol=1e-15)
