"""Pins of the oracle's expert-parallel plan and forward (CPU).

The plan is checked against brute-force counts, against the bijectivity and
segment order of its send positions, and by sending each assignment's index
through dispatch, grouping and return; the receive order against a direct
construction; the G-rank forward against the single-device forward of every
rank's tokens (expert parallelism moves rows, it does not change a row's
arithmetic)."""
import numpy as np
import pytest

from oracle import ep as EP
from oracle import moe as M
from synth import CONFIGS, expert_weights, make_inputs


def _ids(rng, T, k, E):
    if T == 0:
        return np.zeros((0, k), np.int64)
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])


@pytest.mark.parametrize("shared", [False, True])
@pytest.mark.parametrize("G,rank", [(1, 0), (2, 1), (4, 2), (8, 7)])
def test_counts_brute_force(shared, G, rank):
    rng = np.random.default_rng(G * 10 + rank)
    T, k, E = 37, 4, 16
    ids = _ids(rng, T, k, E)
    segs, counts, s2s = EP.dispatch_plan(ids, E, G, rank, shared)
    El = E // G
    for r in range(G):
        for j in range(El):
            assert counts[r, j] == int(np.sum(ids == r * El + j))
        assert counts[r, El] == (T if shared and r == rank else 0)
        assert len(segs[r]) == counts[r].sum()


@pytest.mark.parametrize("shared", [False, True])
def test_send_positions_bijective_and_ordered(shared):
    rng = np.random.default_rng(3)
    T, k, E, G, rank = 29, 3, 12, 3, 1
    ids = _ids(rng, T, k, E)
    segs, counts, s2s = EP.dispatch_plan(ids, E, G, rank, shared)
    R = T * k + (T if shared else 0)
    assert sorted(s2s.tolist()) == list(range(R))
    bounds = np.concatenate([[0], np.cumsum(counts.sum(axis=1))])
    El = E // G
    for r in range(G):
        seg = segs[r]
        assert [s2s[a] for a, _ in seg] == list(range(bounds[r], bounds[r + 1]))
        routed = [(e, a) for a, e in seg if e < E]
        assert routed == sorted(routed)                      # by expert, then assignment
        assert all(r * El <= e < (r + 1) * El for e, _ in routed)
        tail = [a for a, e in seg if e == E]
        assert tail == (list(range(T * k, T * k + T)) if shared and r == rank else [])
        assert seg[len(routed):] == [(a, E) for a in tail]  # shared rows close the segment


def test_receive_order_direct():
    counts_in = np.array([[2, 0, 1], [1, 3, 0], [0, 1, 2]])
    off, r2g = EP.receive_order(counts_in)
    assert off.tolist() == [0, 3, 7, 10]
    # arrivals: src0: j0 j0 j2 | src1: j0 j1 j1 j1 | src2: j1 j2 j2
    assert r2g.tolist() == [0, 1, 7, 2, 3, 4, 5, 6, 8, 9]


@pytest.mark.parametrize("shared", [False, True])
def test_payload_round_trip(shared):
    """Each assignment's index, sent through the plan, grouped, and returned,
    lands back at its own send position."""
    rng = np.random.default_rng(11)
    G, E, k = 4, 16, 3
    Ts = [5, 0, 13, 8]
    ids = [_ids(rng, T, k, E) for T in Ts]
    plans = [EP.dispatch_plan(ids[s], E, G, s, shared) for s in range(G)]
    back = [np.full(len(p[2]), -1) for p in plans]
    for r in range(G):
        counts_in = np.stack([plans[s][1][r] for s in range(G)])
        off, r2g = EP.receive_order(counts_in)
        payload = [(s, a) for s in range(G) for a, _ in plans[s][0][r]]
        grouped = [None] * len(payload)
        for i, item in enumerate(payload):
            grouped[r2g[i]] = item
        # grouped rows of local expert j all carry expert j
        for j in range(len(off) - 1):
            for s, a in grouped[off[j]:off[j + 1]]:
                e = dict(plans[s][0][r])[a]
                assert (e - r * (E // G) if e < E else E // G) == j
        for i, (s, a) in enumerate(payload):
            back[s][plans[s][2][a]] = a
    for s in range(G):
        inv = np.empty_like(plans[s][2])
        inv[plans[s][2]] = np.arange(len(inv))
        assert back[s].tolist() == inv.tolist()


def _layer_weights(cfg):
    q = {}

    def weights(e):
        if e not in q:
            a, b = expert_weights(cfg, e, 0)
            q[e] = (*M.quantize_expert_weights(a.numpy()), *M.quantize_expert_weights(b.numpy()))
        return q[e]
    return weights


@pytest.mark.parametrize("G,shared", [(2, False), (4, True)])
def test_forward_equals_single_device(G, shared):
    cfg = CONFIGS["tiny"].scaled(E=8, k=2, shared=shared, name="tiny_ep")
    weights = _layer_weights(cfg)
    Et = cfg.E + int(shared)
    gs_a1 = np.full(Et, 0.0012672061566263437, np.float32)
    gs_a2 = np.full(Et, 0.00016923830844461918, np.float32)
    xs, lgs = [], []
    for r, T in enumerate([9, 16, 1, 4][:G]):
        x, lg, _ = make_inputs(cfg.scaled(T=T), seed=100 + r)
        xs.append(x.float().numpy())
        lgs.append(lg.numpy())
    outs, recv = EP.ep_forward(xs, lgs, cfg.k, cfg.E, G, shared, True, weights, gs_a1, gs_a2)
    for r in range(G):
        ref = M.moe_forward(xs[r], lgs[r], None, cfg.k, True, shared, weights, gs_a1, gs_a2)
        assert np.array_equal(outs[r]["out"], ref["out"])
        # the returned rows are the single-device y rows, moved to their send positions
        assert np.array_equal(outs[r]["y_back"][outs[r]["src_to_send"]], ref["y"][ref["src_to_perm"]])
