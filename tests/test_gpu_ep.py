"""GPU parity of the expert-parallel steps (dispatch, receive, local experts,
return, combine), with G ranks emulated on one GPU: the exchanges are tensor
slices (each receiver takes its segment of every sender's buffer), the kernels
are the library's.

Integer and byte results are compared with the oracle's plan bit for bit
(send positions, per-expert counts, the quantized send rows, the grouped
order and offsets, the grouped A1 operand).  Every rank's output must equal
the single-device forward of its own tokens bit for bit: expert parallelism
moves rows, and a row's arithmetic (quantization, both GEMMs, the combine in
slot order) does not depend on the rows around it.  The single-device forward
is itself checked against the oracle in test_gpu_forward.py.
"""
import numpy as np
import pytest
import torch

from oracle import ep as EP
from oracle import formats as F
from oracle import moe as M
from synth import CONFIGS, expert_weights, make_inputs
from tests.nvf_testutil import ensure_built, row_tiles, tiled_unpack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvf():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as m
    return m


def _scales(Et):
    # distinct per-expert activation scales, so that a scale taken from the wrong expert shows
    gs_a1 = (0.0012672061566263437 * (1.0 + 0.03 * np.arange(Et))).astype(np.float32)
    gs_a2 = (0.00016923830844461918 * (1.0 + 0.02 * np.arange(Et))).astype(np.float32)
    return gs_a1, gs_a2


class EmulatedRanks:
    """G ranks on one GPU: tokens, routing and dispatch per rank."""

    def __init__(self, nvf, cfg, G, Ts, seed=0):
        self.nvf, self.cfg, self.G = nvf, cfg, G
        self.El = cfg.E // G
        Et = cfg.E_total
        gs_a1, gs_a2 = _scales(Et)
        self.gs_a1_np, self.gs_a2_np = gs_a1, gs_a2
        self.gs_a1, self.gs_a2 = torch.from_numpy(gs_a1).cuda(), torch.from_numpy(gs_a2).cuda()
        self.xs, self.logits, self.routes, self.sends = [], [], [], []
        for r, T in enumerate(Ts):
            x, lg, _ = make_inputs(cfg.scaled(T=T), seed=seed + 17 * r)
            x, lg = x.cuda(), lg.cuda()
            route = nvf.route_permute(lg, cfg.k, shared=cfg.shared)
            self.xs.append(x)
            self.logits.append(lg)
            self.routes.append(route)
            self.sends.append(nvf.ep_dispatch(x, route, cfg.E, cfg.k, cfg.shared, G, r, self.gs_a1))

    def exchange(self, r):
        """Receiver r: the rows every source sent it, sources back to back, and its counts."""
        rows, counts = [], []
        for s in range(self.G):
            send, cnt, _ = self.sends[s]
            b = np.concatenate([[0], np.cumsum(cnt.sum(dim=1).cpu().numpy())])
            rows.append(send[b[r]:b[r + 1]])
            counts.append(cnt[r])
        return torch.cat(rows), torch.stack(counts).contiguous()

    def run(self, w_locals, out_dtype=torch.float32, fused=False):
        """fused: the down GEMM stores y rows in received order (row map);
        else y in grouped order and the return kernel reorders it."""
        nvf, cfg, G = self.nvf, self.cfg, self.G
        y_ret, recv_counts, grouped = [], [], []
        for r in range(G):
            recv, rc = self.exchange(r)
            n = int(rc.sum().item())
            g = nvf.ep_receive(recv, rc, self.El, cfg.shared, cfg.H, n)
            y = nvf.moe_experts(w_locals[r], g["a1"], n, g["offsets"], g["tile_offsets"],
                                nvf.ep_local_scales(self.gs_a1, cfg.E, G, r, cfg.shared),
                                nvf.ep_local_scales(self.gs_a2, cfg.E, G, r, cfg.shared), out_dtype,
                                y_rows=g["grp_to_recv"] if fused else None)
            y_ret.append(y if fused else nvf.ep_return(y, g["recv_to_grp"]))
            recv_counts.append(rc)
            grouped.append(g)
        outs = []
        for s in range(G):
            back = []
            for r in range(G):
                b = np.concatenate([[0], np.cumsum(recv_counts[r].sum(dim=1).cpu().numpy())])
                back.append(y_ret[r][b[s]:b[s + 1]])
            y_back = torch.cat(back)
            T = self.xs[s].shape[0]
            outs.append(nvf.moe_combine(y_back, self.routes[s]["topk_w"], self.sends[s][2], T, cfg.k, cfg.shared))
        return outs, grouped


def _weights(nvf, cfg, experts):
    """Prepared weights of the given global experts (the shared one, id E, last)."""
    routed = [e for e in experts if e < cfg.E]
    return nvf.prepare_weights(len(routed), cfg.H, cfg.I, cfg.shared, lambda j: expert_weights(cfg, experts[j], 0))


@pytest.mark.parametrize("G,shared,Ts", [(2, False, [40, 7]), (4, True, [12, 0, 300, 5]), (8, False, [33] * 8)])
def test_layer_matches_single_device(nvf, G, shared, Ts):
    cfg = CONFIGS["tiny"].scaled(E=16, k=4, shared=shared, name="tiny_ep")
    ranks = EmulatedRanks(nvf, cfg, G, Ts)
    El = cfg.E // G
    tail = [cfg.E] if shared else []
    w_locals = [_weights(nvf, cfg, list(range(r * El, (r + 1) * El)) + tail) for r in range(G)]
    outs, _ = ranks.run(w_locals)
    fused, _ = ranks.run(w_locals, fused=True)
    code, detail = nvf.device_status()
    assert code == 0, (code, detail)
    for r in range(G):
        assert torch.equal(outs[r], fused[r])
    w_full = _weights(nvf, cfg, list(range(cfg.E)) + tail)
    for r in range(G):
        if Ts[r] == 0:
            assert outs[r].shape[0] == 0
            continue
        ref = nvf.moe_forward(w_full, ranks.xs[r], ranks.logits[r], cfg.k, ranks.gs_a1, ranks.gs_a2)
        assert torch.equal(outs[r], ref), f"rank {r}: max diff {(outs[r] - ref).abs().max().item()}"


# Above 256 tokens a rank's dispatch runs token by token (a place pass, then a
# quantize-and-store pass): 300 and 260 tokens take that path.  Up to 4096
# received rows the receive plans inside the scatter kernel; the two ranks of
# 1200 + 1100 tokens receive ~4600 rows each, past that.
@pytest.mark.parametrize("shared,Ts", [(False, [9, 70, 0, 31]), (True, [9, 70, 0, 31]), (True, [300, 5, 260, 0]),
                                       (False, [300, 5, 260, 0]), (True, [1200, 1100])])
def test_dispatch_and_receive_match_the_oracle(nvf, shared, Ts):
    cfg = CONFIGS["tiny"].scaled(E=16, k=4, shared=shared, name="tiny_ep")
    G = len(Ts)
    ranks = EmulatedRanks(nvf, cfg, G, Ts, seed=5)
    El, H = cfg.E // G, cfg.H
    plans = []
    for r in range(G):
        ids = ranks.routes[r]["topk_ids"].cpu().numpy()
        segs, counts, s2s = EP.dispatch_plan(ids, cfg.E, G, r, shared)
        plans.append((segs, counts))
        send, cnt, g_s2s = ranks.sends[r]
        assert np.array_equal(cnt.cpu().numpy(), counts)
        assert np.array_equal(g_s2s.cpu().numpy(), s2s)
        # every send row is the oracle's NVFP4 of its token with its expert's scale
        rows = send.cpu().numpy()
        x = ranks.xs[r].float().cpu().numpy()
        T = Ts[r]
        order = [(a, e) for d in range(G) for a, e in segs[d]]
        for pos, (a, e) in enumerate(order):
            t = int(M.assignment_token(np.array([a]), T, cfg.k)[0])
            qc, qs = F.quantize_rows(x[t:t + 1], ranks.gs_a1_np[e])
            assert np.array_equal(rows[pos, :H // 2], qc[0]), (r, pos)
            assert np.array_equal(rows[pos, H // 2:H // 2 + H // 16], qs[0]), (r, pos)
    for r in range(G):
        recv, rc = ranks.exchange(r)
        n = int(rc.sum().item())
        g = nvf.ep_receive(recv, rc, El, shared, H, n)
        off, r2g = EP.receive_order(np.stack([plans[s][1][r] for s in range(G)]))
        assert np.array_equal(g["offsets"].cpu().numpy(), off[:El + int(shared) + 1])
        assert np.array_equal(g["recv_to_grp"].cpu().numpy(), r2g)
        assert np.array_equal(g["grp_to_recv"].cpu().numpy()[r2g], np.arange(n))
        assert np.array_equal(g["tile_offsets"].cpu().numpy(), M.tile_offsets(np.diff(off[:El + int(shared) + 1])))
        # the grouped operand holds each received row at its grouped position
        tile, rr = row_tiles(n, off[:El + int(shared) + 1], g["tile_offsets"].cpu().numpy())
        codes, scales = tiled_unpack(g["a1"].cpu().numpy(), H, tile, rr)
        rows = recv.cpu().numpy()
        assert np.array_equal(codes[r2g], rows[:, :H // 2])
        assert np.array_equal(scales[r2g], rows[:, H // 2:H // 2 + H // 16])


def test_combine_entry_point(nvf):
    """nvf_moe_combine on the single-device y reproduces the forward's output."""
    cfg = CONFIGS["tiny"].scaled(T=40, shared=True, name="tiny_shared")
    x, lg, _ = make_inputs(cfg, 0)
    w = nvf.prepare_weights(cfg.E, cfg.H, cfg.I, True, lambda e: expert_weights(cfg, e, 0))
    gs_a1, gs_a2 = (torch.from_numpy(v).cuda() for v in _scales(cfg.E_total))
    ws = nvf.workspace(cfg.T, w, cfg.k)
    out = nvf.moe_forward(w, x.cuda(), lg.cuda(), cfg.k, gs_a1, gs_a2, ws=ws)
    L = nvf.workspace_layout(cfg.T, cfg.E, cfg.H, cfg.I, cfg.k, True)
    R = L["R"]
    y = ws[L["y"]:L["y"] + 4 * R * cfg.H].view(torch.float32).view(R, cfg.H)
    tw = ws[L["topk_w"]:L["topk_w"] + 4 * cfg.T * cfg.k].view(torch.float32).view(cfg.T, cfg.k)
    s2p = ws[L["src_to_perm"]:L["src_to_perm"] + 4 * R].view(torch.int32)
    got = nvf.moe_combine(y, tw, s2p, cfg.T, cfg.k, True)
    assert torch.equal(got, out)


def test_argument_validation(nvf):
    cfg = CONFIGS["tiny"].scaled(E=16, k=4, name="tiny_ep")
    x, lg, _ = make_inputs(cfg, 0)
    route = nvf.route_permute(lg.cuda(), cfg.k)
    g = torch.ones(cfg.E, device="cuda")
    with pytest.raises(nvf.NvfError, match="divide"):
        nvf.ep_dispatch(x.cuda(), route, cfg.E, cfg.k, False, 3, 0, g)
    with pytest.raises(nvf.NvfError, match="rank"):
        nvf.ep_dispatch(x.cuda(), route, cfg.E, cfg.k, False, 4, 4, g)


@pytest.mark.parametrize("G,El,shared", [(2, 2100, True), (3, 40, False)])
def test_receive_many_cells(nvf, G, El, shared):
    """A receive over many (source, expert) cells, most of them empty: past 4096
    cells the plan comes from its own kernel (2 x 2101 cells), else from the
    scatter kernel.  Rows are arbitrary bytes: the receive only moves them."""
    H = 256
    rng = np.random.default_rng(G * 1000 + El)
    J = El + 1
    counts = np.zeros((G, J), np.int32)
    nz = rng.choice(G * J, size=min(60, G * J), replace=False)
    counts.reshape(-1)[nz] = rng.integers(1, 4, size=nz.size)
    if not shared:
        counts[:, El] = 0
    n = int(counts.sum())
    row_bytes = nvf.ep_row_bytes(H)
    rows = rng.integers(0, 256, size=(n, row_bytes), dtype=np.uint8)
    g = nvf.ep_receive(torch.from_numpy(rows).cuda(), torch.from_numpy(counts).cuda(), El, shared, H, n)
    code, detail = nvf.device_status()
    assert code == 0, (code, detail)
    off, r2g = EP.receive_order(counts)
    Et = El + int(shared)
    assert np.array_equal(g["offsets"].cpu().numpy(), off[:Et + 1])
    assert np.array_equal(g["recv_to_grp"].cpu().numpy(), r2g)
    assert np.array_equal(g["tile_offsets"].cpu().numpy(), M.tile_offsets(np.diff(off[:Et + 1])))
    tile, rr = row_tiles(n, off[:Et + 1], g["tile_offsets"].cpu().numpy())
    codes, scales = tiled_unpack(g["a1"].cpu().numpy(), H, tile, rr)
    assert np.array_equal(codes[r2g], rows[:, :H // 2])
    assert np.array_equal(scales[r2g], rows[:, H // 2:H // 2 + H // 16])
