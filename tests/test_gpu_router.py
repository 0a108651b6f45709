"""GPU parity of the router gate (nvf_router_gemm) and of the layer run from
the hidden states (nvfp4_moe_forward_gated) against the oracle.

Logits: each is a sum of H exact products of bf16 values accumulated in FP32
on the tensor cores.  Any accumulation order of n terms is within
(n - 1) * u * sum|x_h w_h| of the exact sum (u = 2^-23 covers a truncating FP32
accumulator as well as a rounding one), which is the per-element bound used
here.  Routing and everything after it are checked on the GPU's own logits
(the selection is an argmax: both sides decide it in the same precision).
"""
import numpy as np
import pytest
import torch

from oracle import moe as M
from synth import CONFIGS, expert_weights, gate_weights, make_inputs
from tests.nvf_testutil import ensure_built, rel_err

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module")
def nvf():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as m
    return m


def _check_logits(got, xb, wb):
    x = xb.float().numpy().astype(np.float64)
    w = wb.float().numpy().astype(np.float64)
    ref = M.router_logits(x, w)
    bound = (x.shape[1] - 1) * 2.0 ** -23 * (np.abs(x) @ np.abs(w).T)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= bound), (err.max(), bound.min())
    return ref


# Above 64 tokens the K split is the largest power of two S <= 8 with
# ceil(T / 128) * ceil(n / 256) * S <= SMs (152) that divides H / 64: 65 and
# 128 tokens run S = 4 (H = 256), 300 tokens S = 8, 4096 tokens S = 4, 6000
# tokens S = 2, 10000 tokens S = 1 (a cluster of one); 513 gate rows take
# three 256-row blocks, the last with 16.
@pytest.mark.parametrize("T,H,n", [(1, 256, 8), (37, 2048, 129), (64, 128, 9), (65, 256, 33), (128, 256, 33),
                                   (300, 2048, 128), (4096, 2048, 129), (256, 4096, 513), (6000, 512, 40),
                                   (10000, 256, 33), (100, 256, 1)])
def test_router_gemm_matches_the_oracle(nvf, T, H, n):
    g = torch.Generator().manual_seed(T + H + n)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    w = (torch.randn(n, H, generator=g) * 0.02).to(torch.bfloat16)
    got = nvf.router_gemm(x.cuda(), w.cuda())
    code, detail = nvf.device_status()
    assert code == 0, (code, detail)
    _check_logits(got.cpu().numpy(), x, w)


def test_router_gemm_row_stride_and_exact_case(nvf):
    """Small integers are exact in bf16 and their sums exact in FP32: the GPU
    must give exactly the integer dot products, written with a row stride."""
    T, H, n = 130, 128, 40
    g = torch.Generator().manual_seed(7)
    x = torch.randint(-3, 4, (T, H), generator=g).to(torch.bfloat16)
    w = torch.randint(-3, 4, (n, H), generator=g).to(torch.bfloat16)
    out = torch.full((T, 48), 12345.0, device="cuda")
    nvf.router_gemm(x.cuda(), w.cuda(), logits=out[:, :].as_strided((T, n), (48, 1)))
    o = out.cpu().numpy()
    assert np.array_equal(o[:, :n], (x.float() @ w.float().T).numpy())
    assert np.all(o[:, n:] == 12345.0)          # columns past n untouched


def _layer(cfg):
    x, _, _ = make_inputs(cfg, 0)
    return x


@pytest.mark.parametrize("gated,T", [(False, 40), (True, 40), (True, 300)])
def test_layer_from_hidden_states(nvf, gated, T):
    """Router gate + layer, with and without the shared expert's gate, against
    the oracle on the GPU's logits; routing bit-exact.  40 tokens take the
    CUDA-core gate, 300 the tensor-core one (K split over a cluster)."""
    cfg = CONFIGS["tiny"].scaled(T=T, shared=True, name="tiny_shared")
    x = _layer(cfg)
    wg = gate_weights(cfg, 0, shared_gate=gated)
    w = nvf.prepare_weights(cfg.E, cfg.H, cfg.I, True, lambda e: expert_weights(cfg, e, 0))
    gs_a1 = np.full(cfg.E_total, 0.0012672061566263437, np.float32)
    gs_a2 = np.full(cfg.E_total, 0.00016923830844461918, np.float32)
    ws = nvf.workspace(cfg.T, w, cfg.k)
    out = nvf.moe_forward_gated(w, x.cuda(), wg.cuda(), cfg.k, torch.from_numpy(gs_a1).cuda(),
                                torch.from_numpy(gs_a2).cuda(), shared_gate=gated, ws=ws)
    code, detail = nvf.device_status()
    assert code == 0, (code, detail)
    L = nvf.workspace_layout(cfg.T, cfg.E, cfg.H, cfg.I, cfg.k, True)
    ncol = cfg.E + int(gated)
    lg = ws[L["logits"]:L["logits"] + 4 * cfg.T * ncol].view(torch.float32).cpu().numpy().reshape(cfg.T, ncol)
    _check_logits(lg, x, wg)
    ids = ws[L["topk_ids"]:L["topk_ids"] + 4 * cfg.T * cfg.k].view(torch.int32).cpu().numpy().reshape(cfg.T, cfg.k)
    ref_ids, _ = M.route(lg[:, :cfg.E], None, cfg.k, True)
    assert np.array_equal(ids, ref_ids)
    q = {e: (*M.quantize_expert_weights(a.numpy()), *M.quantize_expert_weights(b.numpy()))
         for e in range(cfg.E_total) for a, b in [expert_weights(cfg, e, 0)]}
    ref = M.moe_forward(x.float().numpy(), lg[:, :cfg.E], None, cfg.k, True, True, lambda e: q[e], gs_a1, gs_a2,
                        shared_gate_logit=lg[:, cfg.E] if gated else None)
    assert rel_err(out.cpu().numpy(), ref["out"]) <= TOL
    if not gated:
        # the plain forward on the same logits gives the same bits
        plain = nvf.moe_forward(w, x.cuda(), torch.from_numpy(np.ascontiguousarray(lg)).cuda(), cfg.k,
                                torch.from_numpy(gs_a1).cuda(), torch.from_numpy(gs_a2).cuda())
        assert torch.equal(plain, out)


def test_argument_validation(nvf):
    x = torch.zeros(4, 100, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(8, 100, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nvf.NvfError, match="H=100"):
        nvf.router_gemm(x, w)
    cfg = CONFIGS["tiny"]
    wts = nvf.prepare_weights(cfg.E, cfg.H, cfg.I, False, lambda e: expert_weights(cfg, e, 0))
    xx = torch.zeros(4, cfg.H, dtype=torch.bfloat16, device="cuda")
    wg = torch.zeros(cfg.E + 1, cfg.H, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(cfg.E, device="cuda")
    with pytest.raises(nvf.NvfError, match="shared_gate"):
        nvf.moe_forward_gated(wts, xx, wg, cfg.k, g, g, shared_gate=True)
