"""nvfp4_prepare_weights through the C ABI, then nvfp4_moe_forward on what it made.

The weights are handed to the library as one FP32 (or BF16) stack and the
layer runs on the library's output with no Python arithmetic in between: the
prepared codes, scales and global scales must equal the oracle's quantization
of the same values bit for bit, preparing in expert chunks must give the same
bytes as one call, and the layer's output must be within 5e-3 * rms of the
oracle's forward pass.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import moe as M
from synth import CONFIGS, expert_weights, make_inputs
from tests.nvf_testutil import ensure_built, rel_err, w13_prepared_rows, weight_unpack

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module")
def nvf():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as m
    return m


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _stacks(cfg, dtype):
    w13 = torch.stack([expert_weights(cfg, e, 0)[0] for e in range(cfg.E_total)]).to(dtype)
    w2 = torch.stack([expert_weights(cfg, e, 0)[1] for e in range(cfg.E_total)]).to(dtype)
    return w13, w2


def _prepare(nvf, cfg, w13_src, w2_src, chunks):
    L = nvf.lib()
    Et, H, I = cfg.E_total, cfg.H, cfg.I
    w13 = torch.full((nvf.tiled_bytes(Et * 2 * I, 0, H),), 0xA5, dtype=torch.uint8, device="cuda")
    w2 = torch.full((nvf.tiled_bytes(Et * H, 0, I),), 0xA5, dtype=torch.uint8, device="cuda")
    gs13 = torch.full((Et,), -1.0, device="cuda")
    gs2 = torch.full((Et,), -1.0, device="cuda")
    code = nvf.NVF_F32 if w13_src.dtype == torch.float32 else nvf.NVF_BF16
    e0 = 0
    for n in chunks:
        a, b = w13_src[e0:e0 + n].cuda().contiguous(), w2_src[e0:e0 + n].cuda().contiguous()
        st = L.nvfp4_prepare_weights(_p(a), _p(b), code, e0, n, H, I, _p(w13), _p(gs13), _p(w2), _p(gs2), _stream())
        assert st == 0, L.nvf_last_error_message()
        e0 += n
    torch.cuda.synchronize()
    return w13, gs13, w2, gs2


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_prepared_weights_equal_the_oracle(nvf, dtype):
    cfg = CONFIGS["tiny"]
    w13_src, w2_src = _stacks(cfg, dtype)
    w13, gs13, w2, gs2 = _prepare(nvf, cfg, w13_src, w2_src, [cfg.E_total])
    perm = w13_prepared_rows(cfg.I)
    n13, n2 = nvf.tiled_bytes(2 * cfg.I, 0, cfg.H), nvf.tiled_bytes(cfg.H, 0, cfg.I)
    for e in range(cfg.E_total):
        c13, s13, g13 = M.quantize_expert_weights(w13_src[e].float().numpy())
        c2, s2, g2 = M.quantize_expert_weights(w2_src[e].float().numpy())
        gc, gsc = weight_unpack(w13[e * n13:(e + 1) * n13].cpu().numpy(), cfg.H, 2 * cfg.I, 2 * cfg.I)
        assert np.array_equal(gc, c13[perm]) and np.array_equal(gsc, s13[perm])
        gc, gsc = weight_unpack(w2[e * n2:(e + 1) * n2].cpu().numpy(), cfg.I, cfg.H, cfg.H)
        assert np.array_equal(gc, c2) and np.array_equal(gsc, s2)
        assert gs13[e].item() == g13 and gs2[e].item() == g2


def test_chunked_preparation_equals_one_call(nvf):
    cfg = CONFIGS["tiny"]
    w13_src, w2_src = _stacks(cfg, torch.float32)
    one = _prepare(nvf, cfg, w13_src, w2_src, [cfg.E_total])
    parts = _prepare(nvf, cfg, w13_src, w2_src, [3, 1, cfg.E_total - 4])
    for a, b in zip(one, parts):
        assert torch.equal(a, b)


def test_zero_expert_gets_unit_scale(nvf):
    cfg = CONFIGS["tiny"]
    w13_src, w2_src = _stacks(cfg, torch.float32)
    w13_src[2].zero_()
    w13, gs13, w2, gs2 = _prepare(nvf, cfg, w13_src, w2_src, [cfg.E_total])
    assert gs13[2].item() == 1.0
    n13 = nvf.tiled_bytes(2 * cfg.I, 0, cfg.H)
    gc, gsc = weight_unpack(w13[2 * n13:3 * n13].cpu().numpy(), cfg.H, 2 * cfg.I, 2 * cfg.I)
    assert not gc.any() and not gsc.any()


def test_prepare_then_forward_through_the_c_abi(nvf):
    """Prepare, workspace layout and forward as a C caller would make them."""
    cfg = CONFIGS["tiny"]
    L = nvf.lib()
    w13_src, w2_src = _stacks(cfg, torch.float32)
    w13, gs13, w2, gs2 = _prepare(nvf, cfg, w13_src, w2_src, [cfg.E_total])
    x, logits, _ = make_inputs(cfg, 0)
    x, logits = x.cuda(), logits.cuda()
    gs_a1 = np.full(cfg.E_total, 0.0012672061566263437, np.float32)
    gs_a2 = np.full(cfg.E_total, 0.00016923830844461918, np.float32)
    d_gs_a1, d_gs_a2 = torch.from_numpy(gs_a1).cuda(), torch.from_numpy(gs_a2).cuda()
    cw = nvf.MoEWeightsC(cfg.E, cfg.H, cfg.I, 0, w13.data_ptr(), gs13.data_ptr(), w2.data_ptr(), gs2.data_ptr())
    lay = nvf.WorkspaceLayoutC()
    assert L.nvfp4_moe_workspace_layout(cfg.T, cfg.E, cfg.H, cfg.I, cfg.k, 0, ctypes.byref(lay)) == 0
    ws = torch.empty(lay.total, dtype=torch.uint8, device="cuda")
    out = torch.empty(cfg.T, cfg.H, device="cuda")
    st = L.nvfp4_moe_forward(ctypes.byref(cw), _p(x), _p(logits), None, cfg.T, cfg.k, 1, _p(d_gs_a1), _p(d_gs_a2),
                             nvf.NVF_F32, _p(out), None, _p(ws), lay.total, None, _stream())
    assert st == 0, L.nvf_last_error_message()
    code, detail = nvf.device_status()
    assert code == 0, (code, detail)
    q = {e: (*M.quantize_expert_weights(w13_src[e].numpy()), *M.quantize_expert_weights(w2_src[e].numpy()))
         for e in range(cfg.E_total)}
    ref = M.moe_forward(x.float().cpu().numpy(), logits.cpu().numpy(), None, cfg.k, True, False, lambda e: q[e],
                        gs_a1, gs_a2)
    assert rel_err(out.cpu().numpy(), ref["out"]) <= TOL


def test_argument_validation(nvf):
    L = nvf.lib()
    z = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    f = torch.zeros(64, device="cuda")
    args = lambda H, I, dt=0, n=1: (_p(z), _p(z), dt, 0, n, H, I, _p(z), _p(f), _p(z), _p(f), _stream())
    assert L.nvfp4_prepare_weights(*args(200, 128)) == 1     # H not a multiple of 128
    assert L.nvfp4_prepare_weights(*args(256, 96)) == 1      # I not a multiple of 64
    assert L.nvfp4_prepare_weights(*args(256, 128, dt=7)) == 1
    assert L.nvfp4_prepare_weights(*args(256, 128, n=0)) == 1
    assert b"n_experts" in L.nvf_last_error_message()
