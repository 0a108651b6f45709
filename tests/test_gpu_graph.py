"""The layer step captured as a CUDA graph (nvf_moe_graph_*): copies in, the
layer, copy out, replayed by one launch.  Its result must equal the separate
calls' (nvfp4_moe_forward on the same inputs) bit for bit -- the graph runs the
same kernels -- and a launch must see new host inputs."""
import ctypes

import numpy as np
import pytest
import torch

from synth import CONFIGS, expert_weights, make_inputs
from tests.nvf_testutil import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvf():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as m
    return m


@pytest.mark.parametrize("shared,out_dtype,with_bias,T", [(False, torch.bfloat16, False, 24),
                                                          (True, torch.float32, False, 24),
                                                          (False, torch.bfloat16, True, 24),
                                                          (True, torch.bfloat16, False, 300)])
def test_graph_step_equals_the_separate_calls(nvf, shared, out_dtype, with_bias, T):
    cfg = CONFIGS["tiny"].scaled(T=T, shared=shared, name="tiny_graph")
    w = nvf.prepare_weights(cfg.E, cfg.H, cfg.I, shared, lambda e: expert_weights(cfg, e, 0))
    gs_a1 = torch.full((cfg.E_total,), 0.0012672061566263437, device="cuda")
    gs_a2 = torch.full((cfg.E_total,), 0.00016923830844461918, device="cuda")
    # a selection bias that changes which experts win
    bias = torch.linspace(-1.0, 1.0, cfg.E, device="cuda") if with_bias else None
    g = nvf.MoEGraph(w, cfg.T, cfg.k, gs_a1, gs_a2, bias=bias, out_dtype=out_dtype)
    for seed in (0, 1):                      # the second launch sees new host inputs
        x, lg, _ = make_inputs(cfg, seed)
        g.x.copy_(x)
        g.logits.copy_(lg)
        g.launch()
        torch.cuda.synchronize()
        code, detail = nvf.device_status()
        assert code == 0, (code, detail)
        ref = nvf.moe_forward(w, x.cuda(), lg.cuda(), cfg.k, gs_a1, gs_a2, bias=bias, out_dtype=out_dtype)
        assert torch.equal(g.out, ref.cpu()), seed
    g.close()


def test_pageable_host_memory_is_rejected(nvf):
    cfg = CONFIGS["tiny"]
    w = nvf.prepare_weights(cfg.E, cfg.H, cfg.I, False, lambda e: expert_weights(cfg, e, 0))
    gs = torch.ones(cfg.E, device="cuda")
    x = np.zeros((cfg.T, cfg.H), np.uint16)
    lg = np.zeros((cfg.T, cfg.E), np.float32)
    out = np.zeros((cfg.T, cfg.H), np.uint16)
    cw = w.c_struct()
    h = ctypes.c_void_p()
    st = nvf.lib().nvf_moe_graph_create(ctypes.byref(cw), cfg.T, cfg.k, 1, gs.data_ptr(), gs.data_ptr(), None,
                                        x.ctypes.data, lg.ctypes.data, out.ctypes.data, nvf.NVF_BF16,
                                        ctypes.byref(h))
    assert st == 1 and b"page-locked" in nvf.lib().nvf_last_error_message()
    assert h.value is None


def test_separate_input_buffers(nvf):
    """x and logits in separate page-locked buffers (two copies a step)."""
    cfg = CONFIGS["tiny"].scaled(T=20, name="tiny_graph2")
    w = nvf.prepare_weights(cfg.E, cfg.H, cfg.I, False, lambda e: expert_weights(cfg, e, 0))
    gs = torch.full((cfg.E,), 0.0012672061566263437, device="cuda")
    gs2 = torch.full((cfg.E,), 0.00016923830844461918, device="cuda")
    x, lg, _ = make_inputs(cfg, 3)
    xh, lh = x.clone().pin_memory(), lg.clone().pin_memory()
    oh = torch.zeros(cfg.T, cfg.H, dtype=torch.bfloat16).pin_memory()
    cw = w.c_struct()
    h = ctypes.c_void_p()
    st = nvf.lib().nvf_moe_graph_create(ctypes.byref(cw), cfg.T, cfg.k, 1, gs.data_ptr(), gs2.data_ptr(), None,
                                        xh.data_ptr(), lh.data_ptr(), oh.data_ptr(), nvf.NVF_BF16, ctypes.byref(h))
    assert st == 0, nvf.lib().nvf_last_error_message()
    assert nvf.lib().nvf_moe_graph_launch(h, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    torch.cuda.synchronize()
    ref = nvf.moe_forward(w, x.cuda(), lg.cuda(), cfg.k, gs, gs2, out_dtype=torch.bfloat16)
    assert torch.equal(oh, ref.cpu())
    assert nvf.lib().nvf_moe_graph_destroy(h) == 0
