"""GPU parity of routing and permutation against the oracle (ids, offsets, permutation bit-exact)."""
import numpy as np
import pytest
import torch

from oracle import moe as M
from synth import CONFIGS, make_inputs
from tests.nvf_testutil import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvf():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as m
    return m


def _compare(nvf, logits, bias, k, renorm, shared):
    T, E = logits.shape
    o = nvf.route_permute(logits.cuda(), k, None if bias is None else bias.cuda(), renorm, shared)
    torch.cuda.synchronize()
    o = {n: v.cpu().numpy() for n, v in o.items()}
    ids, w = M.route(logits.numpy(), None if bias is None else bias.numpy(), k, renorm)
    counts, offs, p2s, s2p = M.permute(ids, E, shared)
    assert np.array_equal(o["topk_ids"], ids)
    assert np.allclose(o["topk_w"], w, rtol=1e-6, atol=1e-7)
    assert np.array_equal(o["expert_offsets"], offs)
    assert np.array_equal(o["tile_offsets"], M.tile_offsets(counts))
    assert np.array_equal(o["perm_to_src"], p2s)
    assert np.array_equal(o["src_to_perm"], s2p)
    assert np.array_equal(o["perm_token"], M.assignment_token(p2s, T, k))


@pytest.mark.parametrize("name", list(CONFIGS))
def test_configs(nvf, name):
    cfg = CONFIGS[name]
    _, logits, bias = make_inputs(cfg, seed=0)
    _compare(nvf, logits, bias, cfg.k, cfg.renormalize, cfg.shared)


@pytest.mark.parametrize("T,E,k,shared,renorm", [(1, 1, 1, False, True), (3, 32, 32, False, True),
                                                  (70, 1024, 10, True, False), (129, 7, 3, True, True),
                                                  (5000, 64, 6, False, False)])
def test_shapes(nvf, T, E, k, shared, renorm):
    logits = torch.randn(T, E, generator=torch.Generator().manual_seed(T + E))
    _compare(nvf, logits, None, k, renorm, shared)


def test_ties_go_to_lower_expert(nvf):
    logits = torch.zeros(200, 40)
    logits[:, 7] = 1.0
    logits[:, 3] = 1.0
    logits[::3, 30] = 1.0
    _compare(nvf, logits, None, 5, True, False)
    q = torch.round(torch.randn(300, 64, generator=torch.Generator().manual_seed(9)) * 2) / 2   # many equal values
    _compare(nvf, q, None, 8, True, True)


def test_empty_batch(nvf):
    o = nvf.route_permute(torch.zeros(0, 16, device="cuda"), 4, None, True, True)
    torch.cuda.synchronize()
    assert o["expert_offsets"].cpu().tolist() == [0] * 18
    assert o["tile_offsets"].cpu().tolist() == [0] * 18
