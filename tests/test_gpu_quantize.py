"""GPU parity of the NVFP4 quantizer and global scale against the oracle (bit-exact)."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from tests.nvf_testutil import ensure_built, row_tiles, tiled_unpack, weight_unpack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvf():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as m
    return m


def _gpu_quant(nvf, x, gs, layout=0, **kw):
    g = torch.tensor([gs], dtype=torch.float32, device="cuda") if np.isscalar(gs) else gs
    c, s = nvf.quantize(x, g, layout, **kw)
    torch.cuda.synchronize()
    return c.cpu().numpy(), (None if s is None else s.cpu().numpy())


def _check_rowmajor(nvf, x, gs):
    codes, scales = _gpu_quant(nvf, x.cuda(), np.float32(gs))
    ref_c, ref_s = F.quantize_rows(x.float().numpy(), np.float32(gs))
    rows, K = x.shape
    assert np.array_equal(scales[: rows * K // 16].reshape(rows, K // 16), ref_s)
    assert np.array_equal(codes, ref_c)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,K", [(1, 64), (37, 256), (300, 2048), (5, 4096)])
def test_random_rows(nvf, dtype, rows, K):
    g = torch.Generator().manual_seed(rows * K)
    x = (torch.randn(rows, K, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 2)).to(dtype)
    amax = float(x.float().abs().max())
    for gs in (F.global_scale(amax), np.float32(amax / 300.0), np.float32(amax / 10000.0)):
        _check_rowmajor(nvf, x, gs)


def test_every_bf16_value(nvf):
    bits = np.arange(65536, dtype=np.uint32) << 16
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    vals = vals[np.abs(vals) < 1e30]
    n = len(vals) // 64 * 64
    x = torch.from_numpy(vals[:n].reshape(-1, 64).copy()).to(torch.bfloat16)
    for gs in (1.0, 1e-3, 7.5, 1e-20):
        _check_rowmajor(nvf, x, np.float32(gs))


def test_ties_signed_zero_and_saturation(nvf):
    # gs = 1 and a block amax of 6 give r = 1, so x itself is rounded to E2M1.
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -5.0, -0.1, -0.0, 0.0, 0.1, 6.0, -6.0]
    row = np.array(mids * 4, np.float32)
    x = torch.from_numpy(np.stack([row, np.zeros(64, np.float32), -np.zeros(64, np.float32),
                                   row * 1e30]))
    _check_rowmajor(nvf, x, np.float32(1.0))
    _check_rowmajor(nvf, x.to(torch.bfloat16), np.float32(1.0))


@pytest.mark.parametrize("groups,group_rows", [(1, 517), (3, 384), (2, 512)])
@pytest.mark.parametrize("K", [512, 320, 64])
def test_weight_layout(nvf, groups, group_rows, K):
    """TILED (weights): groups of rows with one global scale each; paired
    36864-byte units, and an odd last tile per group (517 and 384 rows)."""
    rows = groups * group_rows
    x = torch.randn(rows, K, generator=torch.Generator().manual_seed(3 + groups)).to(torch.bfloat16)
    gs = np.array([F.global_scale(float(x[g * group_rows:(g + 1) * group_rows].float().abs().max()))
                   for g in range(groups)], np.float32)
    ref_c, ref_s = F.quantize_rows(x.float().numpy(), np.repeat(gs, group_rows))
    buf, _ = nvf.quantize(x.cuda(), torch.tensor(gs, device="cuda"), layout=1, groups=groups)
    c, s_ = weight_unpack(buf.cpu().numpy(), K, rows, group_rows)
    assert np.array_equal(c, ref_c)
    assert np.array_equal(s_, ref_s)


@pytest.mark.parametrize("K", [512, 320, 64])
def test_grouped_activation_layout(nvf, K):
    """TILED_GROUPED (activations): per-group 128-row tiles, empty groups included."""
    rows = 517
    x = torch.randn(rows, K, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    gs = F.global_scale(float(x.float().abs().max()))
    ref_c, ref_s = F.quantize_rows(x.float().numpy(), gs)
    sizes = np.array([0, 130, 1, 0, 256, 127, 3], np.int64)
    sizes[-1] = rows - sizes[:-1].sum()
    offs = np.concatenate([[0], np.cumsum(sizes)])
    tiles = np.concatenate([[0], np.cumsum((sizes + 127) // 128)])
    gsv = torch.full((len(sizes),), float(gs), dtype=torch.float32, device="cuda")
    buf, _ = _gpu_quant(nvf, x.cuda(), gsv, layout=2,
                        offsets=torch.tensor(offs, dtype=torch.int32, device="cuda"),
                        tile_offsets=torch.tensor(tiles, dtype=torch.int32, device="cuda"))
    tile, r = row_tiles(rows, offs, tiles)
    c, s_ = tiled_unpack(buf, K, tile, r)
    assert np.array_equal(c, ref_c)
    assert np.array_equal(s_, ref_s)


def test_gather_and_per_group_scales(nvf):
    T, K = 40, 256
    x = torch.randn(T, K, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    gather = np.random.default_rng(5).integers(0, T, 100).astype(np.int32)
    offs = np.array([0, 30, 30, 100], np.int64)
    gs = np.array([0.002, 0.5, 0.0007], np.float32)
    c, s = _gpu_quant(nvf, x.cuda(), torch.tensor(gs, device="cuda"), layout=0,
                      gather=torch.tensor(gather, device="cuda"),
                      offsets=torch.tensor(offs, dtype=torch.int32, device="cuda"))
    xf = x.float().numpy()[gather]
    rgs = np.repeat(gs, np.diff(offs))
    ref_c, ref_s = F.quantize_rows(xf, rgs)
    assert np.array_equal(c, ref_c)
    assert np.array_equal(s[: 100 * K // 16].reshape(100, -1), ref_s)


def test_global_scale(nvf):
    x = torch.randn(6, 1000, generator=torch.Generator().manual_seed(6)) * torch.arange(1, 7)[:, None]
    x[2] = 0
    gs = nvf.global_scale(x.cuda(), groups=6).cpu().numpy()
    ref = [F.global_scale(np.max(np.abs(r))) for r in x.numpy()]
    assert np.array_equal(gs, np.array(ref, np.float32))
    xb = x.to(torch.bfloat16)
    gsb = nvf.global_scale(xb.cuda(), groups=3).cpu().numpy()
    ref_b = [F.global_scale(np.max(np.abs(r))) for r in xb.float().numpy().reshape(3, -1)]
    assert np.array_equal(gsb, np.array(ref_b, np.float32))
