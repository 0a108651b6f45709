"""GPU parity of the grouped block-scaled FP4 GEMM (tcgen05) against the oracle.

Operands are built on the host (random codes, or the oracle's quantization of
random float32 data) and fed unchanged to both sides.  An exact special case
(power-of-two scales, small K) must match bit for bit; random cases must stay
within 5e-3 * rms of the oracle's float64 result.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import moe as M
from tests.nvf_testutil import ensure_built, rel_err, row_tiles, tiled_pack, weight_pack

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module")
def nvf():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as m
    return m


def _pack(q):
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def _run(nvf, a_codes, a_scales, sizes, w_codes, w_scales, gs_a, gs_w, out_dtype=torch.float32, pad_rows=0):
    sizes = np.asarray(sizes, np.int64)
    G, N, Kh = w_codes.shape
    K = 2 * Kh
    offs = np.concatenate([[0], np.cumsum(sizes)])
    tiles = M.tile_offsets(sizes)
    R = int(offs[-1])
    rows = max(R + pad_rows, 1)
    ta, ra = row_tiles(R, offs, tiles)
    A = tiled_pack(a_codes, a_scales, K, ta, ra, nvf.tiled_bytes(rows, G, K))
    B = weight_pack(w_codes.reshape(G * N, Kh), w_scales.reshape(G * N, K // 16), K, N, nvf.tiled_bytes(G * N, 0, K))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    D = nvf.grouped_gemm(dev(A), rows, dev(B), dev(np.asarray(gs_a, np.float32)), dev(np.asarray(gs_w, np.float32)),
                         dev(offs.astype(np.int32)), dev(tiles.astype(np.int32)), N, K, out_dtype)
    code, detail = nvf.device_status()
    assert code == 0, f"device error word {code} at {detail}"
    return D.float().cpu().numpy()[:R], offs


def test_exact_special_case(nvf):
    """E2M1 codes x scales in {1/2, 1, 2}: every partial sum is exact in FP32,
    so the GPU must equal the oracle bit for bit.  Distinct per-row, per-block
    scales and asymmetric codes pin the nibble order and the scale-atom layout."""
    rng = np.random.default_rng(0)
    sizes = [130, 0, 1, 127, 128]
    G, N, K = len(sizes), 256, 512
    R = sum(sizes)
    q_a = rng.integers(0, 16, (R, K)).astype(np.uint8)
    q_w = rng.integers(0, 16, (G, N, K)).astype(np.uint8)
    s_choices = np.array([0x30, 0x38, 0x40], np.uint8)   # 0.5, 1, 2
    s_a = s_choices[rng.integers(0, 3, (R, K // 16))]
    s_w = s_choices[rng.integers(0, 3, (G, N, K // 16))]
    D, offs = _run(nvf, _pack(q_a), s_a, sizes, _pack(q_w), s_w, np.ones(G), np.ones(G))
    ref = M.grouped_gemm(_pack(q_a), s_a, offs, np.ones(G, np.float32), _pack(q_w), s_w, np.ones(G, np.float32))
    assert np.array_equal(D, ref.astype(np.float32)), f"max abs diff {np.max(np.abs(D - ref))}"


def test_exact_single_element_probes(nvf):
    """One nonzero code per row at a chosen K position and one nonzero scale
    block: locates each K index and each scale byte exactly."""
    G, N, K = 1, 128, 256
    R = 128
    q_a = np.zeros((R, K), np.uint8)
    s_a = np.full((R, K // 16), 0x38, np.uint8)
    for r in range(R):
        q_a[r, (r * 37) % K] = 2          # value 1.0 at one K position per row
        s_a[r, (r * 37 % K) // 16] = 0x40  # its block scale 2.0
    q_w = np.zeros((G, N, K), np.uint8)
    s_w = np.full((G, N, K // 16), 0x38, np.uint8)
    for n in range(N):
        q_w[0, n, :] = (n % 7) + 1         # distinct positive values per column
        s_w[0, n, n % (K // 16)] = 0x30
    D, offs = _run(nvf, _pack(q_a), s_a, [R], _pack(q_w), s_w, [1.0], [1.0])
    ref = M.grouped_gemm(_pack(q_a), s_a, offs, np.ones(1, np.float32), _pack(q_w), s_w, np.ones(1, np.float32))
    assert np.array_equal(D, ref.astype(np.float32))


@pytest.mark.parametrize("sizes,N,K", [
    ([5], 128, 64),
    ([0, 1, 127, 128, 129], 256, 256),
    ([300, 7, 0, 0, 45], 384, 320),
    ([33, 200], 128, 128),
    ([1] * 40, 256, 2048),
    ([8065, 0, 513], 1536, 2048),
])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_random_within_tolerance(nvf, sizes, N, K, out_dtype):
    rng = np.random.default_rng(sum(sizes) + N + K)
    G = len(sizes)
    R = sum(sizes)
    a = rng.standard_normal((R, K)).astype(np.float32)
    gs_a = np.full(G, F.global_scale(np.abs(a).max() if R else 1.0), np.float32)
    a_c, a_s = F.quantize_rows(a, gs_a[0])
    w = (rng.standard_normal((G, N, K)) * 0.02).astype(np.float32)
    qw = [M.quantize_expert_weights(w[g]) for g in range(G)]
    w_c = np.stack([q[0] for q in qw])
    w_s = np.stack([q[1] for q in qw])
    gs_w = np.array([q[2] for q in qw], np.float32)
    D, offs = _run(nvf, a_c, a_s, sizes, w_c, w_s, gs_a, gs_w, out_dtype, pad_rows=3)
    ref = M.grouped_gemm(a_c, a_s, offs, gs_a, w_c, w_s, gs_w)
    err = rel_err(D, ref)
    if out_dtype == torch.float32:
        assert err <= TOL, err
    else:
        # bf16 output: the same bound plus one bf16 rounding of each element
        rms = np.sqrt(np.mean(ref ** 2))
        assert np.all(np.abs(D - ref) <= TOL * rms + np.abs(ref) * 2.0 ** -8)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_split_last_round(nvf, out_dtype):
    """Few row blocks and a large row capacity: the launch gets one CTA per SM
    and every 256-column block is split into two 128-column tiles (the kernel
    halves the last round when it would leave most CTAs idle)."""
    rng = np.random.default_rng(11)
    sizes = [5, 7, 130, 0, 64]
    G, N, K = len(sizes), 512, 320
    R = sum(sizes)
    a = rng.standard_normal((R, K)).astype(np.float32)
    gs_a = np.full(G, F.global_scale(np.abs(a).max()), np.float32)
    a_c, a_s = F.quantize_rows(a, gs_a[0])
    w = (rng.standard_normal((G, N, K)) * 0.02).astype(np.float32)
    qw = [M.quantize_expert_weights(w[g]) for g in range(G)]
    w_c = np.stack([q[0] for q in qw])
    w_s = np.stack([q[1] for q in qw])
    gs_w = np.array([q[2] for q in qw], np.float32)
    D, offs = _run(nvf, a_c, a_s, sizes, w_c, w_s, gs_a, gs_w, out_dtype, pad_rows=30000)
    ref = M.grouped_gemm(a_c, a_s, offs, gs_a, w_c, w_s, gs_w)
    rms = np.sqrt(np.mean(ref ** 2))
    bound = TOL * rms + (np.abs(ref) * 2.0 ** -8 if out_dtype == torch.bfloat16 else 0.0)
    assert np.all(np.abs(D - ref) <= bound)


@pytest.mark.parametrize("rows", [1, 16, 300])
def test_dense_linear(nvf, rows):
    """A dense NVFP4 W4A4 linear layer is the grouped GEMM with one group: the
    pages' second workload (gate_up with K = 5120) at a reduced N."""
    rng = np.random.default_rng(rows)
    N, K = 512, 5120
    a = rng.standard_normal((rows, K)).astype(np.float32)
    gs_a = np.array([F.global_scale(np.abs(a).max())], np.float32)
    a_c, a_s = F.quantize_rows(a, gs_a[0])
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w_c, w_s, g = M.quantize_expert_weights(w)
    gs_w = np.array([g], np.float32)
    D, offs = _run(nvf, a_c, a_s, [rows], w_c[None], w_s[None], gs_a, gs_w)
    ref = M.grouped_gemm(a_c, a_s, offs, gs_a, w_c[None], w_s[None], gs_w)
    assert rel_err(D, ref) <= TOL


@pytest.mark.parametrize("rows", [1, 300, 2048])
def test_dense_linear_pages_shape(nvf, rows):
    """The dense W4A4 linear at the pages' gate_up shape (N = 34816, K = 5120),
    through the product path: activations and weights quantized on the GPU, then
    the grouped GEMM with one group.  The oracle quantizes the same float rows
    (same global scales, an input here) and computes 256 sampled output columns."""
    N, K = 34816, 5120
    g = torch.Generator(device="cuda").manual_seed(4096 + rows)
    w = torch.randn(N, K, generator=g, device="cuda") * 0.02
    a = torch.randn(rows, K, generator=g, device="cuda")
    gs_w = np.float32(F.global_scale(np.float32(w.abs().max().item())))
    gs_a = np.float32(F.global_scale(np.float32(a.abs().max().item())))
    dev32 = lambda v: torch.tensor([v], dtype=torch.float32, device="cuda")
    B, _ = nvf.quantize(w, dev32(gs_w), layout=nvf.LAYOUT_TILED)
    offs = torch.tensor([0, rows], dtype=torch.int32, device="cuda")
    tiles = torch.tensor([0, (rows + 127) // 128], dtype=torch.int32, device="cuda")
    A, _ = nvf.quantize(a, dev32(gs_a), layout=nvf.LAYOUT_TILED_GROUPED, offsets=offs, tile_offsets=tiles)
    D = nvf.grouped_gemm(A, rows, B, dev32(gs_a), dev32(gs_w), offs, tiles, N, K, torch.float32)
    code, detail = nvf.device_status()
    assert code == 0, f"device error word {code} at {detail}"
    cols = np.sort(np.random.default_rng(rows).choice(N, 256, replace=False))
    w_c, w_s = F.quantize_rows(w[torch.from_numpy(cols).cuda()].cpu().numpy(), gs_w)
    a_c, a_s = F.quantize_rows(a.cpu().numpy(), gs_a)
    ref = M.grouped_gemm(a_c, a_s, np.array([0, rows]), np.array([gs_a]), w_c[None], w_s[None], np.array([gs_w]))
    assert rel_err(D[:rows].cpu().numpy()[:, cols], ref) <= TOL


def test_argument_validation(nvf):
    z = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    f = torch.ones(1, dtype=torch.float32, device="cuda")
    o = torch.tensor([0, 0], dtype=torch.int32, device="cuda")
    with pytest.raises(nvf.NvfError, match="N=100"):
        nvf.grouped_gemm(z, 2, z, f, f, o, o, 100, 256)
    with pytest.raises(nvf.NvfError, match="K=100"):
        nvf.grouped_gemm(z, 2, z, f, f, o, o, 128, 100)
