"""GPU parity of the weight-only NVFP4 grouped GEMM (W4A16) against the oracle.

Activations are FP16 values, or BF16 values that the kernel rounds to FP16
(the oracle takes the same rounded values).  An exact special case (power-of-two scales,
small-integer activations, codes from the E2M1 table) must match bit for bit
and pins the nibble order and the scale placement; random cases must stay
within 5e-3 * rms of the oracle's float64 result.
"""
import numpy as np
import pytest
import torch

from oracle import moe as M
from tests.nvf_testutil import ensure_built, rel_err, weight_pack

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module")
def nvf():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as m
    return m


def _pack(q):
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def _run(nvf, a_f16, sizes, w_codes, w_scales, gs_w, out_dtype=torch.float32, a_torch=None):
    sizes = np.asarray(sizes, np.int64)
    G, N, Kh = w_codes.shape
    K = 2 * Kh
    offs = np.concatenate([[0], np.cumsum(sizes)])
    tiles = M.tile_offsets(sizes)
    B = weight_pack(w_codes.reshape(G * N, Kh), w_scales.reshape(G * N, K // 16), K, N, nvf.tiled_bytes(G * N, 0, K))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    A = a_torch.cuda() if a_torch is not None else torch.from_numpy(np.ascontiguousarray(a_f16)).cuda()
    if A.shape[0] == 0:
        A = torch.zeros(1, K, dtype=A.dtype, device="cuda")
    D = nvf.w4a16_grouped_gemm(A[: max(int(offs[-1]), 1)], dev(B), dev(np.asarray(gs_w, np.float32)),
                               dev(offs.astype(np.int32)), dev(tiles.astype(np.int32)), N, K, out_dtype)
    code, detail = nvf.device_status()
    assert code == 0, f"device error word {code} at {detail}"
    return D.float().cpu().numpy()[: int(offs[-1])], offs


def _random_weights(rng, G, N, K):
    w = (rng.standard_normal((G, N, K)) * 0.02).astype(np.float32)
    qw = [M.quantize_expert_weights(w[g]) for g in range(G)]
    return np.stack([q[0] for q in qw]), np.stack([q[1] for q in qw]), np.array([q[2] for q in qw], np.float32)


def test_exact_special_case(nvf):
    rng = np.random.default_rng(0)
    sizes = [130, 0, 1, 64]
    G, N, K = len(sizes), 256, 512
    R = sum(sizes)
    q_w = rng.integers(0, 16, (G, N, K)).astype(np.uint8)
    s_choices = np.array([0x30, 0x38, 0x40], np.uint8)      # 0.5, 1, 2
    s_w = s_choices[rng.integers(0, 3, (G, N, K // 16))]
    a = rng.integers(-2, 3, (R, K)).astype(np.float16)
    gs = np.ones(G, np.float32)
    D, offs = _run(nvf, a, sizes, _pack(q_w), s_w, gs)
    ref = M.grouped_w4a16(a.astype(np.float64), offs, _pack(q_w), s_w, gs)
    assert np.array_equal(D, ref.astype(np.float32)), f"max abs diff {np.max(np.abs(D - ref))}"


@pytest.mark.parametrize("sizes,N,K", [
    ([5], 128, 64),
    ([0, 1, 127, 128, 129], 256, 256),
    ([300, 7, 0, 45], 384, 320),
    ([1] * 40, 256, 2048),
])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_random_within_tolerance(nvf, sizes, N, K, out_dtype):
    rng = np.random.default_rng(sum(sizes) + N + K)
    G, R = len(sizes), sum(sizes)
    # BF16 activations rounded to FP16 (what a caller of the W4A16 path passes)
    a = torch.randn(R, K, generator=torch.Generator().manual_seed(R + K)).to(torch.bfloat16).to(torch.float16).numpy()
    w_c, w_s, gs_w = _random_weights(rng, G, N, K)
    D, offs = _run(nvf, a, sizes, w_c, w_s, gs_w, out_dtype)
    ref = M.grouped_w4a16(a.astype(np.float64), offs, w_c, w_s, gs_w)
    if out_dtype == torch.float32:
        assert rel_err(D, ref) <= TOL
    else:
        rms = np.sqrt(np.mean(ref ** 2))
        assert np.all(np.abs(D - ref) <= TOL * rms + np.abs(ref) * 2.0 ** -8)


def test_decode_shape(nvf):
    """The decode layer's gate_up shape: one row in each of 24 experts, N = 1536, K = 2048."""
    rng = np.random.default_rng(5)
    G, N, K = 24, 1536, 2048
    a = torch.randn(G, K, generator=torch.Generator().manual_seed(5)).to(torch.float16).numpy()
    w_c, w_s, gs_w = _random_weights(rng, G, N, K)
    D, offs = _run(nvf, a, [1] * G, w_c, w_s, gs_w)
    assert rel_err(D, M.grouped_w4a16(a.astype(np.float64), offs, w_c, w_s, gs_w)) <= TOL


@pytest.mark.parametrize("N,K", [(640, 320), (1536, 512)])
def test_many_items_per_cta(nvf, N, K):
    """More work items (token tile x weight pair) than SMs: every CTA runs
    several, so the rings wrap across items; N = 640 ends each group with an
    unpaired weight tile, K = 320 with a partial K tile; one group spans three
    token tiles."""
    rng = np.random.default_rng(N + K)
    sizes = list(rng.integers(0, 4, 150)) + [300] + list(rng.integers(0, 3, 50))
    G, R = len(sizes), int(sum(sizes))
    a = torch.randn(R, K, generator=torch.Generator().manual_seed(N)).to(torch.float16).numpy()
    w_c, w_s, gs_w = _random_weights(rng, G, N, K)
    D, offs = _run(nvf, a, sizes, w_c, w_s, gs_w)
    assert rel_err(D, M.grouped_w4a16(a.astype(np.float64), offs, w_c, w_s, gs_w)) <= TOL


def test_bf16_activations_exact(nvf):
    """Small integers are exact in BF16 and FP16: BF16 input gives the oracle's bits."""
    rng = np.random.default_rng(7)
    sizes = [40, 1, 129]
    G, N, K = len(sizes), 256, 256
    R = sum(sizes)
    q_w = rng.integers(0, 16, (G, N, K)).astype(np.uint8)
    s_w = np.array([0x30, 0x38, 0x40], np.uint8)[rng.integers(0, 3, (G, N, K // 16))]
    a = rng.integers(-4, 5, (R, K)).astype(np.float32)
    gs = np.ones(G, np.float32)
    D, offs = _run(nvf, None, sizes, _pack(q_w), s_w, gs, a_torch=torch.from_numpy(a).to(torch.bfloat16))
    ref = M.grouped_w4a16(a.astype(np.float64), offs, _pack(q_w), s_w, gs)
    assert np.array_equal(D, ref.astype(np.float32))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_bf16_activations_random(nvf, out_dtype):
    """BF16 activations are rounded to FP16 by the kernel: the result equals the
    FP16 path on the rounded values bit for bit, and the oracle on them within
    the tolerance."""
    rng = np.random.default_rng(8)
    sizes = [0, 3, 130, 17]
    G, N, K = len(sizes), 384, 320
    R = sum(sizes)
    a_bf = torch.randn(R, K, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    a16 = a_bf.to(torch.float16).numpy()           # round to nearest, what the kernel does
    w_c, w_s, gs_w = _random_weights(rng, G, N, K)
    D_bf, offs = _run(nvf, None, sizes, w_c, w_s, gs_w, out_dtype, a_torch=a_bf)
    D_16, _ = _run(nvf, a16, sizes, w_c, w_s, gs_w, out_dtype)
    assert np.array_equal(D_bf, D_16)
    ref = M.grouped_w4a16(a16.astype(np.float64), offs, w_c, w_s, gs_w)
    rms = np.sqrt(np.mean(ref ** 2))
    bound = TOL * rms + (np.abs(ref) * 2.0 ** -8 if out_dtype == torch.bfloat16 else 0.0)
    assert np.all(np.abs(D_bf - ref) <= bound)


def test_argument_validation(nvf):
    z = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    a = torch.zeros(4, 100, dtype=torch.float16, device="cuda")
    f = torch.ones(1, device="cuda")
    o = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
    with pytest.raises(nvf.NvfError, match="K=100"):
        nvf.w4a16_grouped_gemm(a, z, f, o, o, 128, 100)
    with pytest.raises(TypeError):
        nvf.w4a16_grouped_gemm(a.float(), z, f, o, o, 128, 64)
    # an activation type code other than FP16 / BF16, straight through the C ABI
    D = torch.zeros(4, 128, device="cuda")
    st = nvf.lib().nvfp4_w4a16_grouped_gemm(a.data_ptr(), nvf.NVF_F32, 4, 100, z.data_ptr(), f.data_ptr(),
                                            o.data_ptr(), o.data_ptr(), 1, 128, 64, nvf.NVF_F32, D.data_ptr(), 128,
                                            None)
    assert st == 1 and b"a_dtype" in nvf.lib().nvf_last_error_message()
