"""moe_route_permute_noalloc: routing without caller-provided scratch.

Some callers cannot allocate device memory (their framework's allocator owns
every allocation, or an allocation's implicit synchronisation is not
acceptable on their path), so the library offers this variant whose scratch is
a fixed array inside the library.  This test calls it through the C ABI and
checks that it gives exactly what moe_route_permute gives with a workspace, on
two calls in a row (the second call sees whatever the first left in the shared
array).  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.nvf_testutil import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nvf():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as m
    return m


def _outputs(T, E, k, shared):
    R = T * k + (T if shared else 0)
    Et = E + int(shared)
    mk = lambda n, dt=torch.int32: torch.full((max(n, 1),), -7, dtype=dt, device="cuda")
    return dict(topk_ids=mk(T * k), topk_w=mk(T * k, torch.float32), expert_offsets=mk(Et + 1),
                tile_offsets=mk(Et + 1), perm_to_src=mk(R), src_to_perm=mk(R), perm_token=mk(R))


def _call(nvf, name, logits, bias, k, renorm, shared):
    T, E = logits.shape
    o = _outputs(T, E, k, shared)
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    args = [p(logits), p(bias), T, E, k, int(renorm), int(shared), p(o["topk_ids"]), p(o["topk_w"]),
            p(o["expert_offsets"]), p(o["tile_offsets"]), p(o["perm_to_src"]), p(o["src_to_perm"]),
            p(o["perm_token"])]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    L = nvf.lib()
    if name == "moe_route_permute":
        n = ctypes.c_size_t(0)
        assert L.moe_route_permute_workspace_size(T, E, ctypes.byref(n)) == 0
        ws = torch.empty(n.value, dtype=torch.uint8, device="cuda")
        st = L.moe_route_permute(*args, p(ws), n.value, stream)
    else:
        st = L.moe_route_permute_noalloc(*args, stream)
    assert st == 0, L.nvf_last_error_message()
    torch.cuda.synchronize()
    return {n: v.cpu() for n, v in o.items()}


@pytest.mark.parametrize("first,second", [((8192, 256, 8, False, True), (32, 128, 8, False, True)),
                                          ((256, 512, 10, True, True), (4096, 128, 8, False, False))])
def test_matches_workspace_entry_point_on_consecutive_calls(nvf, first, second):
    for T, E, k, shared, zipf in (first, second):
        g = torch.Generator().manual_seed(T + E)
        logits = torch.randn(T, E, generator=g).cuda()
        bias = (-1.2 * torch.log(torch.arange(1, E + 1, dtype=torch.float64))).float().cuda() if zipf else None
        ref = _call(nvf, "moe_route_permute", logits, bias, k, True, shared)
        got = _call(nvf, "moe_route_permute_noalloc", logits, bias, k, True, shared)
        for name in ref:
            if name == "topk_w":
                # same kernels on the same inputs: equal; the tests' tolerance (1e-6 relative) is the bound
                assert torch.allclose(got[name], ref[name], rtol=1e-6, atol=0), name
            else:
                assert torch.equal(got[name], ref[name]), name


def _scratch_need(nvf, T, E):
    n = ctypes.c_size_t(0)
    assert nvf.lib().moe_route_permute_workspace_size(T, E, ctypes.byref(n)) == 0
    return n.value


def test_largest_call_that_fits_matches_workspace_entry_point(nvf):
    """T = 32736 tokens with 256 experts needs just under the 2 MiB of fixed
    scratch (2 * 1023 * 256 + 256 words); it must run and agree with the
    workspace entry point, twice in a row."""
    T, E, k = 32736, 256, 8
    need = _scratch_need(nvf, T, E)
    assert need == (2 * 1023 * E + E) * 4 and (2 << 20) - 2048 < need <= (2 << 20)
    g = torch.Generator().manual_seed(5)
    logits = torch.randn(T, E, generator=g).cuda()
    ref = _call(nvf, "moe_route_permute", logits, None, k, True, False)
    for _ in range(2):
        got = _call(nvf, "moe_route_permute_noalloc", logits, None, k, True, False)
        for name in ref:
            if name == "topk_w":
                assert torch.allclose(got[name], ref[name], rtol=1e-6, atol=0), name
            else:
                assert torch.equal(got[name], ref[name]), name


def test_smallest_call_that_does_not_fit_is_refused(nvf):
    """One token more (a 1024th word column per expert) needs 2 MiB + 1 KB:
    refused with NVF_ERR_WORKSPACE before anything is launched or written."""
    T, E, k = 32737, 256, 8
    assert _scratch_need(nvf, T, E) > (2 << 20)
    logits = torch.zeros(T, E, device="cuda")
    o = _outputs(T, E, k, False)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = nvf.lib().moe_route_permute_noalloc(p(logits), None, T, E, k, 1, 0, *[p(o[n]) for n in o], None)
    assert st == 3, nvf.lib().nvf_last_error_message()
    assert b"fixed" in nvf.lib().nvf_last_error_message()
    torch.cuda.synchronize()
    assert all(bool((v == -7).all()) for v in o.values())   # nothing was written


def test_argument_errors_match_workspace_entry_point(nvf):
    """A bad argument gets the status moe_route_permute returns (checked first)."""
    L = nvf.lib()
    for T, E, k in ((16, 8, 0), (16, 2000, 4), (-1, 8, 2)):
        a = L.moe_route_permute(None, None, T, E, k, 1, 0, None, None, None, None, None, None, None, None, 0, None)
        b = L.moe_route_permute_noalloc(None, None, T, E, k, 1, 0, None, None, None, None, None, None, None, None)
        assert a == b == 1, (T, E, k, a, b)


def test_rejects_sizes_beyond_the_fixed_scratch(nvf):
    T, E = 1 << 16, 1024
    n = ctypes.c_size_t(0)
    nvf.lib().moe_route_permute_workspace_size(T, E, ctypes.byref(n))
    assert n.value > (2 << 20)
    st = nvf.lib().moe_route_permute_noalloc(None, None, T, E, 8, 1, 0, None, None, None, None, None, None, None,
                                             None)
    assert st == 3   # NVF_ERR_WORKSPACE, before anything is launched
    assert b"fixed" in nvf.lib().nvf_last_error_message()
