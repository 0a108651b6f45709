"""The C ABI library builds, loads and exports every declared entry point;
host-only entry points behave as documented (CPU, no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

from tests.nvf_testutil import ROOT, ensure_built, w13_prepared_rows

HEADER = os.path.join(ROOT, "include", "nvfp4moe.h")


@pytest.fixture(scope="module")
def nvf():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as m
    m.lib()
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z_0-9]*\s*\**\s+\**([a-z_][a-z_0-9]*)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_four_method_entry_points():
    names = declared_functions()
    for n in ("nvfp4_quantize", "moe_route_permute", "nvfp4_grouped_gemm", "nvfp4_moe_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(nvf):
    L = nvf.lib()
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(L, n), f"{n} not exported"
        assert n in nvf.SIGNATURES, f"{n} has no binding signature"


def test_host_helpers(nvf):
    L = nvf.lib()
    assert L.nvf_abi_version() == 100
    assert L.nvf_status_string(1) == b"NVF_ERR_INVALID_ARG"
    assert list(nvf.w13_row_map(128)) == list(w13_prepared_rows(128))
    assert sorted(nvf.w13_row_map(192)) == list(range(384))
    with pytest.raises(nvf.NvfError):
        nvf.w13_row_map(100)
    assert nvf.tiled_bytes(300, 4, 256) == (3 + 4) * 1 * 18432
    assert nvf.tiled_bytes(256, 0, 768) == 2 * 3 * 18432


def test_workspace_layout(nvf):
    L = nvf.workspace_layout(256, 512, 4096, 1024, 10, True)
    assert L["R"] == 256 * 11
    offs = [L[n] for n in ("topk_ids", "topk_w", "expert_offsets", "tile_offsets", "perm_to_src", "src_to_perm",
                           "perm_token", "route_scratch", "tile_group", "a1", "a2", "y", "logits")]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs) and L["logits"] >= L["y"] + L["R"] * 4096 * 4
    assert L["total"] >= L["logits"] + 256 * 513 * 4
    with pytest.raises(nvf.NvfError):
        nvf.workspace_layout(16, 8, 200, 128, 2, False)       # H not a multiple of 128
    with pytest.raises(nvf.NvfError):
        nvf.workspace_layout(16, 8, 256, 128, 9, False)       # k > E


def test_compute_entry_points_fail_cleanly_without_a_gpu(nvf):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    L = nvf.lib()
    st = L.nvfp4_quantize(None, 0, 0, 64, 64, None, None, None, 1, None, None, None, 0, None)
    assert st in (2, 4)   # unsupported device / CUDA error: no CPU fallback
    assert L.nvf_last_error_message()


def test_route_entry_points_report_the_same_status_without_a_gpu(nvf):
    """The no-alloc routing call makes the device check first, like the
    workspace call: without a usable GB300 both return the same status and
    neither touches its scratch."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    L = nvf.lib()
    a = L.moe_route_permute(None, None, 16, 8, 2, 1, 0, None, None, None, None, None, None, None, None, 0, None)
    b = L.moe_route_permute_noalloc(None, None, 16, 8, 2, 1, 0, None, None, None, None, None, None, None, None)
    assert a == b and a in (2, 4)
