"""Failure detection on the GPU without a fault: every pipeline wait in the
library's kernels is bounded.  The self-test entry point runs one such wait on
a barrier that nothing will ever complete; the wait must give up after its
limit, report through the device error word, and leave the context usable."""
import time

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


def test_expired_wait_is_reported_and_the_context_survives(nvf):
    assert nvf.device_status() == (0, 0)
    t0 = time.perf_counter()
    nvf.selftest_bounded_wait(20_000_000)          # 20 ms
    code, detail = nvf.device_status()              # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert code == 6 and detail == 0
    assert 0.015 <= elapsed < 5.0
    assert nvf.device_status() == (0, 0)            # the word was cleared
    # the context still runs kernels correctly
    x = torch.randn(8, 256, device="cuda")
    gs = nvf.global_scale(x)
    assert torch.isfinite(gs).all() and gs.item() == pytest.approx(x.abs().max().item() / 2688, rel=1e-6)


def test_selftest_argument_check(nvf):
    with pytest.raises(nvf.NvfError, match="limit_ns"):
        nvf.selftest_bounded_wait(10)
