"""CPU oracle for the NVFP4 mixture-of-experts expert computation.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this package:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code, tables or helpers with the CUDA
library; the two meet only on buffers drawn by ``synth``.

The oracle is plain and slow on purpose: numpy, float32 exactly where the
method rounds to float32 (block amax, scale and code decisions), float64
everywhere else (GEMM sums, SiLU, softmax, combine).  Every function names the
page passage it follows.  The sources are four web pages:

  * vLLM PR #29242 "[Kernel] Add NVFP4 MoE CUTLASS support for SM120"
  * FlashInfer issue #2723 "SM120 (RTX Blackwell) NVFP4 MoE: CUTLASS Grouped
    Block-Scaled GEMM Produces Invalid Output; FlashInfer Requires Extensive
    Patching"
  * vLLM PR #35737 "[NVFP4] NVFP4 MOE emulation fallback for H100/MI300/MI350"
  * unsloth "Report: NVFP4 kernel selection on SM120/SM121"

Pins (tests/test_oracle_*.py) tie each function to something other than
itself: closed forms of the formats, torch's float8 cast, independent scalar
encoders, brute-force sorts and exact rational arithmetic.  Every function here
is pinned; none is "parity unpinned".
"""
from . import ep, formats, moe  # noqa: F401
