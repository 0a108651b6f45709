"""Write tests/golden/activation_scales.json: static activation global scales.

The layer's activation quantizers use static FP32 global scales (one value per
expert array, all equal here).  Reading adopted for the pages' silence on how
they are set: calibrate them on the layer's own synthetic input with the
oracle,
    gs_a1 = amax(x) / 2688,
    gs_a2 = amax(h) / 2688, h = silu(gate) * up from the oracle's GEMM1,
where 2688 = 6 * 448 (largest E2M1 value times largest E4M3 value).
Runs only the oracle (CPU) and the seeded generator; takes minutes for the
two largest layers.

    python tests/golden/make_activation_scales.py [config ...]
"""
import json
import os
import sys
import time

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import formats as F  # noqa: E402
from oracle import moe as M  # noqa: E402
from synth import CONFIGS, expert_weights, make_inputs  # noqa: E402

OUT = os.path.join(HERE, "activation_scales.json")


def calibrate(cfg, seed=0):
    x, logits, bias = make_inputs(cfg, seed)
    xf = x.to(torch.float32).numpy()
    gs_a1 = F.global_scale(np.max(np.abs(xf)))
    ids, _ = M.route(logits.numpy(), None if bias is None else bias.numpy(), cfg.k, cfg.renormalize)
    counts, offsets, p2s, _ = M.permute(ids, cfg.E, cfg.shared)
    tok = M.assignment_token(p2s, cfg.T, cfg.k)
    hmax = np.float32(0.0)
    for e in range(cfg.E_total):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        w13, _ = expert_weights(cfg, e, seed)
        c13, s13, g13 = M.quantize_expert_weights(w13.numpy())
        ac, asc = F.quantize_rows(xf[tok[lo:hi]], gs_a1)
        c1 = np.float64(M.alpha(gs_a1, g13)) * M.block_scaled_matmul(ac, asc, c13, s13)
        h = M.swiglu(c1, cfg.I).astype(np.float32)
        hmax = max(hmax, np.float32(np.max(np.abs(h))))
    return float(gs_a1), float(F.global_scale(hmax))


def main(names):
    data = json.load(open(OUT)) if os.path.exists(OUT) else {}
    data["_source"] = ("gs_a1 = amax(x)/2688 and gs_a2 = amax(h)/2688 from the oracle on the seed-0 "
                       "synthetic layer (CPU generator); written by make_activation_scales.py")
    for n in names:
        t = time.time()
        a1, a2 = calibrate(CONFIGS[n])
        data[n] = {"seed": 0, "gs_a1": a1, "gs_a2": a2}
        print(n, a1, a2, f"{time.time() - t:.1f}s", flush=True)
        json.dump(data, open(OUT, "w"), indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:] or list(CONFIGS))
