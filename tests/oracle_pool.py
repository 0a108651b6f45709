"""Parallel evaluation of the oracle's per-expert weight quantization.

The oracle is plain numpy and quantizes one expert at a time; large layers
touch hundreds of experts, so the tests fan the experts out over a process
pool.  The pool uses the "spawn" start method (safe after CUDA has been
initialised in the parent).
"""
import multiprocessing as mp
import os

import numpy as np

_POOL = None


def pool():
    global _POOL
    if _POOL is None:
        ctx = mp.get_context("spawn")
        _POOL = ctx.Pool(max(1, min(16, os.cpu_count() or 1)), initializer=_init)
    return _POOL


def _init():
    import torch
    torch.set_num_threads(1)


def _quant_pair(args):
    from oracle import moe as M
    w13, w2 = args
    return (*M.quantize_expert_weights(w13), *M.quantize_expert_weights(w2))


def _quant_generated(args):
    from synth import expert_weights
    cfg, e, seed = args
    w13, w2 = expert_weights(cfg, e, seed, device="cpu")
    return _quant_pair((w13.numpy(), w2.numpy()))


def quantize_generated(cfg, experts, seed=0):
    """Oracle weights of CPU-generated experts: {e: (c13, s13, gs13, c2, s2, gs2)}."""
    experts = list(experts)
    res = pool().map(_quant_generated, [(cfg, e, seed) for e in experts], chunksize=1)
    return dict(zip(experts, res))


def quantize_arrays(pairs):
    """Oracle weights of given FP32 arrays: {e: (...)} for pairs {e: (w13, w2)}."""
    keys = list(pairs)
    res = pool().map(_quant_pair, [pairs[e] for e in keys], chunksize=1)
    return dict(zip(keys, res))
