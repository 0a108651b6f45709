"""Workload shapes and seeded generators for the NVFP4 MoE expert computation.

The five layer shapes follow the model families the source pages run: a
Qwen3-30B-A3B-class MoE (128 experts, top-8; vLLM PR #29242 "Test Result" and
vLLM PR #35737 "Purpose") at decode and prefill batch sizes, a 397B-A17B-class
layer with 512 routed experts plus one shared expert and top-10 routing
(FlashInfer issue #2723, "Model" table), a tiny layer for brute-force checks,
and a skewed-routing stress case.

Recipe (all draws are float32, standard normal scaled where stated):
  * x       : N(0, 1) of shape [T, H], rounded to bfloat16 (round-to-nearest-even).
  * logits  : N(0, 1) of shape [T, E] (float32).
  * bias    : only for the skewed case: bias_e = -s * ln(e + 1) (Zipf exponent s),
              evaluated in float64 and rounded to float32.
  * w13[e]  : 0.02 * N(0, 1) of shape [2I, H]; rows [0, I) are the gate
              projection, rows [I, 2I) the up projection.
  * w2[e]   : 0.02 * N(0, 1) of shape [H, I].
Every tensor has its own generator seeded from (seed, stream, expert), so any
expert's weights can be drawn on their own.  On device "cpu" the CPU generator
is used; on a CUDA device torch's CUDA generator is used (a different stream of
numbers with the same distribution) so that multi-GB weight sets are drawn in
seconds.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int          # tokens
    H: int          # hidden size
    I: int          # expert intermediate size
    E: int          # routed experts
    k: int          # experts per token
    shared: bool = False       # one always-on shared expert (id E)
    zipf_s: float | None = None  # per-expert routing bias exponent
    renormalize: bool = True
    description: str = field(default="", compare=False)

    @property
    def E_total(self) -> int:
        return self.E + (1 if self.shared else 0)

    @property
    def R(self) -> int:
        """Permuted rows: T*k routed assignments plus T shared-expert rows."""
        return self.T * self.k + (self.T if self.shared else 0)

    def scaled(self, **kw) -> "LayerConfig":
        d = dict(self.__dict__)
        d.update(kw)
        return LayerConfig(**d)


CONFIGS = {
    "tiny": LayerConfig("tiny", T=16, H=256, I=128, E=8, k=2,
                        description="tiny NVFP4 MoE layer, top-2"),
    "decode": LayerConfig("decode", T=32, H=2048, I=768, E=128, k=8,
                          description="30B-A3B-shaped layer at decode batch 32"),
    "prefill": LayerConfig("prefill", T=4096, H=2048, I=768, E=128, k=8,
                           description="30B-A3B-shaped layer, 4096-token prefill"),
    "large": LayerConfig("large", T=256, H=4096, I=1024, E=512, k=10, shared=True,
                         description="397B-A17B-shaped layer, 512 routed + 1 shared, top-10"),
    "skewed": LayerConfig("skewed", T=8192, H=4096, I=1536, E=256, k=8, zipf_s=1.2,
                          description="Zipf(1.2)-biased routing stress, 8192 tokens"),
}

_STREAM_X, _STREAM_LOGITS, _STREAM_W13, _STREAM_W2, _STREAM_GATE = 1, 2, 3, 4, 5


def _seed(seed: int, stream: int, index: int = 0) -> int:
    return (seed * 1_000_003 + stream * 65_537 + index * 7919 + 12345) & ((1 << 62) - 1)


def _gen(device, seed: int, stream: int, index: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(seed, stream, index))
    return g


def zipf_bias(E: int, s: float) -> torch.Tensor:
    """bias_e = -s * ln(e + 1): log of the unnormalised Zipf pmf of rank e + 1."""
    return torch.tensor([-s * math.log(e + 1.0) for e in range(E)], dtype=torch.float64).to(torch.float32)


def make_inputs(cfg: LayerConfig, seed: int = 0, device="cpu"):
    """Activations (bf16 [T,H]), router logits (fp32 [T,E]) and optional bias (fp32 [E])."""
    x = torch.randn(cfg.T, cfg.H, generator=_gen(device, seed, _STREAM_X), device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    logits = torch.randn(cfg.T, cfg.E, generator=_gen(device, seed, _STREAM_LOGITS), device=device,
                         dtype=torch.float32)
    bias = zipf_bias(cfg.E, cfg.zipf_s).to(device) if cfg.zipf_s is not None else None
    return x, logits, bias


def expert_weights(cfg: LayerConfig, e: int, seed: int = 0, device="cpu"):
    """FP32 weights of expert e (e == E is the shared expert): w13 [2I,H], w2 [H,I]."""
    w13 = torch.randn(2 * cfg.I, cfg.H, generator=_gen(device, seed, _STREAM_W13, e), device=device,
                      dtype=torch.float32) * 0.02
    w2 = torch.randn(cfg.H, cfg.I, generator=_gen(device, seed, _STREAM_W2, e), device=device,
                     dtype=torch.float32) * 0.02
    return w13, w2


def gate_weights(cfg: LayerConfig, seed: int = 0, shared_gate: bool = False, device="cpu"):
    """Router gate rows, bf16 [E (+1), H]: 0.02 * N(0, 1) drawn in FP32 and rounded
    to bf16 (so x . w_gate has a spread like the N(0, 1) logits of the recipe);
    with shared_gate, one more row that gates the shared expert."""
    n = cfg.E + (1 if shared_gate else 0)
    w = torch.randn(n, cfg.H, generator=_gen(device, seed, _STREAM_GATE), device=device,
                    dtype=torch.float32) * 0.02
    return w.to(torch.bfloat16)
