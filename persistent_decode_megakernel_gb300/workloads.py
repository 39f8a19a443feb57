"""Seeded synthetic workloads: decoder shapes, weights, token streams and pre-RoPE K/V.

This module only draws random numbers and lays them out.  It holds none of the decoder's
arithmetic (no norm, projection, rotation or attention), so both the CUDA path and the CPU
oracle can take their inputs from it without sharing any computation.

The shapes are Llama-shaped decoders sized like the models on the MegaBake decode leaderboard
(project website, "Decode leaderboard": SmolLM-135M, Qwen2-0.5B, SmolLM-1.7B) plus a tiny
decoder for fast checks and a long-context variant of the 135M shape ("Where it breaks today":
long-context split attention).  The pages benchmark real Hugging Face checkpoints; seeded random
weights with the same shapes stand in for them (the values change neither bytes nor flops).

Generation order for one torch.Generator seeded with `seed` (fixed so results are reproducible):
  embedding E, then for each layer: [attn_norm], wq, wk, wv, (bq, bk, bv), wo, [mlp_norm],
  w_gate, w_up, w_down; then [final_norm]; then the token stream; then (long-context only)
  K_raw for all layers, then V_raw for all layers.
Norm gains are exactly 1.0 and draw nothing, unless `random_gains=True`, which draws them
uniform in [0.5, 1.5) at their position in the order above (used to exercise the gain).
Weights are N(0, 0.02) drawn in fp32, then rounded to bf16 (round to nearest even).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import torch


@dataclasses.dataclass(frozen=True)
class DecoderShape:
    name: str
    n_layers: int
    hidden: int
    intermediate: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    vocab: int
    kv_capacity: int
    rms_eps: float
    rope_theta: float
    qkv_bias: bool
    steps: int          # teacher-forced decode steps
    pos0: int = 0       # position of the first decode step
    prefill: int = 0    # cache rows 0..prefill-1 filled from K_raw / V_raw before decoding

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads

    def param_count(self) -> int:
        """Parameters of the decoder with tied embeddings (norm gains and biases included)."""
        H, I, d = self.hidden, self.intermediate, self.head_dim
        qd, kvd = self.n_heads * d, self.n_kv_heads * d
        per_layer = H * qd + 2 * H * kvd + qd * H + 3 * H * I + 2 * H
        if self.qkv_bias:
            per_layer += qd + 2 * kvd
        return self.n_layers * per_layer + self.vocab * H + H


SHAPES: Dict[str, DecoderShape] = {
    s.name: s
    for s in [
        DecoderShape("tiny", 2, 256, 688, 4, 2, 64, 4096, 128, 1e-5, 1e4, False, steps=32),
        DecoderShape("smollm-135m", 30, 576, 1536, 9, 3, 64, 49152, 128, 1e-5, 1e4, False, steps=128),
        DecoderShape("qwen2-0.5b", 24, 896, 4864, 14, 2, 64, 151936, 128, 1e-6, 1e6, True, steps=128),
        DecoderShape("smollm-135m-long", 30, 576, 1536, 9, 3, 64, 49152, 8192, 1e-5, 1e4, False,
                     steps=64, pos0=4096, prefill=4096),
        DecoderShape("smollm-1.7b", 24, 2048, 8192, 32, 32, 64, 49152, 128, 1e-5, 1e4, False, steps=64),
    ]
}

LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "bq", "bk", "bv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")


@dataclasses.dataclass
class Workload:
    shape: DecoderShape
    embed: torch.Tensor                       # bf16 [V, H]
    final_norm: torch.Tensor                  # bf16 [H]
    layers: List[Dict[str, Optional[torch.Tensor]]]
    tokens: torch.Tensor                      # int64 [steps]
    k_raw: Optional[torch.Tensor] = None      # fp32 [L, nkv, prefill, d]   (pre-RoPE)
    v_raw: Optional[torch.Tensor] = None      # fp32 [L, nkv, prefill, d]

    @property
    def positions(self) -> List[int]:
        return [self.shape.pos0 + i for i in range(self.shape.steps)]


def _normal_bf16(g: torch.Generator, shape, std: float = 0.02) -> torch.Tensor:
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def _gain(g: torch.Generator, n: int, random_gains: bool) -> torch.Tensor:
    if random_gains:
        return (0.5 + torch.rand(n, generator=g, dtype=torch.float32)).to(torch.bfloat16)
    return torch.ones(n, dtype=torch.bfloat16)


def generate(shape: DecoderShape | str, seed: int = 0, random_gains: bool = False,
             steps: Optional[int] = None) -> Workload:
    """Draw the workload for `shape` (see the module docstring for the fixed order)."""
    if isinstance(shape, str):
        shape = SHAPES[shape]
    g = torch.Generator().manual_seed(seed)
    H, I, d = shape.hidden, shape.intermediate, shape.head_dim
    qd, kvd = shape.n_heads * d, shape.n_kv_heads * d
    embed = _normal_bf16(g, (shape.vocab, H))
    layers = []
    for _ in range(shape.n_layers):
        w: Dict[str, Optional[torch.Tensor]] = {}
        w["attn_norm"] = _gain(g, H, random_gains)
        w["wq"] = _normal_bf16(g, (qd, H))
        w["wk"] = _normal_bf16(g, (kvd, H))
        w["wv"] = _normal_bf16(g, (kvd, H))
        if shape.qkv_bias:
            w["bq"] = _normal_bf16(g, (qd,))
            w["bk"] = _normal_bf16(g, (kvd,))
            w["bv"] = _normal_bf16(g, (kvd,))
        else:
            w["bq"] = w["bk"] = w["bv"] = None
        w["wo"] = _normal_bf16(g, (H, qd))
        w["mlp_norm"] = _gain(g, H, random_gains)
        w["w_gate"] = _normal_bf16(g, (I, H))
        w["w_up"] = _normal_bf16(g, (I, H))
        w["w_down"] = _normal_bf16(g, (H, I))
        layers.append(w)
    final_norm = _gain(g, H, random_gains)
    n_steps = shape.steps if steps is None else steps
    tokens = torch.randint(0, shape.vocab, (shape.steps,), generator=g, dtype=torch.int64)[:n_steps]
    k_raw = v_raw = None
    if shape.prefill:
        k_raw = torch.randn((shape.n_layers, shape.n_kv_heads, shape.prefill, d), generator=g, dtype=torch.float32)
        v_raw = torch.randn((shape.n_layers, shape.n_kv_heads, shape.prefill, d), generator=g, dtype=torch.float32)
    if n_steps != shape.steps:
        shape = dataclasses.replace(shape, steps=n_steps)
    return Workload(shape, embed, final_norm, layers, tokens, k_raw, v_raw)


def scaled_down(shape: DecoderShape, **overrides) -> DecoderShape:
    """A copy of `shape` with some fields replaced (used for small edge-case decoders)."""
    return dataclasses.replace(shape, **overrides)
