"""Seeded synthetic inputs for the MoE layer.

This module only draws random numbers and rounds them to the storage type; it
holds none of the layer's arithmetic, so both the CUDA path's tests/bench and
the float64 oracle can consume it without sharing any method code.

Recipe (one PCG64 stream per tensor, float32 draws):
  x ~ N(0, 1)                      seed 0
  W_r ~ N(0, 1/d_model)            seed 1
  W_gate, W_up ~ N(0, 1/d_model)   seeds 2, 3
  W_down ~ N(0, 1/d_hidden)        seed 4
  shared gate/up ~ N(0, 1/d_model), shared down ~ N(0, 1/shared_hidden)  seeds 5, 6, 7
  G (upstream gradient) ~ N(0, 1)  seed 8
Router weights are i.i.d. with no expert bias (routing skew 0), which is the
uniform-routing setting of the benchmark pages' layer suites.  For bfloat16
configurations every tensor is rounded to bfloat16 (round to nearest even)
and the rounded values are what both sides receive.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class MoEConfig:
    tokens: int
    d_model: int = 512
    d_hidden: int = 1024
    experts: int = 8
    top_k: int = 2
    shared_hidden: int = 0
    dtype: str = "bf16"          # "bf16" or "f32"
    name: str = field(default="", compare=False)
    capacity: int = 0            # pairs per expert; 0 = dropless
    skew: float = 0.0            # router bias ramp (0 = no bias: uniform routing)

    @property
    def pairs(self) -> int:
        return self.tokens * self.top_k


# The workloads of the benchmark pages (E8/k2 layer suite at three token
# counts, the fine-grained E64/k4 layer and the E64/k8 decoder block with a
# shared expert), by name.
CONFIGS = {
    "e8k2_f32_4k": MoEConfig(4096, 512, 1024, 8, 2, 0, "f32", "e8k2_f32_4k"),
    "e8k2_bf16_32k": MoEConfig(32768, 512, 1024, 8, 2, 0, "bf16", "e8k2_bf16_32k"),
    "e8k2_f32_128k": MoEConfig(131072, 512, 1024, 8, 2, 0, "f32", "e8k2_f32_128k"),
    "e8k2_bf16_128k": MoEConfig(131072, 512, 1024, 8, 2, 0, "bf16", "e8k2_bf16_128k"),
    "e64k4_bf16_32k": MoEConfig(32768, 512, 256, 64, 4, 0, "bf16", "e64k4_bf16_32k"),
    "decoder_bf16_16k": MoEConfig(16384, 512, 128, 64, 8, 1024, "bf16", "decoder_bf16_16k"),
    "decoder_bf16_128k": MoEConfig(131072, 512, 128, 64, 8, 1024, "bf16", "decoder_bf16_128k"),
}


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns
    float32 holding exactly representable bfloat16 values."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bfloat16-exact."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _normal(seed: int, shape, std: float) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(seed))
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def make_inputs(cfg: MoEConfig, seed_offset: int = 0, with_upstream: bool = True) -> dict:
    """All tensors of one layer invocation as float32 numpy arrays (bfloat16
    exact when cfg.dtype == "bf16").  Keys: x, w_router, w_gate, w_up, w_down,
    ws_gate, ws_up, ws_down (None without a shared expert), upstream, and
    router_bias: None at skew 0, else the float32 ramp
    b_e = skew * 4 * (E - 1 - 2e) / (E - 1), +4 skew logit standard deviations
    on expert 0 down to -4 skew on expert E-1 (the logits x W_r have unit
    variance here), which skews the routing towards the low experts."""
    T, d, h, E, hs = cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.shared_hidden
    s = seed_offset
    out = {
        "x": _normal(s + 0, (T, d), 1.0),
        "w_router": _normal(s + 1, (d, E), d ** -0.5),
        "w_gate": _normal(s + 2, (E, d, h), d ** -0.5),
        "w_up": _normal(s + 3, (E, d, h), d ** -0.5),
        "w_down": _normal(s + 4, (E, h, d), h ** -0.5),
        "ws_gate": None, "ws_up": None, "ws_down": None,
        "upstream": _normal(s + 8, (T, d), 1.0) if with_upstream else None,
    }
    if hs > 0:
        out["ws_gate"] = _normal(s + 5, (d, hs), d ** -0.5)
        out["ws_up"] = _normal(s + 6, (d, hs), d ** -0.5)
        out["ws_down"] = _normal(s + 7, (hs, d), hs ** -0.5)
    if cfg.dtype == "bf16":
        for k, v in list(out.items()):
            if v is not None:
                out[k] = bf16_round(v)
    out["router_bias"] = None
    if cfg.skew and E > 1:
        ramp = (E - 1 - 2 * np.arange(E, dtype=np.float64)) / (E - 1)
        out["router_bias"] = (cfg.skew * 4.0 * ramp).astype(np.float32)
    return out


def params_of(inputs: dict) -> dict:
    """The parameter subset of ``make_inputs``'s result."""
    keys = ("w_router", "w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down", "router_bias")
    return {k: inputs[k] for k in keys}
