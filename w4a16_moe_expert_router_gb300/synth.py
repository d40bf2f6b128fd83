"""Seeded synthetic inputs for the W4A16 MoE expert layer.

This module only draws random numbers with stated distributions and shapes; it
holds none of the layer's arithmetic (no unpacking, dequantisation, routing or
matrix products), so both the CPU oracle and the GPU library can be fed from it.

Workloads.  The 256-token canvas, 128 experts and top-8 routing are the model
card's ("srswti/axe-diffusion-ksl-xe", "what the model is"); 64 tokens is the
smallest canvas of the block-diffusion loop ("mlxcel block-diffusion" docs); the
expert width f=704 is the down_proj contraction dim the model card states under
"requirements".  The hidden size d=2048 is not printed on the pages and is this
library's choice for the synthetic layer.

  tiny        T=16,   d=256,  f=128, E=8,   k=2, groups 64/64
  canvas64    T=64,   d=2048, f=704, E=128, k=8, groups 64/64
  canvas256   T=256,  d=2048, f=704, E=128, k=8, groups 64/64
  stack30     30 layers of canvas256, each followed by an fp32 RMSNorm, gamma ~ N(1, 0.1)
  zipf1024    T=1024, d=2048, f=704, E=128, k=8, groups 128/64, logits biased by
              -1.1*ln(e+1) per expert (log of a Zipf(s=1.1) weight) to skew the load

Distributions: packed weight bytes uniform over 0..255 (two independent uniform
nibbles); scale fp16(U(0.005, 0.02)); zero-point fp16(U(6, 9)); x fp16(N(0,1));
router logits fp32 N(0,1); for the MoE block around the layer, router weights
fp16(N(0, 1/d)) and a pre-norm weight N(1, 0.1).  Every tensor draws from its own stream, derived from
(seed, layer, tensor number) in a fixed order, so any tensor can be regenerated
alone.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    tokens: int
    hidden: int
    inter: int
    experts: int
    top_k: int
    group_gate_up: int
    group_down: int
    layers: int = 1
    zipf_s: float = 0.0        # 0 = unbiased N(0,1) logits
    rmsnorm: bool = False      # fp32 RMSNorm after every layer (gamma ~ N(1, 0.1))
    activation: int = 0        # 0 = GELU tanh form, 1 = GELU erf form
    reduction: int = 0         # 0 = each weight dequantised, 1 = group-factorised expert GEMMs
    format: int = 0            # 0 = asymmetric zero-point, 1 = affine bias (MLX), 2 = symmetric (GPTQ)

    def weight_bytes_per_expert(self) -> int:
        """Packed nibbles plus fp16 scale and zero of both projections."""
        d, f, g1, g2 = self.hidden, self.inter, self.group_gate_up, self.group_down
        return 2 * f * d // 2 + 2 * f * (d // g1) * 4 + d * f // 2 + d * (f // g2) * 4


WORKLOADS = {
    "tiny": Workload("tiny", 16, 256, 128, 8, 2, 64, 64),
    "canvas64": Workload("canvas64", 64, 2048, 704, 128, 8, 64, 64),
    "canvas256": Workload("canvas256", 256, 2048, 704, 128, 8, 64, 64),
    "stack30": Workload("stack30", 256, 2048, 704, 128, 8, 64, 64, layers=30, rmsnorm=True),
    "zipf1024": Workload("zipf1024", 1024, 2048, 704, 128, 8, 128, 64, zipf_s=1.1),
}

# tensor numbers of the derived streams (fixed order)
_X, _LOGITS, _GUQ, _GUS, _GUZ, _DQ, _DS, _DZ, _GAMMA, _ROUTER, _GAMMA_PRE = range(11)


def _rng(seed: int, layer: int, tensor: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, layer, tensor]))


def _half_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a.astype(np.float16)).view(np.uint16)


def make_x(w: Workload, seed: int = 0, tokens: int | None = None) -> np.ndarray:
    """Activations, fp16 bit patterns [T][d]."""
    T = w.tokens if tokens is None else tokens
    return _half_bits(_rng(seed, 0, _X).standard_normal((T, w.hidden), dtype=np.float32))


def make_logits(w: Workload, seed: int = 0, layer: int = 0, tokens: int | None = None) -> np.ndarray:
    """Router logits fp32 [T][E]; N(0,1), plus -s*ln(e+1) when the workload is Zipf-skewed."""
    T = w.tokens if tokens is None else tokens
    lg = _rng(seed, layer, _LOGITS).standard_normal((T, w.experts), dtype=np.float32)
    if w.zipf_s:
        lg = (lg + (-w.zipf_s * np.log(np.arange(1, w.experts + 1, dtype=np.float64))).astype(np.float32)[None, :])
    return np.ascontiguousarray(lg, dtype=np.float32)


def make_weights(w: Workload, seed: int = 0, layer: int = 0) -> dict:
    """Canonical quantised weights of one layer (all experts).

    gate_up_q [E][2f][d/2] u8, gate_up_scale/zero [E][2f][d/g1] fp16 bits,
    down_q [E][d][f/2] u8, down_scale/zero [E][d][f/g2] fp16 bits.
    """
    E, d, f, g1, g2 = w.experts, w.hidden, w.inter, w.group_gate_up, w.group_down
    gus = _half_bits(_rng(seed, layer, _GUS).uniform(0.005, 0.02, (E, 2 * f, d // g1)))
    ds = _half_bits(_rng(seed, layer, _DS).uniform(0.005, 0.02, (E, d, f // g2)))
    return {
        "gate_up_q": _rng(seed, layer, _GUQ).integers(0, 256, (E, 2 * f, d // 2), dtype=np.uint8),
        "gate_up_scale": gus,
        "gate_up_zero": _second(w, _rng(seed, layer, _GUZ).uniform(6.0, 9.0, (E, 2 * f, d // g1)), gus),
        "down_q": _rng(seed, layer, _DQ).integers(0, 256, (E, d, f // 2), dtype=np.uint8),
        "down_scale": ds,
        "down_zero": _second(w, _rng(seed, layer, _DZ).uniform(6.0, 9.0, (E, d, f // g2)), ds),
    }


def _second(w: Workload, z: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """The per-group value stored beside the scale: the zero-point z (format 0), the
    affine bias b = fp16(-z * s) of the same dequantised range (format 1), or 8 (format 2,
    where it is not read)."""
    if w.format == 1:
        return _half_bits(-z * scale_bits.view(np.float16).astype(np.float64))
    if w.format == 2:
        return np.full(z.shape, 0x4800, np.uint16)
    return _half_bits(z)


def make_gamma(w: Workload, seed: int = 0, layer: int = 0) -> np.ndarray:
    """RMSNorm weight fp32 [d] ~ N(1, 0.1)."""
    return np.ascontiguousarray(1.0 + 0.1 * _rng(seed, layer, _GAMMA).standard_normal(w.hidden), dtype=np.float32)


def make_router(w: Workload, seed: int = 0, layer: int = 0) -> np.ndarray:
    """Router weights of the MoE block, fp16 bit patterns [E][d] ~ fp16(N(0, 1/d)), so
    that logits of a normalised input are ~N(0, 1) like the layer's own synthetic logits."""
    a = _rng(seed, layer, _ROUTER).standard_normal((w.experts, w.hidden)) / np.sqrt(w.hidden)
    return _half_bits(a)


def make_gamma_pre(w: Workload, seed: int = 0, layer: int = 0) -> np.ndarray:
    """Pre-norm weight of the MoE block, fp32 [d] ~ N(1, 0.1)."""
    return np.ascontiguousarray(1.0 + 0.1 * _rng(seed, layer, _GAMMA_PRE).standard_normal(w.hidden), dtype=np.float32)
