"""Seeded synthetic inputs for the fused MoE layer.

This module is shared by the CUDA path's tests/benchmark and by the CPU oracle's
tests. It holds input generation only: no step of the MoE computation lives here.

Recipe (all configs):
  * numpy PCG64 streams, float32 standard normals. Three independent streams
    per seed: ``default_rng((seed, 0))`` draws hidden; ``default_rng((seed,
    1))`` draws router_w, w_gate_up, w_down in that order; ``default_rng((seed,
    2))`` draws the expert-rank permutation of the Zipf logit bias (skewed
    sweep only). The weights therefore do not depend on T: the decode,
    prefill and sweep workloads of one model shape share one layer.
  * Each tensor is scaled by its standard deviation in float32 and rounded
    once to bf16 (round to nearest, ties to even); both sides then read the
    same bf16 bit patterns, carried as ``uint16`` arrays.
  * Layouts follow the stacked-expert packing of the weight loader described
    on "模型与权重加载" (streaming loader, step 4): ``w_gate_up[E, 2I, H]`` with
    gate rows first, ``w_down[E, H, I]``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class MoEShape:
    name: str
    T: int
    H: int
    E: int
    top_k: int
    I: int
    renorm: bool
    w_std: float = 0.02
    router_std: Optional[float] = None  # defaults to w_std
    x_std: float = 1.0
    zipf_s: Optional[float] = None      # per-expert logit bias drawn for a Zipf load
    seed: int = 0

    def with_T(self, T: int) -> "MoEShape":
        return dataclasses.replace(self, T=T, name=f"{self.name}_T{T}")


# The workloads: a tiny parity case, the Qwen3-30B-A3B-shaped decode and
# prefill layers, the Qwen3-235B-A22B-shaped large prefill layer and the
# skewed-load sweep (one shape per T).
TINY = MoEShape("tiny", T=16, H=128, E=8, top_k=2, I=64, renorm=True)
DECODE = MoEShape("decode_qwen3_30b_a3b", T=64, H=2048, E=128, top_k=8, I=768, renorm=True)
PREFILL = MoEShape("prefill_qwen3_30b_a3b", T=4096, H=2048, E=128, top_k=8, I=768, renorm=True)
LARGE = MoEShape("prefill_qwen3_235b_a22b", T=8192, H=4096, E=128, top_k=8, I=1536,
                 renorm=True, w_std=0.015, router_std=0.015)
SWEEP_T = (1, 8, 32, 128, 512, 2048, 16384)
SWEEP = MoEShape("zipf_sweep", T=1, H=2048, E=128, top_k=8, I=768, renorm=False, zipf_s=1.1)
WORKLOADS = {s.name: s for s in (TINY, DECODE, PREFILL, LARGE)}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Input generation only (the values are finite normals)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
    return (b >> np.uint32(16)).astype(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape, std: float, chunk: int = 1 << 24) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        v = rng.standard_normal(m, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[s:s + m] = f32_to_bf16_bits(v)
    return out.reshape(shape)


def zipf_logit_bias(E: int, s: float, perm: np.ndarray) -> np.ndarray:
    """bias[e] = ln(q_rank(e)) with q_r proportional to r^-s over ranks 1..E.

    Expert e gets rank perm[e]+1. A logit bias of ln(q) multiplies that expert's
    unnormalised softmax mass by q, which skews the router's load towards a
    Zipf(s) profile (the top experts saturate at one row per token)."""
    r = np.arange(1, E + 1, dtype=np.float64)
    q = r ** (-s)
    q /= q.sum()
    return np.log(q[perm]).astype(np.float32)


def make_inputs(shape: MoEShape, weights: bool = True) -> dict:
    """Draw the inputs of one MoE layer call. Returns a dict of numpy arrays:
    hidden[T,H], router_w[E,H], w_gate_up[E,2I,H], w_down[E,H,I] (uint16 bf16
    bits) and router_bias[E] (float32, or None)."""
    d = {"hidden": make_hidden(shape)}
    d.update(make_weights(shape, experts=weights))
    d["router_bias"] = make_router_bias(shape)
    return d


def make_hidden(shape: MoEShape) -> np.ndarray:
    rng = np.random.default_rng((shape.seed, 0))
    return _normal_bf16(rng, (shape.T, shape.H), shape.x_std)


def make_weights(shape: MoEShape, experts: bool = True) -> dict:
    """router_w [E,H] and (if experts) w_gate_up [E,2I,H], w_down [E,H,I]."""
    rng = np.random.default_rng((shape.seed, 1))
    H, E, I = shape.H, shape.E, shape.I
    rstd = shape.router_std if shape.router_std is not None else shape.w_std
    d = {"router_w": _normal_bf16(rng, (E, H), rstd)}
    if experts:
        d["w_gate_up"] = _normal_bf16(rng, (E, 2 * I, H), shape.w_std)
        d["w_down"] = _normal_bf16(rng, (E, H, I), shape.w_std)
    return d


def make_router_bias(shape: MoEShape):
    if shape.zipf_s is None:
        return None
    perm = np.random.default_rng((shape.seed, 2)).permutation(shape.E)
    return zipf_logit_bias(shape.E, shape.zipf_s, perm)


def random_small_inputs(seed: int, T: int, H: int, E: int, I: int,
                        x_std: float = 1.0, w_std: float = 0.1,
                        bias: bool = False) -> dict:
    """Small random cases for property tests (same recipe, free shapes)."""
    rng = np.random.default_rng((seed, 3))
    d = {"hidden": _normal_bf16(rng, (T, H), x_std),
         "router_w": _normal_bf16(rng, (E, H), w_std),
         "w_gate_up": _normal_bf16(rng, (E, 2 * I, H), w_std),
         "w_down": _normal_bf16(rng, (E, H, I), w_std),
         "router_bias": None}
    if bias:
        d["router_bias"] = rng.standard_normal(E, dtype=np.float32)
    return d


def make_norm_inputs(seed: int, T: int, H: int, residual_std: float = 2.0) -> dict:
    """Inputs of the add + RMSNorm step before the layer (stream (seed, 4)):
    x (the attention output) ~ N(0, 1), residual ~ N(0, residual_std^2) and
    the norm weight 1 + N(0, 0.25^2), all rounded once to bf16."""
    rng = np.random.default_rng((seed, 4))
    return {"x": _normal_bf16(rng, (T, H), 1.0),
            "residual": _normal_bf16(rng, (T, H), residual_std),
            "norm_w": f32_to_bf16_bits(1.0 + 0.25 * rng.standard_normal(H, dtype=np.float32))}


def make_dense_weights(seed: int, H: int, I: int, std: float = 0.02) -> dict:
    """Weights of a dense gated MLP (stream (seed, 5)): w_gate_up [2I, H]
    (gate rows first) and w_down [H, I], N(0, std^2) rounded to bf16."""
    rng = np.random.default_rng((seed, 5))
    return {"w_gate_up": _normal_bf16(rng, (2 * I, H), std),
            "w_down": _normal_bf16(rng, (H, I), std)}
