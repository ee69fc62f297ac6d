"""Seeded synthetic inputs for the ternary linear layer.

This module only draws random numbers; it holds none of the layer's
arithmetic.  The same host arrays feed the CUDA library and the CPU oracle.

Distributions (stand-ins for the real model weights and activations of a
27B ternary hybrid model, which are not available):
* codes: i.i.d. uniform over {-1, 0, +1} (int8);
* scales: fp16_rn(0.02 * |N(0,1)| + 1e-3), one per 128 elements of a row;
* activations: bf16_rn(N(0,1)); a fixed, seeded set of round(frac * K)
  channels (the same for every token) is multiplied by an outlier factor.
Each of codes, scales and activations draws from its own PCG64 stream
spawned from the seed, so changing one shape does not change the others.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

GROUP = 128


def _streams(seed: int):
    ss = np.random.SeedSequence(seed)
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(4)]


def make_codes(seed: int, n: int, k: int) -> np.ndarray:
    rng = _streams(seed)[0]
    return (rng.integers(0, 3, size=(n, k), dtype=np.int8) - 1).astype(np.int8)


def make_scales(seed: int, n: int, k: int) -> np.ndarray:
    rng = _streams(seed)[1]
    g = k // GROUP
    s = 0.02 * np.abs(rng.standard_normal((n, g))) + 1e-3
    return s.astype(np.float16)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even) bit patterns, via torch's CPU cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def make_activations(seed: int, m: int, k: int, outlier_frac: float,
                     outlier_mult: float):
    """Returns (bf16 bit patterns uint16 [M,K], the same values as fp32)."""
    st = _streams(seed)
    n_out = int(round(outlier_frac * k))
    chans = np.sort(st[2].choice(k, size=n_out, replace=False)) if n_out else \
        np.zeros(0, dtype=np.int64)
    x = st[3].standard_normal((m, k)).astype(np.float32)
    if n_out:
        x[:, chans] *= np.float32(outlier_mult)
    bits = to_bf16_bits(x)
    return bits, bf16_bits_to_f32(bits)


@dataclass(frozen=True)
class Layer:
    name: str
    k: int
    n: int
    outlier_frac: float
    outlier_mult: float


# Shapes of the workloads (a 27B ternary hybrid model's linear layers).
TINY = Layer("tiny 1024->256", 1024, 256, 0.01, 20.0)
GATE_UP = Layer("gate/up 5120->34816", 5120, 34816, 0.001, 50.0)
DOWN = Layer("down 17408->5120", 17408, 5120, 0.001, 50.0)
QKV = Layer("qkv 5120->10240", 5120, 10240, 0.001, 50.0)
O_PROJ = Layer("o 5120->5120", 5120, 5120, 0.001, 50.0)
STACK_LAYERS = (QKV, O_PROJ, GATE_UP, DOWN)


@dataclass
class LayerData:
    layer: Layer
    codes: np.ndarray       # int8 [N,K]
    scales: np.ndarray      # fp16 [N,G]
    x_bits: np.ndarray      # uint16 bf16 bits [M,K]
    x: np.ndarray           # fp32 copy of the bf16 values [M,K]


def make_layer(layer: Layer, m: int, seed: int = 0, n: int | None = None) -> LayerData:
    """Seeded inputs of one layer; ``n`` overrides the row count (for samples)."""
    nn = layer.n if n is None else n
    codes = make_codes(seed, nn, layer.k)
    scales = make_scales(seed, nn, layer.k)
    xb, xf = make_activations(seed, m, layer.k, layer.outlier_frac, layer.outlier_mult)
    return LayerData(layer, codes, scales, xb, xf)
