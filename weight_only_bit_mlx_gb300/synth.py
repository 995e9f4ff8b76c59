"""Seeded synthetic inputs for the weight-only quantized linear path.

This module only draws random numbers; it holds none of the method's arithmetic
(no unpacking, dequantization or dot products), so both the CUDA path and the
float64 oracle can be fed from it without sharing any computation.

Recipe (shapes and value ranges of the MLX affine 4/6/8-bit, group-64 workloads):

* generator: numpy PCG64, ``default_rng([seed, config_id, tensor_id])``;
* a weight tensor draws, in this order, its packed words, its scales, its biases;
* packed words are uniform uint32.  Every b-bit field of a uniform word stream is
  uniform on {0 .. 2^b - 1}, so this is exactly q ~ U{0..2^b-1} for 4, 6 and 8 bits
  without any packing code here;
* scale ~ U(0.005, 0.02) and bias ~ U(-0.1, 0.1), drawn in float64, cast to float32,
  then rounded to bfloat16 with round-to-nearest-even;
* activations x ~ N(0, 1) with the same float32 -> bfloat16 rounding, drawn last
  from their own generator.

bfloat16 values are carried as their raw uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np

GROUP = 64


def rng_for(seed: int, config_id: int, tensor_id: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(config_id), int(tensor_id)])


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def words_per_row(k: int, bits: int) -> int:
    if k % GROUP:
        raise ValueError("k must be a multiple of 64")
    return k * bits // 32


def make_weight(n: int, k: int, bits: int, seed: int = 0, config_id: int = 0,
                tensor_id: int = 0) -> dict:
    """Random packed weight: ``wq`` uint32 [n, k*bits/32], ``scales``/``biases`` bf16 bits [n, k/64]."""
    g = rng_for(seed, config_id, tensor_id)
    wq = g.integers(0, 2**32, size=(n, words_per_row(k, bits)), dtype=np.uint64).astype(np.uint32)
    scales = f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(n, k // GROUP)))
    biases = f32_to_bf16_bits(g.uniform(-0.1, 0.1, size=(n, k // GROUP)))
    return {"wq": wq, "scales": scales, "biases": biases, "n": n, "k": k, "bits": bits}


def make_x(rows: int, k: int, seed: int = 0, config_id: int = 0, tensor_id: int = 1000) -> np.ndarray:
    """Random activations as bf16 bits [rows, k], x ~ N(0, 1)."""
    g = rng_for(seed, config_id, tensor_id)
    return f32_to_bf16_bits(g.standard_normal(size=(rows, k)))


# Inputs of the steps after the projections (QK norm + partial RoPE + KV store, and
# post-add / next-norm).  Recipe: projection outputs (q, k, v, y) ~ N(0, sigma^2) in
# float32; norm weights ~ U(0.5, 1.5) rounded to bf16; the residual stream ~ N(0, 1)
# rounded to bf16; positions uniform on {lo .. hi-1} as int32.
def make_f32(rows: int, n: int, sigma: float = 1.0, seed: int = 0, config_id: int = 0,
             tensor_id: int = 2000) -> np.ndarray:
    g = rng_for(seed, config_id, tensor_id)
    return (sigma * g.standard_normal(size=(rows, n))).astype(np.float32)


def make_bf16(shape, lo: float | None = None, hi: float | None = None, seed: int = 0, config_id: int = 0,
              tensor_id: int = 3000) -> np.ndarray:
    """bf16 bits: U(lo, hi) when both are given, else N(0, 1)."""
    g = rng_for(seed, config_id, tensor_id)
    a = g.uniform(lo, hi, size=shape) if lo is not None else g.standard_normal(size=shape)
    return f32_to_bf16_bits(a)


def make_pos(rows: int, lo: int, hi: int, seed: int = 0, config_id: int = 0, tensor_id: int = 4000) -> np.ndarray:
    g = rng_for(seed, config_id, tensor_id)
    return g.integers(lo, hi, size=rows).astype(np.int32)
