"""Float64 CPU oracle for the decoder steps that follow the quantized projections.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute
this module: only ``tests/`` and ``__graft_entry__.smoke()`` use it.  It shares no
code with the CUDA library; both sides are fed the same seeded inputs.

Sources (TensorFold pull requests; quoted by page title and section):

* PR #1696 (LFM3 on Intel Iris Xe), "What it adds": "QK norm with partial RoPE",
  decode "fuses ... RoPE with the KV store", "the conv state and KV rings".
* PR #1514 (LFM3-1.7B on Apple Metal), "What changes": "post-add/next-norm fusion"
  keeps the retained rounding boundaries.

The pages name these steps but print no formula or constant.  Readings (the plain,
standard definitions; every constant is an argument, none is assumed):

* QK norm: RMS normalisation of each head vector separately,
      xhat_j = x_j / sqrt(mean_j(x_j^2) + eps) * w_j        (w: one bf16 weight per
  head dimension, shared by all heads of q, another for k).
* Partial RoPE, rotate-half form on the first rot_dim dimensions of a head (rot_dim
  even, <= head_dim; the rest pass through): for i < rot_dim / 2, with
      theta_i = pos * base^(-2 i / rot_dim),
      (a, b) = (x_i, x_{i + rot_dim/2})  ->  (a cos theta_i - b sin theta_i,
                                              a sin theta_i + b cos theta_i).
* KV store: the normed, rotated k and the plain v of stream r go to slot
  pos[r] mod ring_len of that stream's ring, rounded to bf16; the attention input q
  (normed and rotated) is rounded to bf16 as well.
* Post-add / next-norm: the residual stream is stored in bf16 (its retained rounding
  boundary): r' = bf16(r + y), then out = bf16(r' / sqrt(mean(r'^2) + eps) * gamma)
  computed from the stored r'.

Pinned by tests/test_post_oracle_pins.py (hand-computed values, closed forms,
invariants, planted mutants).
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(u16) -> np.ndarray:
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(a) -> np.ndarray:
    """Round-to-nearest-even float64 -> bf16 bit patterns (through float32, which is
    exact for the values involved up to the final rounding)."""
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def rms_norm_heads(x: np.ndarray, w: np.ndarray, head_dim: int, eps: float) -> np.ndarray:
    """RMS-normalise every head_dim-long head of each row of x (float64), times w."""
    rows, n = x.shape
    h = x.reshape(rows, n // head_dim, head_dim)
    ms = (h * h).mean(axis=2, keepdims=True)
    return (h / np.sqrt(ms + eps) * w.reshape(1, 1, head_dim)).reshape(rows, n)


def rope_partial(x: np.ndarray, pos: np.ndarray, head_dim: int, rot_dim: int, base: float) -> np.ndarray:
    """Rotate-half RoPE on the first rot_dim dimensions of every head (float64)."""
    rows, n = x.shape
    h = x.reshape(rows, n // head_dim, head_dim).copy()
    half = rot_dim // 2
    if half == 0:
        return h.reshape(rows, n)
    i = np.arange(half, dtype=np.float64)
    inv_freq = base ** (-2.0 * i / rot_dim)
    theta = np.asarray(pos, dtype=np.float64).reshape(rows, 1) * inv_freq.reshape(1, half)
    cos, sin = np.cos(theta)[:, None, :], np.sin(theta)[:, None, :]
    a = h[:, :, :half].copy()
    b = h[:, :, half:rot_dim].copy()
    h[:, :, :half] = a * cos - b * sin
    h[:, :, half:rot_dim] = a * sin + b * cos
    return h.reshape(rows, n)


def qk_norm_rope(q, k, v, q_w_bits, k_w_bits, pos, head_dim, rot_dim, base, eps):
    """q, k, v: float64 [rows, heads * head_dim] (the projection outputs).  Returns
    float64 (q_out, k_out, v_out) before the final bf16 rounding."""
    qw, kw = bf16_bits_to_f64(q_w_bits), bf16_bits_to_f64(k_w_bits)
    q_out = rope_partial(rms_norm_heads(np.asarray(q, np.float64), qw, head_dim, eps), pos, head_dim, rot_dim, base)
    k_out = rope_partial(rms_norm_heads(np.asarray(k, np.float64), kw, head_dim, eps), pos, head_dim, rot_dim, base)
    return q_out, k_out, np.asarray(v, np.float64)


def resid_rms_norm(r_bits, y, gamma_bits, eps):
    """Post-add / next-norm: returns (r' bf16 bits, normalised float64 before the final
    bf16 rounding).  r_bits: bf16 [rows, n]; y: float [rows, n]; gamma_bits: bf16 [n]."""
    r = bf16_bits_to_f64(r_bits) + np.asarray(y, np.float64)
    r_new = f64_to_bf16_bits(r)
    rn = bf16_bits_to_f64(r_new)
    ms = (rn * rn).mean(axis=1, keepdims=True)
    return r_new, rn / np.sqrt(ms + eps) * bf16_bits_to_f64(gamma_bits).reshape(1, -1)
