"""Float64 CPU oracle for MLX-style affine weight-only quantized linear layers.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or execute
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the CUDA
library (no kernels, headers, helpers or tables); both sides are fed the same seeded
inputs as raw bit patterns.

What it computes is the plain definition of the operation, written out in float64:

    w[n, k]  = scale[n, k // 64] * q[n, k] + bias[n, k // 64]
    y[r, n]  = sum_k w[n, k] * x[r, k]
    A[r, n]  = sum_k |w[n, k] * x[r, k]|      (scale of the acceptance bound)

Sources (TensorFold pull requests; quoted by page title and section):

* PR #1696 (LFM3 on Intel Iris Xe), "What it adds": weights are loaded as MLX 4-bit,
  group 64, "as stored" and dequantized inside the kernels; decode fuses w1 + w3 +
  SwiGLU and the four attention matvecs; the prompt GEMM sums each output as an fma
  chain per 64-wide k block and adds the blocks in order.  Summation order changes
  rounding only, so the exact value that every order approximates is the plain
  sum above; the order itself is checked GPU-against-GPU, not here.
* PR #1514 (LFM3-1.7B on Apple Metal), "What changes": MLX 4/6/8-bit checkpoints;
  paired FFN projections keep their retained rounding boundaries (the SwiGLU output
  is stored in bf16 before the down projection).
* PR #1696, "What it adds": a numpy float64 reference is the precedent for checking
  each kernel.

Readings where the pages are silent (the pages print no formula or bit layout):

* W is [n, k] with k contiguous; each row is a little-endian bit stream stored in
  uint32 words, value k occupying bits [bits*k, bits*k + bits) of its row.  For 4 and
  8 bits this is "field (k mod 32/bits) of word k // (32/bits), lowest field first";
  for 6 bits a field may straddle two words.
* dequantization is w = scale * q + bias with unsigned q; scale and bias are bf16
  per (row, 64-wide group along k).
* silu(t) = t / (1 + exp(-t)).

Pinned by tests/test_oracle_pins.py (brute force in exact rationals, hand-packed
fixtures under tests/golden/, closed forms and invariants).
"""
from __future__ import annotations

import numpy as np

GROUP = 64


def bf16_bits_to_f64(u16) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def unpack_q(wq, bits: int, k: int) -> np.ndarray:
    """Integer codes q[n, k] (int64) from packed rows of uint32 words.

    Value j of a row sits at bit offset bits*j of the row's little-endian stream.
    """
    wq = np.asarray(wq, dtype=np.uint32)
    n, nwords = wq.shape
    if nwords * 32 != k * bits:
        raise ValueError(f"row has {nwords} words, expected {k * bits // 32}")
    pos = bits * np.arange(k, dtype=np.int64)
    word = pos // 32
    off = (pos % 32).astype(np.uint64)
    nxt = np.minimum(word + 1, nwords - 1)
    lo = wq[:, word].astype(np.uint64)
    hi = wq[:, nxt].astype(np.uint64)
    # a field that runs past its word continues in the low bits of the next word
    straddle = (off + bits) > 32
    hi = np.where(straddle[None, :], hi, np.uint64(0))
    both = lo | (hi << np.uint64(32))
    return ((both >> off[None, :]) & np.uint64((1 << bits) - 1)).astype(np.int64)


def dequant(wq, scales, biases, bits: int, k: int) -> np.ndarray:
    """w[n, k] = scale[n, k//64] * q[n, k] + bias[n, k//64] in float64."""
    q = unpack_q(wq, bits, k).astype(np.float64)
    s = bf16_bits_to_f64(scales)
    b = bf16_bits_to_f64(biases)
    gidx = np.arange(k) // GROUP
    return s[:, gidx] * q + b[:, gidx]


def qlinear(x_bits, wq, scales, biases, bits: int):
    """y64[r, n] = sum_k w[n, k] x[r, k] and A[r, n] = sum_k |w[n, k] x[r, k]|.

    ``x_bits`` is bf16 bits [rows, k]; the weight arrays are as stored.
    """
    x = bf16_bits_to_f64(np.atleast_2d(x_bits))
    k = x.shape[1]
    w = dequant(wq, scales, biases, bits, k)
    return x @ w.T, np.abs(x) @ np.abs(w).T


def qlinear_w(x_bits, weight: dict):
    """``qlinear`` on a weight dict with keys wq, scales, biases, bits."""
    return qlinear(x_bits, weight["wq"], weight["scales"], weight["biases"], weight["bits"])


def silu(t):
    """silu(t) = t / (1 + exp(-t)) in float64."""
    t = np.asarray(t, dtype=np.float64)
    with np.errstate(over="ignore"):
        return t / (1.0 + np.exp(-t))


def ffn_swiglu(x_bits, w1: dict, w3: dict):
    """Fused FFN gate/up stage: a = w1 x, c = w3 x, h = silu(a) * c (all float64).

    Returns (a64, A_a, c64, A_c, h64).
    """
    a, aa = qlinear_w(x_bits, w1)
    c, ac = qlinear_w(x_bits, w3)
    return a, aa, c, ac, silu(a) * c


def pgemm(X_bits, weight: dict):
    """Prompt-window GEMM: the same linear map applied to every row of X."""
    return qlinear_w(X_bits, weight)
