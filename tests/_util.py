"""Shared helpers of the GPU tests (test code only)."""
from __future__ import annotations

import numpy as np
import torch

from oracle import qlinear_oracle as orc
from weight_only_bit_mlx_gb300 import synth


def tol(A):
    """Acceptance bound per output: 1e-5 * sum|w x| + 1e-6."""
    return 1e-5 * np.asarray(A) + 1e-6


def assert_close(y_gpu, y64, A, what=""):
    y = y_gpu.detach().float().cpu().numpy().astype(np.float64) if isinstance(y_gpu, torch.Tensor) else y_gpu
    err = np.abs(y - y64)
    bound = tol(A)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outputs out of tolerance; worst at {i}: "
                             f"gpu {y[i]!r} oracle {y64[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")
    return float((err / bound).max()) if err.size else 0.0


def weight(n, k, bits, seed=0, config_id=0, tensor_id=0):
    return synth.make_weight(n, k, bits, seed=seed, config_id=config_id, tensor_id=tensor_id)


def dev_weight(w):
    from weight_only_bit_mlx_gb300.qlinear import QWeight
    return QWeight.from_numpy(w)


def dev_x(xbits):
    from weight_only_bit_mlx_gb300.qlinear import bf16_from_bits
    return bf16_from_bits(xbits)


def h_bound(a64, aa, c64, ac, h64):
    """Bound for bf16(silu(a) * c) given the per-output bounds of a and c."""
    ta, tc = tol(aa), tol(ac)
    return (1.1 * (np.abs(c64) + tc) * ta + (np.abs(orc.silu(a64)) + 1.1 * ta) * tc
            + 2.0 ** -8 * np.abs(h64) + 1e-6)


def pack_codes(q, bits):
    """Pack integer codes q[n, k] into uint32 rows, value j at bit offset bits*j of its
    row's little-endian stream (a field may straddle two words).  Test-side packer,
    vectorised over rows; independent of the oracle's unpacker."""
    q = np.asarray(q, dtype=np.uint64)
    n, k = q.shape
    nw = k * bits // 32
    per = 32 // int(np.gcd(32, bits))        # codes per period of whole words
    wper = per * bits // 32                  # words per period
    words = np.zeros((n, nw + 1), dtype=np.uint64)
    for j in range(per):
        pos = bits * j
        w, off = pos // 32, pos % 32
        v = q[:, j::per] << np.uint64(off)
        words[:, w:nw:wper] |= v & np.uint64(0xFFFFFFFF)
        words[:, w + 1:nw + 1:wper] |= v >> np.uint64(32)
    return words[:, :nw].astype(np.uint32)
