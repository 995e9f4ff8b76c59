"""Pins of the float64 oracle of the post-projection decoder steps (CPU only):
QK norm with partial RoPE and the KV store (TensorFold PR #1696, "What it adds"), and
the post-add / next-norm step (PR #1514, "What changes").  The pages print no formula,
so the pins check the readings stated in oracle/decoder_post_oracle.py against hand-
computed values, closed forms and invariants, and planted mistakes must fail them.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

from oracle import decoder_post_oracle as po


def bf16_bits(values) -> np.ndarray:
    """Test-side bf16 encoding of values that are exactly representable."""
    f = np.asarray(values, dtype=np.float32)
    u = f.view(np.uint32)
    assert ((u & 0xFFFF) == 0).all(), "test value not exact in bf16"
    return (u >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------------- pins
def pin_rms_norm(mod):
    # hand value: head (3, 4), w = 1, eps = 0 -> x / sqrt(12.5)
    got = mod.rms_norm_heads(np.array([[3.0, 4.0]]), np.array([1.0, 1.0]), 2, 0.0)
    assert np.allclose(got, [[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]], rtol=1e-15)
    # closed form: a constant head c gives sign(c) * w / sqrt(1 + eps / c^2)
    c, eps = -2.5, 0.25
    got = mod.rms_norm_heads(np.full((1, 4), c), np.array([1.0, 2.0, 0.5, 3.0]), 4, eps)
    assert np.allclose(got, -np.array([1.0, 2.0, 0.5, 3.0]) / math.sqrt(1 + eps / c ** 2), rtol=1e-14)
    # heads are normalised separately
    x = np.array([[1.0, 1.0, 100.0, 100.0]])
    got = mod.rms_norm_heads(x, np.ones(2), 2, 0.0)
    assert np.allclose(got, [[1, 1, 1, 1]], rtol=1e-14)


def pin_rope(mod):
    # sign convention: (1, 0) -> (cos 1, sin 1); (0, 1) -> (-sin 1, cos 1)
    got = mod.rope_partial(np.array([[1.0, 0.0], [0.0, 1.0]]), np.array([1, 1]), 2, 2, 10000.0)
    assert np.allclose(got, [[math.cos(1), math.sin(1)], [-math.sin(1), math.cos(1)]], rtol=0, atol=1e-15)
    # frequencies: head 4, rot 4, base 10000, pos 100 -> pair 1 turns by 100 * 10000^(-1/2) = 1 rad
    got = mod.rope_partial(np.array([[0.0, 1.0, 0.0, 0.0]]), np.array([100]), 4, 4, 10000.0)
    assert np.allclose(got, [[0.0, math.cos(1), 0.0, math.sin(1)]], rtol=0, atol=1e-13)
    # pair 0 turns by pos radians
    got = mod.rope_partial(np.array([[1.0, 0.0, 0.0, 0.0]]), np.array([3]), 4, 4, 10000.0)
    assert np.allclose(got, [[math.cos(3), 0.0, math.sin(3), 0.0]], rtol=0, atol=1e-15)
    # partial: dimensions past rot_dim pass through; position 0 and rot_dim 0 are the identity
    x = np.arange(1.0, 13.0).reshape(1, 12)
    got = mod.rope_partial(x, np.array([7]), 6, 4, 500.0)
    assert np.array_equal(got[:, [4, 5, 10, 11]], x[:, [4, 5, 10, 11]])
    assert np.array_equal(mod.rope_partial(x, np.array([0]), 6, 4, 500.0), x)
    assert np.array_equal(mod.rope_partial(x, np.array([7]), 6, 0, 500.0), x)
    # rotations compose: pos a then pos b equals pos a + b; each pair keeps its length
    r = np.random.default_rng(0).normal(size=(1, 16))
    a = mod.rope_partial(mod.rope_partial(r, np.array([5]), 16, 12, 1e4), np.array([9]), 16, 12, 1e4)
    assert np.allclose(a, mod.rope_partial(r, np.array([14]), 16, 12, 1e4), rtol=0, atol=1e-12)
    b = mod.rope_partial(r, np.array([123]), 16, 12, 1e4)
    assert np.allclose(r[0, :6] ** 2 + r[0, 6:12] ** 2, b[0, :6] ** 2 + b[0, 6:12] ** 2, rtol=1e-12)


def pin_qk_norm_rope(mod):
    # norm first, then rotation (the order matters with a non-uniform weight):
    # head (1, 0), w = (2, 1), eps 0, pos 1 -> (2 sqrt2 cos 1, 2 sqrt2 sin 1)
    w = bf16_bits([2.0, 1.0])
    q, k, v = mod.qk_norm_rope(np.array([[1.0, 0.0]]), np.array([[1.0, 0.0]]), np.array([[5.0, 6.0]]), w, w,
                               np.array([1]), 2, 2, 10000.0, 0.0)
    want = [[2 * math.sqrt(2) * math.cos(1), 2 * math.sqrt(2) * math.sin(1)]]
    assert np.allclose(q, want, rtol=1e-14) and np.allclose(k, want, rtol=1e-14)
    assert np.array_equal(v, [[5.0, 6.0]])


def pin_resid_norm(mod):
    # r + y exact in bf16: 1.0 + 0.5 = 1.5; one element -> out = gamma (eps 0)
    rb, out = mod.resid_rms_norm(bf16_bits([[1.0]]), np.array([[0.5]]), bf16_bits([3.0]), 0.0)
    assert rb[0, 0] == bf16_bits([1.5])[0] and np.allclose(out, [[3.0]], rtol=1e-15)
    # the stored residual is rounded to bf16 before the norm reads it: 1 + 2^-9 -> 1.0
    rb, out = mod.resid_rms_norm(bf16_bits([[1.0, 1.0]]), np.array([[2.0 ** -9, 0.0]]), bf16_bits([1.0, 1.0]),
                                 0.0)
    assert (rb == bf16_bits([1.0, 1.0])).all() and np.allclose(out, [[1.0, 1.0]], rtol=1e-15)
    # round to nearest even: 1 + 2^-8 is a tie -> 1.0; 1 + 3 * 2^-8 -> 1 + 2^-6 (0x3F82)
    assert po.f64_to_bf16_bits([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]).tolist() == [0x3F80, 0x3F82]


PINS = [pin_rms_norm, pin_rope, pin_qk_norm_rope, pin_resid_norm]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(po)


# ----------------------------------------------------------------------- planted mistakes
class _Mutant:
    def __init__(self, **over):
        # module functions, except qk_norm_rope, which the class composes from them
        self.__dict__.update({n: getattr(po, n) for n in dir(po) if not n.startswith("_") and n != "qk_norm_rope"})
        self.__dict__.update(over)

    def qk_norm_rope(self, q, k, v, qw, kw, pos, hd, rot, base, eps):
        qwf, kwf = po.bf16_bits_to_f64(qw), po.bf16_bits_to_f64(kw)
        if self.__dict__.get("rope_first"):
            return (self.rms_norm_heads(self.rope_partial(q, pos, hd, rot, base), qwf, hd, eps),
                    self.rms_norm_heads(self.rope_partial(k, pos, hd, rot, base), kwf, hd, eps), v)
        return (self.rope_partial(self.rms_norm_heads(q, qwf, hd, eps), pos, hd, rot, base),
                self.rope_partial(self.rms_norm_heads(k, kwf, hd, eps), pos, hd, rot, base), v)


def _rope_sign(x, pos, hd, rot, base):
    return po.rope_partial(x, -np.asarray(pos), hd, rot, base)


def _rope_freq(x, pos, hd, rot, base):
    return po.rope_partial(x, pos, hd, rot, base ** 0.5)


def _norm_whole_row(x, w, hd, eps):
    ms = (x * x).mean(axis=1, keepdims=True)
    rows, n = x.shape
    return ((x / np.sqrt(ms + eps)).reshape(rows, n // hd, hd) * w.reshape(1, 1, hd)).reshape(rows, n)


def _resid_no_round(r_bits, y, g_bits, eps):
    r = po.bf16_bits_to_f64(r_bits) + np.asarray(y, np.float64)
    ms = (r * r).mean(axis=1, keepdims=True)
    return po.f64_to_bf16_bits(r), r / np.sqrt(ms + eps) * po.bf16_bits_to_f64(g_bits).reshape(1, -1)


MUTANTS = {
    "rope_sign": _Mutant(rope_partial=_rope_sign),
    "rope_frequency": _Mutant(rope_partial=_rope_freq),
    "norm_whole_row": _Mutant(rms_norm_heads=_norm_whole_row),
    "rope_before_norm": _Mutant(rope_first=True),
    "residual_not_rounded": _Mutant(resid_rms_norm=_resid_no_round),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mutant(name):
    failures = 0
    for pin in PINS:
        try:
            pin(MUTANTS[name])
        except AssertionError:
            failures += 1
    assert failures >= 1, f"mutant {name} passed every pin"
