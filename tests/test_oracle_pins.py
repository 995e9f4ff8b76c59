"""Pins of the float64 oracle against things other than itself (CPU only).

* hand-packed fixtures with hand-derived values (tests/golden/hand_packed.txt);
* brute force in exact rationals (fractions.Fraction) on tiny shapes, from integer
  codes packed by this file's own packer, never by the oracle;
* closed forms (x = 1, q = 0, one-hot x) and invariants (linearity over disjoint
  supports, permuting whole groups, a row alone equal to the row in a batch);
* silu values and the SwiGLU composition;
* planted mistakes: each mutant oracle (wrong field order, dropped bias, wrong group
  index, transposed weight, sign error, no straddle) must fail at least one pin.

The layout reading being pinned: a weight row is a little-endian bit stream of
uint32 words with value k at bits [bits*k, bits*k + bits); w = scale*q + bias per
64-wide group along k (TensorFold PR #1696, "What it adds": MLX 4-bit group 64 as
stored; PR #1514, "What changes": MLX 4/6/8-bit).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import qlinear_oracle as orc
from weight_only_bit_mlx_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_packed.txt")


# --------------------------------------------------------------------------------------
# test-side helpers (independent of the oracle)
# --------------------------------------------------------------------------------------
def pack_rows(q: np.ndarray, bits: int) -> np.ndarray:
    """Pack integer codes q[n, k] into uint32 words, value k at bit offset bits*k."""
    n, k = q.shape
    words = [[0] * (k * bits // 32) for _ in range(n)]
    for r in range(n):
        for j in range(k):
            v = int(q[r, j])
            assert 0 <= v < (1 << bits)
            pos = bits * j
            words[r][pos // 32] |= (v << (pos % 32)) & 0xFFFFFFFF
            spill = (pos % 32) + bits - 32
            if spill > 0:
                words[r][pos // 32 + 1] |= v >> (bits - spill)
    return np.array(words, dtype=np.uint32)


def bf16_exact(b: int) -> Fraction:
    """Exact rational value of a bf16 bit pattern (finite values only)."""
    sign = -1 if (b >> 15) & 1 else 1
    e = (b >> 7) & 0xFF
    m = b & 0x7F
    assert e != 0xFF
    if e == 0:
        return sign * Fraction(m, 1 << 7) * Fraction(1, 1 << 126)
    val = Fraction(128 + m, 128)
    p = e - 127
    return sign * (val * (1 << p) if p >= 0 else val / (1 << -p))


def exact_linear(q, s_bits, b_bits, x_bits):
    """Exact y[r, n] = sum_k (s*q + b) x and A[r, n] = sum_k |(s*q + b) x| as Fractions."""
    n, k = q.shape
    rows = x_bits.shape[0]
    y = [[Fraction(0)] * n for _ in range(rows)]
    a = [[Fraction(0)] * n for _ in range(rows)]
    for r in range(rows):
        xs = [bf16_exact(int(v)) for v in x_bits[r]]
        for i in range(n):
            acc = Fraction(0)
            aacc = Fraction(0)
            for j in range(k):
                g = j // 64
                w = bf16_exact(int(s_bits[i, g])) * int(q[i, j]) + bf16_exact(int(b_bits[i, g]))
                acc += w * xs[j]
                aacc += abs(w * xs[j])
            y[r][i] = acc
            a[r][i] = aacc
    return y, a


def parse_golden(path=GOLDEN):
    cases, cur = [], None
    for raw in open(path):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(":")
        val = val.strip()
        if key == "case":
            cur = {"name": val, "rows": [], "probes": []}
            cases.append(cur)
        elif key in ("bits", "k"):
            cur[key] = int(val)
        elif key == "row":
            words, scales, biases = (p.strip() for p in val.split("|"))
            cur["rows"].append((
                [int(w, 16) for w in words.split()],
                [int(s, 16) for s in scales.replace("scales:", "").split()],
                [int(b, 16) for b in biases.replace("biases:", "").split()],
            ))
        elif key == "probe":
            lhs, rhs = (p.strip() for p in val.split("->"))
            cur["probes"].append((lhs.split(), [Fraction(v) for v in rhs.split()]))
        else:
            raise ValueError(f"bad golden line {line!r}")
    return cases


def golden_x(probe, k):
    x = np.zeros((1, k), dtype=np.uint16)
    if probe[0] == "ones":
        x[:] = 0x3F80
    else:
        assert probe[0] == "onehot"
        x[0, int(probe[1])] = int(probe[2], 16)
    return x


# --------------------------------------------------------------------------------------
# pin checks, written as functions so that planted mutants can be run through them
# --------------------------------------------------------------------------------------
def check_golden(o=orc):
    for case in parse_golden():
        bits, k = case["bits"], case["k"]
        wq = np.array([r[0] for r in case["rows"]], dtype=np.uint32)
        sc = np.array([r[1] for r in case["rows"]], dtype=np.uint16)
        bi = np.array([r[2] for r in case["rows"]], dtype=np.uint16)
        for probe, want in case["probes"]:
            y, _ = o.qlinear(golden_x(probe, k), wq, sc, bi, bits)
            got = [Fraction(float(v)) for v in y[0]]
            assert got == want, f"{case['name']} {probe}: {got} != {want}"


def check_bruteforce(o=orc, seed=7):
    g = np.random.default_rng(seed)
    for bits in (4, 6, 8):
        for k in (64, 128):
            for n, rows in ((1, 1), (3, 2), (k, 1)):
                q = g.integers(0, 1 << bits, size=(n, k))
                s = synth.f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(n, k // 64)))
                b = synth.f32_to_bf16_bits(g.uniform(-0.1, 0.1, size=(n, k // 64)))
                x = synth.f32_to_bf16_bits(g.standard_normal(size=(rows, k)))
                wq = pack_rows(q, bits)
                y, a = o.qlinear(x, wq, s, b, bits)
                ye, ae = exact_linear(q, s, b, x)
                for r in range(rows):
                    for i in range(n):
                        tol = 1e-14 * float(ae[r][i])
                        assert abs(Fraction(float(y[r, i])) - ye[r][i]) <= tol, (bits, k, n, r, i)
                        assert abs(Fraction(float(a[r, i])) - ae[r][i]) <= tol


def check_closed_forms(o=orc, seed=11):
    g = np.random.default_rng(seed)
    for bits in (4, 6, 8):
        n, k = 5, 192
        q = g.integers(0, 1 << bits, size=(n, k))
        s = synth.f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(n, k // 64)))
        b = synth.f32_to_bf16_bits(g.uniform(-0.1, 0.1, size=(n, k // 64)))
        wq = pack_rows(q, bits)
        sf = np.vectorize(lambda v: float(bf16_exact(int(v))))(s)
        bf = np.vectorize(lambda v: float(bf16_exact(int(v))))(b)
        # x = 1: y = sum_g (s_g * sum_{k in g} q + 64 * b_g)
        ones = np.full((1, k), 0x3F80, dtype=np.uint16)
        y, _ = o.qlinear(ones, wq, s, b, bits)
        qsum = q.reshape(n, k // 64, 64).sum(axis=2)
        want = (sf * qsum + 64.0 * bf).sum(axis=1)
        np.testing.assert_allclose(y[0], want, rtol=1e-14, atol=0)
        # one-hot x at k = j: y = s[:, j//64] * q[:, j] + b[:, j//64]
        for j in (0, 63, 64, 100, 191):
            x = np.zeros((1, k), dtype=np.uint16)
            x[0, j] = 0x3F80
            y, _ = o.qlinear(x, wq, s, b, bits)
            np.testing.assert_array_equal(y[0], sf[:, j // 64] * q[:, j] + bf[:, j // 64])


def check_invariants(o=orc, seed=5):
    for bits in (4, 6, 8):
        w = synth.make_weight(7, 256, bits, seed=seed, config_id=90, tensor_id=bits)
        x = synth.make_x(3, 256, seed=seed, config_id=90)
        y, a = o.qlinear(x, w["wq"], w["scales"], w["biases"], bits)
        # rows computed alone equal rows inside the batch
        for r in range(3):
            yr, _ = o.qlinear(x[r:r + 1], w["wq"], w["scales"], w["biases"], bits)
            np.testing.assert_array_equal(yr[0], y[r])
        # linearity over disjoint supports (x1 + x2 is exact in bf16)
        mask = (np.arange(256) % 3) == 0
        x1 = np.where(mask, x, 0).astype(np.uint16)
        x2 = np.where(~mask, x, 0).astype(np.uint16)
        y1, _ = o.qlinear(x1, w["wq"], w["scales"], w["biases"], bits)
        y2, _ = o.qlinear(x2, w["wq"], w["scales"], w["biases"], bits)
        np.testing.assert_allclose(y1 + y2, y, rtol=0, atol=1e-13 * a.max())
        # permuting whole 64-wide groups of x and W together leaves y unchanged
        perm = np.array([2, 0, 3, 1])
        wpg = 64 * bits // 32
        wq_p = w["wq"].reshape(7, 4, wpg)[:, perm].reshape(7, -1)
        x_p = x.reshape(3, 4, 64)[:, perm].reshape(3, -1)
        yp, _ = o.qlinear(x_p, wq_p, w["scales"][:, perm], w["biases"][:, perm], bits)
        np.testing.assert_allclose(yp, y, rtol=0, atol=1e-13 * a.max())


def check_silu(o=orc):
    assert o.silu(0.0) == 0.0
    assert o.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert o.silu(-1.0) == pytest.approx(-1.0 / (1.0 + math.e), rel=1e-15)
    assert o.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert abs(o.silu(-800.0)) == 0.0
    # silu(t) - silu(-t) = t
    t = np.linspace(-6, 6, 25)
    np.testing.assert_allclose(o.silu(t) - o.silu(-t), t, rtol=0, atol=1e-15)


def check_ffn(o=orc):
    # w3: q = 0, bias 1 -> c = sum(x); w1: q = 1, scale 1, bias 0 -> a = sum(x)
    k = 64
    x = np.zeros((1, k), dtype=np.uint16)
    x[0, 3] = 0x4000  # 2.0
    w1 = {"wq": pack_rows(np.ones((2, k), dtype=np.int64), 4),
          "scales": np.array([[0x3F80], [0x4000]], np.uint16),
          "biases": np.zeros((2, 1), np.uint16), "bits": 4}
    w3 = {"wq": np.zeros((2, 8), np.uint32), "scales": np.full((2, 1), 0x3F80, np.uint16),
          "biases": np.array([[0x3F80], [0xBF80]], np.uint16), "bits": 4}
    a, _, c, _, h = o.ffn_swiglu(x, w1, w3)
    np.testing.assert_array_equal(a[0], [2.0, 4.0])
    np.testing.assert_array_equal(c[0], [2.0, -2.0])
    want = [2.0 / (1 + math.exp(-2.0)) * 2.0, 4.0 / (1 + math.exp(-4.0)) * -2.0]
    np.testing.assert_allclose(h[0], want, rtol=1e-15)


def check_error_bound(o=orc):
    # config-like data: the oracle's own float64 error is far below 1e-12 * A
    bits, n, k = 4, 4, 2048
    g = np.random.default_rng(3)
    q = g.integers(0, 16, size=(n, k))
    s = synth.f32_to_bf16_bits(g.uniform(0.005, 0.02, size=(n, k // 64)))
    b = synth.f32_to_bf16_bits(g.uniform(-0.1, 0.1, size=(n, k // 64)))
    x = synth.f32_to_bf16_bits(g.standard_normal(size=(1, k)))
    y, a = o.qlinear(x, pack_rows(q, bits), s, b, bits)
    ye, ae = exact_linear(q, s, b, x)
    for i in range(n):
        assert abs(Fraction(float(y[0, i])) - ye[0][i]) <= Fraction(1, 10**12) * ae[0][i]


PINS = [check_golden, check_bruteforce, check_closed_forms, check_invariants,
        check_silu, check_ffn, check_error_bound]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin()


def test_packer_roundtrip_matches_fixture():
    # the test-side packer reproduces the hand-packed words of the fixtures
    q = np.zeros((1, 64), dtype=np.int64)
    q[0, :16] = np.arange(16)
    assert list(pack_rows(q, 4)[0, :2]) == [0x76543210, 0xFEDCBA98]
    q6 = np.zeros((1, 64), dtype=np.int64)
    q6[0, :6] = np.arange(6)
    assert list(pack_rows(q6, 6)[0, :2]) == [0x440C2040, 0x00000001]
    q8 = np.zeros((1, 64), dtype=np.int64)
    q8[0, :8] = [0, 1, 2, 3, 1, 127, 128, 255]
    assert list(pack_rows(q8, 8)[0, :2]) == [0x03020100, 0xFF807F01]


# --------------------------------------------------------------------------------------
# planted mistakes: every mutant must fail at least one pin
# --------------------------------------------------------------------------------------
class _Mutant:
    """The oracle with one function replaced."""

    def __init__(self, **over):
        self.__dict__.update({n: getattr(orc, n) for n in dir(orc) if not n.startswith("_")})
        self.__dict__.update(over)
        me = self

        def dequant(wq, scales, biases, bits, k):
            return me._dequant(me, wq, scales, biases, bits, k)

        def qlinear(x_bits, wq, scales, biases, bits):
            return me._qlinear(me, x_bits, wq, scales, biases, bits)

        self.dequant = dequant
        self.qlinear = qlinear
        self.qlinear_w = lambda x, w: self.qlinear(x, w["wq"], w["scales"], w["biases"], w["bits"])
        self.ffn_swiglu = lambda x, w1, w3: _ffn(self, x, w1, w3)

    @staticmethod
    def _dequant(me, wq, scales, biases, bits, k):
        q = me.unpack_q(wq, bits, k).astype(np.float64)
        s, b = me.bf16_bits_to_f64(scales), me.bf16_bits_to_f64(biases)
        gidx = me.group_index(k)
        return me.combine(s[:, gidx], q, b[:, gidx])

    @staticmethod
    def _qlinear(me, x_bits, wq, scales, biases, bits):
        x = me.bf16_bits_to_f64(np.atleast_2d(x_bits))
        w = me.dequant(wq, scales, biases, bits, x.shape[1])
        return me.matvec(x, w), np.abs(x) @ np.abs(w).T


def _ffn(o, x, w1, w3):
    a, aa = o.qlinear_w(x, w1)
    c, ac = o.qlinear_w(x, w3)
    return a, aa, c, ac, o.silu(a) * c


def _base(**over):
    d = dict(group_index=lambda k: np.arange(k) // 64,
             combine=lambda s, q, b: s * q + b,
             matvec=lambda x, w: x @ w.T)
    d.update(over)
    return _Mutant(**d)


def _unpack_high_first(wq, bits, k):
    q = orc.unpack_q(wq, bits, k)
    per = 32 // bits if 32 % bits == 0 else 1
    if per == 1:
        return q
    return q.reshape(q.shape[0], -1, per)[:, :, ::-1].reshape(q.shape[0], k)


def _unpack_no_straddle(wq, bits, k):
    wq = np.asarray(wq, dtype=np.uint32).astype(np.uint64)
    pos = bits * np.arange(k)
    return ((wq[:, pos // 32] >> (pos % 32).astype(np.uint64)) & ((1 << bits) - 1)).astype(np.int64)


MUTANTS = {
    "correct_composition": None,  # sanity: the harness itself passes with no mutation
    "high_field_first": dict(unpack_q=_unpack_high_first),
    "no_straddle": dict(unpack_q=_unpack_no_straddle),
    "bias_dropped": dict(combine=lambda s, q, b: s * q),
    "bias_sign": dict(combine=lambda s, q, b: s * q - b),
    "group_of_32": dict(group_index=lambda k: np.minimum(np.arange(k) // 32, k // 64 - 1)),
    "scale_on_bias": dict(combine=lambda s, q, b: s * (q + b)),
    "weight_transposed": dict(matvec=lambda x, w: (x @ w.T) if w.shape[0] != w.shape[1]
                              else x @ w),
    "silu_sign": dict(silu=lambda t: np.asarray(t, float) / (1.0 + np.exp(np.asarray(t, float)))),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mutant(name):
    over = MUTANTS[name]
    o = _base(**(over or {}))
    failures = 0
    for pin in PINS:
        try:
            pin(o)
        except Exception:  # noqa: BLE001 - a shape error is a failed pin too
            failures += 1
    if over is None:
        assert failures == 0
    else:
        assert failures >= 1, f"mutant {name} passed every pin"
