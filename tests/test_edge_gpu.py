"""Decode and prompt-GEMM parity on the method's degenerate weights.

The acceptance bound |y - y64| <= 1e-5 * sum|w x| + 1e-6 shrinks to 1e-6 where the
dequantized weights vanish, so these rows check that the error of the kernels scales
with |w x| and not with the size of the codes or of the activations:

* zero rows: q = 0 and bias = 0 (any scale) - what an all-zero group quantizes to;
* cancelling rows: q = c and bias = -scale * c with c a power of two, so that the
  bias is exact in bf16 and every dequantized weight is exactly 0 although no code is;
* half-zero rows: every even group zero as above, the odd groups random;
* random rows, with activations ~ N(0, 1) and with large activations (~ 1024 N(0, 1)).

TensorFold PR #1696 (later revision), "What it adds": MLX 4-bit group 64 as stored,
dequantized in-kernel; PR #1514 "What changes": MLX 4/6/8-bit checkpoints.  The
packed rows come from the test's own packer; the expected values from the float64
oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import qlinear_oracle as orc
from tests import _util as U
from weight_only_bit_mlx_gb300 import synth

pytestmark = pytest.mark.gpu

BAND = 64  # rows per pattern


@pytest.fixture(scope="module")
def q():
    from weight_only_bit_mlx_gb300 import qlinear
    assert torch.cuda.is_available()
    return qlinear


def edge_weight(k, bits, cid, tid, order=("zero", "cancel", "halfzero", "random")):
    """A weight of len(order) bands of BAND rows, one pattern per band."""
    n = BAND * len(order)
    w = U.weight(n, k, bits, config_id=cid, tensor_id=tid)
    wq, sc, bi = w["wq"].copy(), w["scales"].copy(), w["biases"].copy()
    g = synth.rng_for(0, cid, tid + 500)
    s64 = orc.bf16_bits_to_f64(sc)
    words_per_group = 2 * bits
    for i, pat in enumerate(order):
        rows = slice(i * BAND, (i + 1) * BAND)
        if pat == "zero":
            wq[rows] = 0
            bi[rows] = 0
        elif pat == "cancel":
            c = 1 << g.integers(0, bits, size=BAND)            # powers of two below 2^bits
            wq[rows] = U.pack_codes(np.repeat(c[:, None], k, axis=1), bits)
            bi[rows] = synth.f32_to_bf16_bits(-(s64[rows] * c[:, None]))  # exact: a power-of-two multiple
        elif pat == "halfzero":
            for gg in range(0, k // 64, 2):
                wq[rows, gg * words_per_group:(gg + 1) * words_per_group] = 0
            bi[rows, 0::2] = 0
    out = dict(w, wq=wq, scales=sc, biases=bi)
    if "cancel" in order:  # the cancelling band really dequantizes to zero
        i = order.index("cancel")
        assert not orc.dequant(wq, sc, bi, bits, k)[i * BAND:(i + 1) * BAND].any()
    return out


def acts(rows, k, cid, big):
    x = synth.make_x(rows, k, config_id=cid)
    if big:  # |x| up to a few thousand: scale the N(0, 1) draw by 2^10 (exact in bf16)
        x = synth.f32_to_bf16_bits(orc.bf16_bits_to_f64(x) * 1024.0)
    return x


CASES = [(bits, k, big) for bits in (4, 6, 8) for k in (2048, 8192) for big in (False, True)]


@pytest.mark.parametrize("bits,k,big", CASES)
def test_edge_rows_mv(q, bits, k, big):
    cid = 90 + bits
    w = edge_weight(k, bits, cid, 1)
    wd = U.dev_weight(w)
    x = acts(16, k, cid, big)
    xd = U.dev_x(x)
    y64, A = orc.qlinear_w(x, w)
    for rows in (1, 16):
        y = q.qlinear_mv_rows(wd, xd[:rows])
        torch.cuda.synchronize()
        U.assert_close(y, y64[:rows], A[:rows], f"mv_rows bits={bits} k={k} big={big} rows={rows}")


@pytest.mark.parametrize("bits,k,big", CASES)
def test_edge_rows_fused_ffn(q, bits, k, big):
    cid = 100 + bits
    w1 = edge_weight(k, bits, cid, 1)
    w3 = edge_weight(k, bits, cid, 3, order=("random", "halfzero", "cancel", "zero"))
    d1, d3 = U.dev_weight(w1), U.dev_weight(w3)
    x = acts(16, k, cid, big)
    xd = U.dev_x(x)
    for rows in (1, 16):
        h = q.qffn_swiglu_mv(d1, d3, xd[:rows])
        a = q.qlinear_mv_rows(d1, xd[:rows])
        c = q.qlinear_mv_rows(d3, xd[:rows])
        assert torch.equal(h, q.qswiglu(a, c)), "fused FFN != unfused"
        torch.cuda.synchronize()
        a64, aa, c64, ac, h64 = orc.ffn_swiglu(x[:rows], w1, w3)
        U.assert_close(a, a64, aa, f"w1 x bits={bits} k={k} rows={rows}")
        U.assert_close(c, c64, ac, f"w3 x bits={bits} k={k} rows={rows}")
        hg = h.float().cpu().numpy().astype(np.float64)
        assert (np.abs(hg - h64) <= U.h_bound(a64, aa, c64, ac, h64)).all(), "h out of propagated bound"


@pytest.mark.parametrize("bits,k,big", CASES)
def test_edge_rows_fused_attention(q, bits, k, big):
    cid = 110 + bits
    orders = [("zero", "cancel", "halfzero", "random"), ("cancel", "random"), ("halfzero", "zero"),
              ("random", "zero", "cancel", "halfzero")]
    ws = [edge_weight(k, bits, cid, t, order=o) for t, o in enumerate(orders)]
    ds = [U.dev_weight(w) for w in ws]
    x = acts(16, k, cid, big)
    xd = U.dev_x(x)
    for rows in (1, 16):
        outs = q.qattn_proj_mv(*ds, xd[:rows])
        torch.cuda.synchronize()
        for t, (w, o) in enumerate(zip(ws, outs)):
            y64, A = orc.qlinear_w(x[:rows], w)
            U.assert_close(o, y64, A, f"attn {t} bits={bits} k={k} rows={rows}")


@pytest.mark.parametrize("bits,k,big", [(b, k, big) for b in (4, 6, 8) for k in (2048, 8192) for big in (False, True)])
def test_edge_rows_pgemm(q, bits, k, big):
    # zero, half-zero and random rows through the prompt GEMM; 300 rows span two 256-row
    # tiles and a ragged tail
    cid = 120 + bits
    w = edge_weight(k, bits, cid, 1, order=("zero", "halfzero", "random"))
    X = acts(300, k, cid, big)
    Y = q.qlinear_pgemm(U.dev_weight(w), U.dev_x(X))
    torch.cuda.synchronize()
    y64, A = orc.pgemm(X, w)
    U.assert_close(Y, y64, A, f"pgemm bits={bits} k={k} big={big}")
