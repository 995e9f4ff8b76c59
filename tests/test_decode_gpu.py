"""Decode kernels on the GPU against the float64 oracle, plus their bit-exact
invariants (N-row vs one-row calls, fused vs unfused, strided activations).

Tolerance (per output): |y - y64| <= 1e-5 * sum|w x| + 1e-6.
TensorFold PR #1696 (later revision), "What it adds": N-row matvecs sum each row as
the one-row kernels do (checked bit for bit); decode fuses w1 + w3 + SwiGLU and the
four attention matvecs (checked against the unfused calls, bit for bit).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import qlinear_oracle as orc
from tests import _util as U
from weight_only_bit_mlx_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    from weight_only_bit_mlx_gb300 import qlinear
    assert torch.cuda.is_available()
    return qlinear


def test_single_qmv_2048(q):
    # single qmv: x [1, 2048], W 2048 -> 2048, 4-bit, seed 0
    w = U.weight(2048, 2048, 4, config_id=0, tensor_id=0)
    x = synth.make_x(1, 2048, config_id=0)
    y = q.qlinear_mv(U.dev_weight(w), U.dev_x(x[0]))
    torch.cuda.synchronize()
    y64, A = orc.qlinear_w(x, w)
    U.assert_close(y.view(1, -1), y64, A, "qmv 2048x2048")


SHAPES = [(2048, 2048), (37, 64), (100, 192), (513, 8192), (16, 512), (520, 1024), (48, 4096)]


@pytest.mark.parametrize("bits", [4, 6, 8])
@pytest.mark.parametrize("n,k", SHAPES)
def test_rows_against_oracle(q, bits, n, k):
    w = U.weight(n, k, bits, config_id=50, tensor_id=bits)
    wd = U.dev_weight(w)
    x = synth.make_x(16, k, config_id=50)
    xd = U.dev_x(x)
    y64, A = orc.qlinear_w(x, w)
    for rows in (1, 3, 8, 9, 16):
        y = q.qlinear_mv_rows(wd, xd[:rows])
        torch.cuda.synchronize()
        U.assert_close(y, y64[:rows], A[:rows], f"bits={bits} n={n} k={k} rows={rows}")


@pytest.mark.parametrize("bits", [4, 6, 8])
@pytest.mark.parametrize("n,k", [(2048, 2048), (100, 192), (513, 8192), (2048, 8192)])
def test_rows_bit_equal_to_single_rows(q, bits, n, k):
    w = U.dev_weight(U.weight(n, k, bits, config_id=51, tensor_id=bits))
    xd = U.dev_x(synth.make_x(16, k, config_id=51))
    singles = torch.stack([q.qlinear_mv(w, xd[r]) for r in range(16)])
    for rows in range(1, 17):
        y = q.qlinear_mv_rows(w, xd[:rows])
        assert torch.equal(y, singles[:rows]), f"rows={rows} differs from one-row calls"
    # any subset of rows, in any position of the batch
    perm = torch.tensor([5, 0, 15, 7, 3])
    y = q.qlinear_mv_rows(w, xd[perm].contiguous())
    assert torch.equal(y, singles[perm])


def test_strided_activations(q):
    n, k = 300, 2048
    w = U.dev_weight(U.weight(n, k, 4, config_id=52))
    x = U.dev_x(synth.make_x(5, k + 64, config_id=52))
    xs = x[:, 64:]  # row stride k + 64, start offset 128 bytes
    y = q.qlinear_mv_rows(w, xs)
    y_ref = q.qlinear_mv_rows(w, xs.contiguous())
    assert torch.equal(y, y_ref)
    yout = torch.full((5, n + 7), float("nan"), device="cuda")
    q.qlinear_mv_rows(w, xs, y=yout[:, :n])
    assert torch.equal(yout[:, :n], y_ref)
    assert torch.isnan(yout[:, n:]).all()


@pytest.mark.parametrize("rows", [1, 2, 4, 8, 16])
def test_fused_ffn_decode(q, rows):
    # fused FFN decode: w1, w3 2048 -> 8192, w2 8192 -> 2048, 4-bit g64
    w1 = U.weight(8192, 2048, 4, config_id=1, tensor_id=1)
    w3 = U.weight(8192, 2048, 4, config_id=1, tensor_id=3)
    w2 = U.weight(2048, 8192, 4, config_id=1, tensor_id=2)
    x = synth.make_x(rows, 2048, config_id=1)
    d1, d3, d2, xd = U.dev_weight(w1), U.dev_weight(w3), U.dev_weight(w2), U.dev_x(x)
    h = q.qffn_swiglu_mv(d1, d3, xd)
    out = q.qlinear_mv_rows(d2, h)
    # fusion on == fusion off, bit for bit
    a = q.qlinear_mv_rows(d1, xd)
    c = q.qlinear_mv_rows(d3, xd)
    assert torch.equal(h, q.qswiglu(a, c))
    torch.cuda.synchronize()
    a64, aa, c64, ac, h64 = orc.ffn_swiglu(x, w1, w3)
    U.assert_close(a, a64, aa, "w1 x")
    U.assert_close(c, c64, ac, "w3 x")
    hg = h.float().cpu().numpy().astype(np.float64)
    bound = U.h_bound(a64, aa, c64, ac, h64)
    assert (np.abs(hg - h64) <= bound).all(), "h out of propagated bound"
    # down projection: oracle applied to the GPU's own bf16 h
    o64, oa = orc.qlinear_w(q.bits_of(h), w2)
    U.assert_close(out, o64, oa, "w2 h")
    # R-row result equals R one-row calls
    for r in range(rows):
        assert torch.equal(q.qffn_swiglu_mv(d1, d3, xd[r]), h[r:r + 1])


@pytest.mark.parametrize("bits,n,k", [(6, 8192, 2048), (8, 8192, 2048), (4, 1000, 192), (6, 37, 64),
                                      (8, 520, 1024)])
@pytest.mark.parametrize("rows", [1, 5, 16])
def test_fused_ffn_bits_and_ragged(q, bits, n, k, rows):
    # the fused w1 + w3 + SwiGLU decode at 6 and 8 bits and on channel counts that leave
    # a ragged last 16-row tile: h against the propagated float64 bound, fused ==
    # unfused and R rows == R one-row calls, bit for bit
    cid = 60 + bits
    w1 = U.weight(n, k, bits, config_id=cid, tensor_id=1)
    w3 = U.weight(n, k, bits, config_id=cid, tensor_id=3)
    x = synth.make_x(rows, k, config_id=cid)
    d1, d3, xd = U.dev_weight(w1), U.dev_weight(w3), U.dev_x(x)
    h = q.qffn_swiglu_mv(d1, d3, xd)
    a = q.qlinear_mv_rows(d1, xd)
    c = q.qlinear_mv_rows(d3, xd)
    assert torch.equal(h, q.qswiglu(a, c))
    torch.cuda.synchronize()
    a64, aa, c64, ac, h64 = orc.ffn_swiglu(x, w1, w3)
    U.assert_close(a, a64, aa, "w1 x")
    U.assert_close(c, c64, ac, "w3 x")
    hg = h.float().cpu().numpy().astype(np.float64)
    assert (np.abs(hg - h64) <= U.h_bound(a64, aa, c64, ac, h64)).all(), "h out of propagated bound"
    for r in (0, rows - 1):
        assert torch.equal(q.qffn_swiglu_mv(d1, d3, xd[r]), h[r:r + 1])


@pytest.mark.parametrize("rows", [1, 4, 16])
@pytest.mark.parametrize("bits", [4, 6, 8])
def test_fused_attention_projections(q, rows, bits):
    # q 2048->2048 (32 heads x 64), k, v 2048->512 (8 KV heads x 64), gate 2048->2048
    ns = {"q": 2048, "k": 512, "v": 512, "g": 2048}
    ws = {t: U.weight(n, 2048, bits, config_id=2, tensor_id=i) for i, (t, n) in enumerate(ns.items())}
    ds = {t: U.dev_weight(w) for t, w in ws.items()}
    x = synth.make_x(rows, 2048, config_id=2)
    xd = U.dev_x(x)
    outs = q.qattn_proj_mv(ds["q"], ds["k"], ds["v"], ds["g"], xd)
    for t, o in zip(ns, outs):
        assert torch.equal(o, q.qlinear_mv_rows(ds[t], xd)), f"fused {t} != unfused"
        y64, A = orc.qlinear_w(x, ws[t])
        U.assert_close(o, y64, A, f"attn {t}")


def test_attention_ragged_heads(q):
    ns = [72, 24, 40, 8]
    ws = [U.weight(n, 320, 6, config_id=53, tensor_id=i) for i, n in enumerate(ns)]
    ds = [U.dev_weight(w) for w in ws]
    x = synth.make_x(3, 320, config_id=53)
    outs = q.qattn_proj_mv(*ds, U.dev_x(x))
    for w, d, o in zip(ws, ds, outs):
        assert torch.equal(o, q.qlinear_mv_rows(d, U.dev_x(x)))
        y64, A = orc.qlinear_w(x, w)
        U.assert_close(o, y64, A, "ragged attention")


def test_deterministic_repeat(q):
    w = U.dev_weight(U.weight(1000, 4096, 4, config_id=54))
    xd = U.dev_x(synth.make_x(7, 4096, config_id=54))
    a = q.qlinear_mv_rows(w, xd)
    b = q.qlinear_mv_rows(w, xd)
    assert torch.equal(a, b)


@pytest.mark.parametrize("bits,k", [(4, 24576), (4, 65536), (6, 12288), (8, 16384)])
def test_several_spans_per_cta(q, bits, k):
    # k large enough that each CTA of the k-split cluster walks more than one span of
    # groups, reusing its shared-memory buffers between spans
    n = 48
    w = U.weight(n, k, bits, config_id=61, tensor_id=bits)
    wd = U.dev_weight(w)
    x = synth.make_x(9, k, config_id=61)
    xd = U.dev_x(x)
    y = q.qlinear_mv_rows(wd, xd)
    y1 = q.qlinear_mv(wd, xd[4])
    torch.cuda.synchronize()
    y64, A = orc.qlinear_w(x, w)
    U.assert_close(y, y64, A, f"bits={bits} k={k}")
    assert torch.equal(y1, y[4])
    assert q.qlinear_last_error() == q.QL_OK
