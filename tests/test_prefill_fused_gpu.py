"""The prompt GEMM with the decoder steps that follow it as its epilogue.

TensorFold PR #1514, "What changes": post-add/next-norm fusion; paired FFN
projections keep their retained rounding boundaries.  PR #1696 (later revision),
"What it adds": decode fuses w1 + w3 + SwiGLU; the prompt GEMM.

* qlinear_pgemm_swiglu: the up projection's GEMM writes h = bf16(silu(a) * c) straight
  from its accumulator; bit-equal to qswiglu(a, qlinear_pgemm(w3, X)) and within the
  bound propagated from the float64 a and c; a window of rows equals those rows of the
  whole prompt.
* qlinear_pgemm_resid_norm: the w2 / o GEMM adds its output into the bf16 residual in its
  epilogue, then the norm runs on the stored residual; both the residual and the normed
  output are bit-equal to qlinear_pgemm followed by qresid_rmsnorm, and within tolerance
  of the float64 definitions.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import decoder_post_oracle as po
from oracle import qlinear_oracle as orc
from tests import _util as U
from weight_only_bit_mlx_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    from weight_only_bit_mlx_gb300 import qlinear
    assert torch.cuda.is_available()
    return qlinear


# the last shape is past the row count from which the codes are converted once per call
# (the window of 100 rows below it is converted inside the GEMM: the two paths meet there)
SHAPES = [(4, 300, 1000, 2048), (6, 517, 512, 1024), (8, 64, 768, 2048), (4, 1024, 8192, 2048),
          (6, 2100, 1024, 2048)]


@pytest.mark.parametrize("bits,m,n,k", SHAPES)
def test_pgemm_swiglu(q, bits, m, n, k):
    cid = 160 + bits
    w1, w3 = U.weight(n, k, bits, config_id=cid, tensor_id=1), U.weight(n, k, bits, config_id=cid, tensor_id=3)
    X = synth.make_x(m, k, config_id=cid)
    d1, d3, Xd = U.dev_weight(w1), U.dev_weight(w3), U.dev_x(X)
    A = q.qlinear_pgemm(d1, Xd)
    C = q.qlinear_pgemm(d3, Xd)
    H = q.qlinear_pgemm_swiglu(d3, Xd, A)
    # fusion on == fusion off, bit for bit
    assert torch.equal(H, q.qswiglu(A, C))
    # a window of rows, alone, equals the same rows of the whole prompt
    lo, hi = min(17, m - 1), min(17 + 100, m)
    assert torch.equal(q.qlinear_pgemm_swiglu(d3, Xd[lo:hi], A[lo:hi]), H[lo:hi])
    torch.cuda.synchronize()
    a64, aa, c64, ac, h64 = orc.ffn_swiglu(X, w1, w3)
    U.assert_close(A, a64, aa, "w1 X")
    U.assert_close(C, c64, ac, "w3 X")
    hg = H.float().cpu().numpy().astype(np.float64)
    assert (np.abs(hg - h64) <= U.h_bound(a64, aa, c64, ac, h64)).all(), "h out of propagated bound"


@pytest.mark.parametrize("bits,m,n,k", [(4, 300, 2048, 8192), (6, 1030, 1000, 2048), (8, 5, 2048, 2048),
                                        (8, 2200, 768, 2048)])
def test_pgemm_resid_norm(q, bits, m, n, k):
    cid = 170 + bits
    w = U.weight(n, k, bits, config_id=cid, tensor_id=1)
    X = synth.make_x(m, k, config_id=cid)
    r0 = synth.make_bf16((m, n), config_id=cid, tensor_id=2)
    gb = synth.make_bf16((n,), 0.5, 1.5, config_id=cid, tensor_id=3)
    wd, Xd, gamma = U.dev_weight(w), U.dev_x(X), U.dev_x(gb)
    eps = 1e-5
    rf = U.dev_x(r0)
    out_f = q.qlinear_pgemm_resid_norm(wd, Xd, rf, gamma, eps)
    rs = U.dev_x(r0)
    Y = q.qlinear_pgemm(wd, Xd)
    out_s = q.qresid_rmsnorm(Y, rs, gamma, eps)
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    assert torch.equal(rf.view(torch.int16), rs.view(torch.int16)), "stored residual"
    assert torch.equal(out_f.view(torch.int16), out_s.view(torch.int16)), "normed output"
    # against the float64 definitions: the residual within the GEMM's tolerance plus half
    # a bf16 ulp, the normed output within half a bf16 ulp plus fp32 error of the
    # oracle's norm of the stored residual
    y64, A = orc.pgemm(X, w)
    rb = q.bits_of(rf)
    r_got = po.bf16_bits_to_f64(rb)
    r64 = po.bf16_bits_to_f64(r0) + y64
    assert (np.abs(r_got - r64) <= U.tol(A) + 2.0 ** -8 * np.abs(r64) + 1e-30).all()
    r_same, o64 = po.resid_rms_norm(rb, np.zeros(rb.shape), gb, float(np.float32(eps)))
    assert np.array_equal(r_same, rb)
    got = po.bf16_bits_to_f64(q.bits_of(out_f))
    assert (np.abs(got - o64) <= 2.0 ** -8 * np.abs(o64) + 1e-5).all()
