"""Full-size checks in the launch configurations the benchmark times: the
full-depth sweep's layer shapes in 4-, 6- and 8-bit, decode at R = 1 and 16, and an
8192-row prompt in windows of 128 against one M = 8192 GEMM (bit for bit), with the
oracle evaluated on sampled rows."""
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


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_sweep_layer_decode(q, bits):
    # one FFN layer and one attention set of the sweep, decode at R = 1 and 16
    w1 = U.weight(8192, 2048, bits, config_id=4, tensor_id=1)
    w3 = U.weight(8192, 2048, bits, config_id=4, tensor_id=3)
    w2 = U.weight(2048, 8192, bits, config_id=4, tensor_id=2)
    attn = [U.weight(n, 2048, bits, config_id=4, tensor_id=10 + i) for i, n in enumerate((2048, 512, 512, 2048))]
    d1, d3, d2 = U.dev_weight(w1), U.dev_weight(w3), U.dev_weight(w2)
    da = [U.dev_weight(w) for w in attn]
    x = synth.make_x(16, 2048, config_id=4)
    xd = U.dev_x(x)
    for rows in (1, 16):
        h = q.qffn_swiglu_mv(d1, d3, xd[:rows])
        out = q.qlinear_mv_rows(d2, h)
        a64, aa, c64, ac, h64 = orc.ffn_swiglu(x[:rows], w1, w3)
        hg = h.float().cpu().numpy().astype(np.float64)
        assert (np.abs(hg - h64) <= U.h_bound(a64, aa, c64, ac, h64)).all()
        o64, oa = orc.qlinear_w(q.bits_of(h), w2)
        U.assert_close(out, o64, oa, f"w2 bits={bits} rows={rows}")
        outs = q.qattn_proj_mv(*da, xd[:rows])
        for w, o in zip(attn, outs):
            y64, A = orc.qlinear_w(x[:rows], w)
            U.assert_close(o, y64, A, f"attn bits={bits} rows={rows}")
    # 16 rows == 16 one-row calls for the down projection over K = 8192
    hh = q.qffn_swiglu_mv(d1, d3, xd)
    y16 = q.qlinear_mv_rows(d2, hh)
    for r in range(16):
        assert torch.equal(q.qlinear_mv(d2, hh[r]), y16[r])


@pytest.mark.parametrize("bits,n,k", [(4, 8192, 2048), (6, 2048, 8192), (8, 2048, 2048)])
def test_prompt_8192_windows_of_128(q, bits, n, k):
    w = U.weight(n, k, bits, config_id=4, tensor_id=20 + bits)
    X = synth.make_x(8192, k, config_id=4, tensor_id=2000)
    wd, Xd = U.dev_weight(w), U.dev_x(X)
    Y = q.qlinear_pgemm(wd, Xd)
    Yw = torch.empty_like(Y)
    for lo in range(0, 8192, 128):
        q.qlinear_pgemm(wd, Xd[lo:lo + 128], Y=Yw[lo:lo + 128])
    assert torch.equal(Yw, Y), "windows of 128 differ from one M = 8192 GEMM"
    rows = np.random.default_rng(bits).choice(8192, size=48, replace=False)
    rows.sort()
    y64, A = orc.pgemm(X[rows], w)
    U.assert_close(Y[torch.from_numpy(rows).cuda()], y64, A, f"pgemm 8192 rows bits={bits}")
