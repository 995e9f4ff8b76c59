"""Copy-draft verification windows (TensorFold PR #1696, "What it adds": streams share
a decode step through N-row matvecs that sum each row as the one-row kernels do, so a
window of drafted tokens is checked in one weight pass): a window of R <= 16 rows
pushed through a whole decoder layer - q/k/v/gate, QK norm + partial RoPE + KV store,
o, post-add / next-norm, w1 + w3 + SwiGLU, w2, post-add / next-norm - gives every row
exactly the bits that row gets when it is stepped alone.  Rows are distinct draft
positions of one stream here, so each row writes its own KV slot."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from tests._util import weight
from weight_only_bit_mlx_gb300 import synth

pytestmark = pytest.mark.gpu

D, DFF, DKV, HD, ROT, RING = 512, 1536, 128, 64, 32, 32


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from weight_only_bit_mlx_gb300 import qlinear
    return qlinear


def make_layer(q, bits, cid):
    def w(n, k, tid):
        return q.QWeight.from_numpy(weight(n, k, bits, config_id=cid, tensor_id=tid))
    L = {"q": w(D, D, 1), "k": w(DKV, D, 2), "v": w(DKV, D, 3), "g": w(D, D, 4), "o": w(D, D, 5),
         "w1": w(DFF, D, 6), "w3": w(DFF, D, 7), "w2": w(D, DFF, 8)}
    bf = lambda a: q.bf16_from_bits(a)  # noqa: E731
    L["qn"] = bf(synth.make_bf16((HD,), 0.5, 1.5, config_id=cid, tensor_id=9))
    L["kn"] = bf(synth.make_bf16((HD,), 0.5, 1.5, config_id=cid, tensor_id=10))
    L["g1"] = bf(synth.make_bf16((D,), 0.5, 1.5, config_id=cid, tensor_id=11))
    L["g2"] = bf(synth.make_bf16((D,), 0.5, 1.5, config_id=cid, tensor_id=12))
    return L


def layer_step(q, L, x, resid, attn, pos, k_ring, v_ring):
    """One decoder layer's linear path for the rows of x (bf16 [R, D]); resid is
    updated in place; returns every output."""
    R = x.shape[0]
    qf, kf, vf, gf = (torch.empty(R, n, device="cuda") for n in (D, DKV, DKV, D))
    q.qattn_proj_mv(L["q"], L["k"], L["v"], L["g"], x, outs=(qf, kf, vf, gf))
    q_out = q.qattn_qknorm_rope_kv(qf, kf, vf, D // HD, DKV // HD, HD, ROT, 1e6, 1e-5, L["qn"], L["kn"], pos,
                                   k_ring, v_ring)
    o = q.qlinear_mv_rows(L["o"], attn)
    x1 = q.qresid_rmsnorm(o, resid, L["g1"], 1e-5)
    h = q.qffn_swiglu_mv(L["w1"], L["w3"], x1)
    y = q.qlinear_mv_rows(L["w2"], h)
    x2 = q.qresid_rmsnorm(y, resid, L["g2"], 1e-5)
    return {"q": qf, "k": kf, "v": vf, "gate": gf, "q_out": q_out, "o": o, "x1": x1, "h": h, "y": y, "x2": x2,
            "resid": resid}


def same_bits(a, b):
    ia = a.view(torch.int16) if a.element_size() == 2 else a.view(torch.int32)
    ib = b.view(torch.int16) if b.element_size() == 2 else b.view(torch.int32)
    return torch.equal(ia, ib)


@pytest.mark.parametrize("bits", [4, 6, 8])
@pytest.mark.parametrize("R", [2, 7, 16])
def test_verification_window_equals_single_steps(q, bits, R):
    cid = 100 * bits + R
    L = make_layer(q, bits, cid)
    x = q.bf16_from_bits(synth.make_x(R, D, config_id=cid, tensor_id=20))
    attn = q.bf16_from_bits(synth.make_x(R, D, config_id=cid, tensor_id=21))
    resid0 = q.bf16_from_bits(synth.make_bf16((R, D), config_id=cid, tensor_id=22))
    # a draft window: consecutive positions of one stream, one ring per row
    pos = torch.arange(1000, 1000 + R, dtype=torch.int32, device="cuda")
    kr = torch.zeros(R, RING, DKV, dtype=torch.bfloat16, device="cuda")
    vr = torch.zeros_like(kr)
    win = layer_step(q, L, x, resid0.clone(), attn, pos, kr, vr)
    for r in range(R):
        kr1 = torch.zeros(1, RING, DKV, dtype=torch.bfloat16, device="cuda")
        vr1 = torch.zeros_like(kr1)
        one = layer_step(q, L, x[r:r + 1].clone(), resid0[r:r + 1].clone(), attn[r:r + 1].clone(), pos[r:r + 1],
                         kr1, vr1)
        for name, t in one.items():
            assert same_bits(t[0], win[name][r]), f"row {r}: {name}"
        assert same_bits(kr1[0], kr[r]) and same_bits(vr1[0], vr[r]), f"row {r}: KV ring"
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    # the window's rows differ from each other (a window of identical rows would pass trivially)
    assert not same_bits(win["x2"][0], win["x2"][1])
