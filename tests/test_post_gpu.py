"""Parity of the post-projection decoder steps with the float64 oracle
(oracle/decoder_post_oracle.py): QK norm + partial RoPE + KV store (TensorFold PR
#1696, "What it adds") and post-add / next-norm (PR #1514, "What changes").

Outputs are bf16.  The kernels compute in fp32 (rotation angles formed and reduced in
float64) and round once,
so each output is within half a bf16 ulp of the float64 value plus the fp32 error:
    |out - o64| <= 2^-8 * |o64| + 1e-5        (values are O(1) after the norm)
and nearly all outputs equal the nearest-even bf16 of o64.  The stored residual is an
integer decision taken in the same precision on both sides (fp32 add, then bf16), so
it is compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import decoder_post_oracle as po
from weight_only_bit_mlx_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from weight_only_bit_mlx_gb300 import qlinear
    return qlinear


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def bits_host(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check_bf16(out_bits, o64, what, min_exact=0.98):
    got = po.bf16_bits_to_f64(out_bits)
    err = np.abs(got - o64)
    bound = 2.0 ** -8 * np.abs(o64) + 1e-5
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} out of tolerance; worst at {i}: "
                             f"gpu {got[i]!r} oracle {o64[i]!r}")
    exact = float((out_bits == po.f64_to_bf16_bits(o64)).mean()) if o64.size else 1.0
    assert exact >= min_exact, f"{what}: only {exact:.4f} of outputs equal bf16(oracle)"


SHAPES = [
    # rows, n_q_heads, n_kv_heads, head_dim, rot_dim, ring_len, pos range
    (1, 32, 8, 64, 64, 64, (0, 1)),          # full rotation, position 0 (identity rotation)
    (3, 16, 4, 128, 64, 16, (0, 4096)),      # partial rotation, ring wrap
    (16, 32, 8, 64, 32, 1024, (0, 1024)),    # 16 streams
    (5, 8, 2, 128, 0, 7, (100, 200)),        # no rotation, odd ring
    (2, 4, 4, 256, 256, 3, (1 << 20, (1 << 20) + 50)),  # large position, widest head
    (4, 6, 2, 96, 48, 8, (-20, 20)),         # head_dim 96; negative positions
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"r{s[0]}_q{s[1]}_kv{s[2]}_hd{s[3]}_rot{s[4]}_L{s[5]}")
def test_qknorm_rope_kv_parity(q, shape):
    rows, nq, nkv, hd, rot, L, (plo, phi) = shape
    cid = hash(shape) % 1000
    base, eps = 1.0e6 if hd == 128 else 1.0e4, 1e-5
    qf = synth.make_f32(rows, nq * hd, 2.0, config_id=cid, tensor_id=1)
    kf = synth.make_f32(rows, nkv * hd, 2.0, config_id=cid, tensor_id=2)
    vf = synth.make_f32(rows, nkv * hd, 1.0, config_id=cid, tensor_id=3)
    qw = synth.make_bf16((hd,), 0.5, 1.5, config_id=cid, tensor_id=4)
    kw = synth.make_bf16((hd,), 0.5, 1.5, config_id=cid, tensor_id=5)
    pos = synth.make_pos(rows, plo, phi, config_id=cid, tensor_id=6)
    sentinel = 0x1234
    k_ring = torch.full((rows, L, nkv * hd), sentinel, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    v_ring = torch.full((rows, L, nkv * hd), sentinel, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    # q with a row stride wider than its heads, to check ldq
    q_wide = torch.zeros(rows, nq * hd + 64, device="cuda")
    q_wide[:, :nq * hd] = torch.from_numpy(qf).cuda()
    q_out = q.qattn_qknorm_rope_kv(q_wide[:, :nq * hd], torch.from_numpy(kf).cuda(), torch.from_numpy(vf).cuda(),
                                   nq, nkv, hd, rot, base, eps, bf16_dev(qw), bf16_dev(kw),
                                   torch.from_numpy(pos).cuda(), k_ring, v_ring)
    torch.cuda.synchronize()
    q64, k64, v64 = po.qk_norm_rope(qf.astype(np.float64), kf.astype(np.float64), vf.astype(np.float64), qw, kw,
                                    pos, hd, rot, float(np.float32(base)), float(np.float32(eps)))
    check_bf16(bits_host(q_out), q64, "q_out")
    kr, vr = bits_host(k_ring), bits_host(v_ring)
    for r in range(rows):
        s = int(pos[r]) % L
        check_bf16(kr[r, s], k64[r], f"k ring r{r}")
        # v is only rounded: bit-exact
        assert np.array_equal(vr[r, s], po.f64_to_bf16_bits(v64[r])), f"v ring r{r}"
        others = [j for j in range(L) if j != s]
        assert (kr[r, others] == sentinel).all() and (vr[r, others] == sentinel).all(), "a slot outside pos % L"


def test_qknorm_rope_kv_deterministic(q):
    rows, nq, nkv, hd, rot, L = 16, 32, 8, 128, 64, 4
    qf = torch.from_numpy(synth.make_f32(rows, nq * hd, config_id=7, tensor_id=1)).cuda()
    kf = torch.from_numpy(synth.make_f32(rows, nkv * hd, config_id=7, tensor_id=2)).cuda()
    vf = torch.from_numpy(synth.make_f32(rows, nkv * hd, config_id=7, tensor_id=3)).cuda()
    w = bf16_dev(synth.make_bf16((hd,), 0.5, 1.5, config_id=7, tensor_id=4))
    pos = torch.from_numpy(synth.make_pos(rows, 0, 100000, config_id=7)).cuda()
    outs = []
    for _ in range(2):
        kr = torch.zeros(rows, L, nkv * hd, dtype=torch.bfloat16, device="cuda")
        vr = torch.zeros_like(kr)
        qo = q.qattn_qknorm_rope_kv(qf, kf, vf, nq, nkv, hd, rot, 1e6, 1e-6, w, w, pos, kr, vr)
        outs.append((bits_host(qo), bits_host(kr), bits_host(vr)))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
    # a stream's result does not depend on the other streams
    one = torch.zeros(1, L, nkv * hd, dtype=torch.bfloat16, device="cuda")
    one_v = torch.zeros_like(one)
    qo1 = q.qattn_qknorm_rope_kv(qf[5:6], kf[5:6], vf[5:6], nq, nkv, hd, rot, 1e6, 1e-6, w, w, pos[5:6], one, one_v)
    assert np.array_equal(bits_host(qo1)[0], outs[0][0][5])
    assert np.array_equal(bits_host(one)[0], outs[0][1][5])


RESID_SHAPES = [(1, 2048), (3, 1000), (16, 2560), (40, 64), (2, 1), (1, 8192), (7, 4099), (2, 20000), (3, 8200)]


@pytest.mark.parametrize("rows,n", RESID_SHAPES)
def test_resid_rmsnorm_parity(q, rows, n):
    cid = rows * 100000 + n
    y = synth.make_f32(rows, n, 0.5, config_id=cid, tensor_id=1)
    r = synth.make_bf16((rows, n), config_id=cid, tensor_id=2)
    gamma = synth.make_bf16((n,), 0.5, 1.5, config_id=cid, tensor_id=3)
    eps = 1e-5
    y_wide = torch.zeros(rows, n + 8, device="cuda")
    y_wide[:, :n] = torch.from_numpy(y).cuda()
    resid = bf16_dev(r)
    out = q.qresid_rmsnorm(y_wide[:, :n], resid, bf16_dev(gamma), eps)
    torch.cuda.synchronize()
    r64, o64 = po.resid_rms_norm(r, y.astype(np.float64), gamma, float(np.float32(eps)))
    assert np.array_equal(bits_host(resid), r64), "stored residual"
    check_bf16(bits_host(out), o64, "normed output")


def test_resid_rmsnorm_zero_row(q):
    # a zero residual row with eps > 0 normalises to zeros (no division by zero)
    n = 512
    y = torch.zeros(2, n, device="cuda")
    resid = torch.zeros(2, n, dtype=torch.bfloat16, device="cuda")
    out = q.qresid_rmsnorm(y, resid, torch.ones(n, dtype=torch.bfloat16, device="cuda"), 1e-6)
    assert (bits_host(out) == 0).all() and (bits_host(resid) == 0).all()


def test_resid_rmsnorm_rows_independent(q):
    rows, n = 16, 2048
    y = torch.from_numpy(synth.make_f32(rows, n, config_id=9)).cuda()
    r0 = bf16_dev(synth.make_bf16((rows, n), config_id=9, tensor_id=2))
    g = bf16_dev(synth.make_bf16((n,), 0.5, 1.5, config_id=9, tensor_id=3))
    ra = r0.clone()
    outa = q.qresid_rmsnorm(y, ra, g, 1e-5)
    rb = r0[4:5].clone()
    outb = q.qresid_rmsnorm(y[4:5], rb, g, 1e-5)
    assert np.array_equal(bits_host(outa)[4], bits_host(outb)[0])
    assert np.array_equal(bits_host(ra)[4], bits_host(rb)[0])


# ---- the post-add / next-norm step as the epilogue of the w2 / o matvec
@pytest.mark.parametrize("bits,rows,n,k", [(4, 1, 2048, 8192), (4, 16, 2048, 2048), (6, 5, 100, 192),
                                           (8, 9, 513, 2048), (4, 3, 4096, 576)])
def test_mv_resid_norm_fused(q, bits, rows, n, k):
    cid = bits * 1000 + rows * 10 + n % 7
    w = q.QWeight.from_numpy(synth.make_weight(n, k, bits, config_id=cid, tensor_id=1))
    x = q.bf16_from_bits(synth.make_x(rows, k, config_id=cid, tensor_id=2))
    r0 = synth.make_bf16((rows, n), config_id=cid, tensor_id=3)
    gamma = bf16_dev(synth.make_bf16((n,), 0.5, 1.5, config_id=cid, tensor_id=4))
    eps = 1e-5
    # fused
    rf = bf16_dev(r0)
    out_f = q.qlinear_mv_resid_norm(w, x, rf, gamma, eps)
    # unfused: the matvec, then the post-add / next-norm kernel
    rs = bf16_dev(r0)
    y = q.qlinear_mv_rows(w, x)
    out_s = q.qresid_rmsnorm(y, rs, gamma, eps)
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    # the stored residual is the same decision in the same precision: bit-equal
    assert np.array_equal(bits_host(rf), bits_host(rs))
    # the normed output against the float64 definition on the stored residual
    rb = bits_host(rf)
    # the oracle's post-add / next-norm of the stored residual with nothing more added
    r_same, o64 = po.resid_rms_norm(rb, np.zeros(rb.shape), bits_host(gamma), float(np.float32(eps)))
    assert np.array_equal(r_same, rb)
    check_bf16(bits_host(out_f), o64, "fused normed output")
    check_bf16(bits_host(out_s), o64, "unfused normed output")
    # repeated launches (the tile counter returns to zero) give the same bits
    rf2 = bf16_dev(r0)
    out_f2 = q.qlinear_mv_resid_norm(w, x, rf2, gamma, eps)
    torch.cuda.synchronize()
    assert np.array_equal(bits_host(out_f2), bits_host(out_f)) and np.array_equal(bits_host(rf2), rb)


def test_mv_resid_norm_rows_independent(q):
    n, k, bits = 2048, 2048, 4
    w = q.QWeight.from_numpy(synth.make_weight(n, k, bits, config_id=77, tensor_id=1))
    x = q.bf16_from_bits(synth.make_x(12, k, config_id=77, tensor_id=2))
    r0 = synth.make_bf16((12, n), config_id=77, tensor_id=3)
    gamma = bf16_dev(synth.make_bf16((n,), 0.5, 1.5, config_id=77, tensor_id=4))
    ra = bf16_dev(r0)
    oa = q.qlinear_mv_resid_norm(w, x, ra, gamma, 1e-5)
    rb = bf16_dev(r0[7:8])
    ob = q.qlinear_mv_resid_norm(w, x[7:8].clone(), rb, gamma, 1e-5)
    torch.cuda.synchronize()
    assert np.array_equal(bits_host(oa)[7], bits_host(ob)[0])
    assert np.array_equal(bits_host(ra)[7], bits_host(rb)[0])
