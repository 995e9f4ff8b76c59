"""Prompt-window GEMM on the GPU: parity with the float64 oracle and bit-exact
invariance of every row across window cuts (TensorFold PR #1696, later revision,
"What it adds" > "Prompt GEMM": blocks added in order so a row's sum does not
depend on how the prompt is cut; "Checks": windows of 64, 128, 256 and a ragged
cut, every row alone equal to the row in a window)."""
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


@pytest.fixture(scope="module")
def prompt(q):
    # prefill pgemm: X bf16 [1024, 2048] ~ N(0, 1); W 2048 -> 8192, 4-bit g64
    w = U.weight(8192, 2048, 4, config_id=3, tensor_id=0)
    X = synth.make_x(1024, 2048, config_id=3)
    wd, Xd = U.dev_weight(w), U.dev_x(X)
    Y = q.qlinear_pgemm(wd, Xd)
    torch.cuda.synchronize()
    return w, X, wd, Xd, Y


def test_prompt_gemm_against_oracle(prompt):
    w, X, wd, Xd, Y = prompt
    y64, A = orc.pgemm(X, w)
    U.assert_close(Y, y64, A, "pgemm 1024x2048x8192")


@pytest.mark.parametrize("cut", [[64] * 16, [128] * 8, [256] * 4, [100, 300, 624]],
                         ids=["w64", "w128", "w256", "ragged"])
def test_window_cuts_bit_exact(q, prompt, cut):
    w, X, wd, Xd, Y = prompt
    lo = 0
    for m in cut:
        Yw = q.qlinear_pgemm(wd, Xd[lo:lo + m])
        assert torch.equal(Yw, Y[lo:lo + m]), f"window [{lo}, {lo + m}) differs"
        lo += m
    assert lo == 1024


def test_rows_alone_bit_exact(q, prompt):
    w, X, wd, Xd, Y = prompt
    for r in [0, 1, 127, 128, 129, 500, 1023]:
        assert torch.equal(q.qlinear_pgemm(wd, Xd[r:r + 1]), Y[r:r + 1]), f"row {r}"


@pytest.mark.parametrize("bits", [4, 6, 8])
@pytest.mark.parametrize("m,n,k", [(77, 200, 64), (130, 1000, 192), (300, 256, 8192), (256, 512, 2048),
                                   (1, 128, 4096)])
def test_shapes_against_oracle(q, bits, m, n, k):
    w = U.weight(n, k, bits, config_id=60, tensor_id=bits)
    X = synth.make_x(m, k, config_id=60)
    wd, Xd = U.dev_weight(w), U.dev_x(X)
    Y = q.qlinear_pgemm(wd, Xd)
    torch.cuda.synchronize()
    y64, A = orc.pgemm(X, w)
    U.assert_close(Y, y64, A, f"pgemm bits={bits} m={m} n={n} k={k}")
    # ragged cut of the same rows
    if m > 3:
        cut = m // 3
        Y2 = torch.cat([q.qlinear_pgemm(wd, Xd[:cut]), q.qlinear_pgemm(wd, Xd[cut:])])
        assert torch.equal(Y2, Y)


def test_strided_input_and_output(q):
    n, k, m = 384, 1024, 200
    w = U.dev_weight(U.weight(n, k, 4, config_id=61))
    Xw = U.dev_x(synth.make_x(m, k + 128, config_id=61))
    Xs = Xw[:, 128:]
    Yref = q.qlinear_pgemm(w, Xs.contiguous())
    Yout = torch.full((m, n + 5), float("nan"), device="cuda")
    q.qlinear_pgemm(w, Xs, Y=Yout[:, :n])
    assert torch.equal(Yout[:, :n], Yref)
    assert torch.isnan(Yout[:, n:]).all()


def test_empty_window(q):
    w = U.dev_weight(U.weight(128, 128, 4, config_id=62))
    Y = q.qlinear_pgemm(w, torch.empty(0, 128, dtype=torch.bfloat16, device="cuda"))
    assert Y.shape == (0, 128)


def test_row_independence_of_other_rows(q):
    # changing other rows of the window must not change a row's bits
    n, k = 256, 2048
    w = U.dev_weight(U.weight(n, k, 4, config_id=63))
    X = U.dev_x(synth.make_x(128, k, config_id=63))
    Y = q.qlinear_pgemm(w, X)
    X2 = X.clone()
    X2[1::2] = X2[1::2] * 3.0
    Y2 = q.qlinear_pgemm(w, X2)
    assert torch.equal(Y[0::2], Y2[0::2])


@pytest.mark.parametrize("bits,k", [(4, 6144), (6, 8192)])
def test_several_tiles_per_cta_long_k(q, bits, k):
    """More 128 x 256 tiles than SMs with a long k (5-6 bias blocks per tile): every
    CTA walks several tiles, and the result must equal windows of 256 rows (one tile
    each) bit for bit, with no timeout, and match the oracle on sampled rows."""
    n, m = 2048, 4864  # 16 x 19 = 304 tiles
    w = U.weight(n, k, bits, config_id=90, tensor_id=bits)
    X = synth.make_x(m, k, config_id=90, tensor_id=1000 + bits)
    wd, Xd = U.dev_weight(w), U.dev_x(X)
    Y = q.qlinear_pgemm(wd, Xd)
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    Yw = torch.empty_like(Y)
    for lo in range(0, m, 256):
        q.qlinear_pgemm(wd, Xd[lo:lo + 256], Y=Yw[lo:lo + 256])
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    assert torch.equal(Yw, Y)
    rows = np.random.default_rng(k).choice(m, size=24, replace=False)
    rows.sort()
    y64, A = orc.pgemm(X[rows], w)
    U.assert_close(Y[torch.from_numpy(rows).cuda()], y64, A, f"pgemm several tiles bits={bits} k={k}")


@pytest.mark.parametrize("bits,m,n,k", [(4, 2300, 1000, 1024), (6, 2049, 333, 2048), (8, 2200, 520, 512),
                                        (4, 2050, 130, 64), (6, 2048, 256, 192), (8, 2100, 300, 8192)])
def test_large_windows_ragged_against_windows(q, bits, m, n, k):
    # From 2048 rows on the codes are converted once per call; below, inside the GEMM.
    # Ragged m and n (partial row and channel tiles), one group (k = 64: three
    # split-sum columns), three groups and 128 groups on the first path against the same
    # rows cut into windows of 512 (the second path), bit for bit, and sampled rows
    # against the float64 oracle.
    w = U.weight(n, k, bits, config_id=62, tensor_id=bits)
    X = synth.make_x(m, k, config_id=62)
    wd, Xd = U.dev_weight(w), U.dev_x(X)
    Y = q.qlinear_pgemm(wd, Xd)
    Yw = torch.cat([q.qlinear_pgemm(wd, Xd[lo:lo + 512]) for lo in range(0, m, 512)])
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    assert torch.equal(Yw, Y), "windows of 512 differ from one call"
    rows = np.sort(np.random.default_rng(bits).choice(m, size=24, replace=False))
    rows[-1] = m - 1  # the last, partial row tile
    y64, A = orc.pgemm(X[rows], w)
    U.assert_close(Y[torch.from_numpy(rows).cuda()], y64, A, f"pgemm bits={bits} m={m} n={n} k={k}")


def test_back_to_back_large_calls_bit_exact(q):
    # Calls of 2048 rows and more convert their codes in a kernel that may start while
    # the previous call's GEMM still runs its last tiles (calls alternate between two
    # buffers of converted codes), and the row sums wait for the kernel before them.
    # Here large calls follow each other with no synchronization, on weights of other
    # shapes and widths, and one call's fused epilogue writes the next call's X.  Every
    # output must equal the same call made alone.
    m, eps = 2048, 1e-5
    specs = [(8192, 8192, 4), (4096, 2048, 6), (2048, 4096, 8), (8192, 2048, 4), (1000, 1024, 8)]
    ws = [U.dev_weight(U.weight(n, k, b, config_id=64, tensor_id=i)) for i, (n, k, b) in enumerate(specs)]
    X8 = U.dev_x(synth.make_x(m, 8192, config_id=64))
    X2 = U.dev_x(synth.make_x(m, 2048, config_id=65))
    X4 = U.dev_x(synth.make_x(m, 4096, config_id=66))
    r0 = U.dev_x(synth.make_bf16((m, 4096), config_id=64, tensor_id=9))
    gamma = U.dev_x(synth.make_bf16((4096,), 0.5, 1.5, config_id=64, tensor_id=10))

    def run():
        r = r0.clone()
        ys = [q.qlinear_pgemm(ws[0], X8)]
        ys.append(q.qlinear_pgemm(ws[1], X2))
        h = q.qlinear_pgemm_resid_norm(ws[1], X2, r, gamma, eps)  # h: [m, 4096] bf16
        ys.append(q.qlinear_pgemm(ws[2], h))                       # X written just before
        ys.append(q.qlinear_pgemm(ws[3], X2))
        ys.append(q.qlinear_pgemm(ws[4], X2[:, :1024].contiguous()))
        ys.append(q.qlinear_pgemm(ws[2], X4))
        return ys, h, r

    ys, h, r = run()  # back to back
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    ref = []
    rr = r0.clone()
    for fn in [lambda: q.qlinear_pgemm(ws[0], X8), lambda: q.qlinear_pgemm(ws[1], X2),
               lambda: q.qlinear_pgemm_resid_norm(ws[1], X2, rr, gamma, eps)]:
        ref.append(fn())
        torch.cuda.synchronize()
    h_ref = ref.pop()
    for w, x in [(ws[2], h_ref), (ws[3], X2), (ws[4], X2[:, :1024].contiguous()), (ws[2], X4)]:
        ref.append(q.qlinear_pgemm(w, x))
        torch.cuda.synchronize()
    assert torch.equal(h.view(torch.int16), h_ref.view(torch.int16)), "fused epilogue output"
    assert torch.equal(r.view(torch.int16), rr.view(torch.int16)), "stored residual"
    for i, (a, b) in enumerate(zip(ys, ref)):
        assert torch.equal(a, b), f"call {i} differs from the same call made alone"


def test_mixed_calls_back_to_back_bit_exact(q):
    # Every call's row-sum pre-pass, every large call's code conversion and every GEMM are
    # launched with programmatic dependent launch, each waiting for the kernel before it
    # before it reads what that kernel may have written.  Here windows of 128 and 600 rows,
    # the no-alloc entry point, large calls (with and without the conversion's early start)
    # and a fused epilogue whose output is the next call's X follow each other with no
    # synchronization.  Every output must equal the same call made alone.
    eps = 1e-5
    w_a = U.dev_weight(U.weight(4096, 2048, 4, config_id=66, tensor_id=1))
    w_b = U.dev_weight(U.weight(2048, 4096, 6, config_id=66, tensor_id=2))
    w_c = U.dev_weight(U.weight(1000, 2048, 8, config_id=66, tensor_id=3))
    X = U.dev_x(synth.make_x(2048, 2048, config_id=67))
    r0 = U.dev_x(synth.make_bf16((600, 4096), config_id=66, tensor_id=9))
    gamma = U.dev_x(synth.make_bf16((4096,), 0.5, 1.5, config_id=66, tensor_id=10))

    def calls(sync):
        out = []

        def step(fn):
            out.append(fn())
            if sync:
                torch.cuda.synchronize()

        r = r0.clone()
        step(lambda: q.qlinear_pgemm(w_a, X[:128]))
        step(lambda: q.qlinear_pgemm(w_c, X))                                   # large, after a small call
        step(lambda: q.qlinear_pgemm_resid_norm(w_a, X[:600], r, gamma, eps))  # h: [600, 4096]
        step(lambda: q.qlinear_pgemm(w_b, out[-1]))                             # X written just before
        step(lambda: q.qlinear_pgemm_noalloc(w_c, X[:128], torch.empty(128, 1000, device=X.device)))
        step(lambda: q.qlinear_pgemm(w_a, X))                                   # large, after a no-alloc call
        step(lambda: q.qlinear_pgemm(w_c, X))                                   # large after large
        step(lambda: q.qlinear_pgemm(w_a, X[100:228]))                          # small after large
        return out, r

    got, r_got = calls(sync=False)
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    ref, r_ref = calls(sync=True)
    assert q.qlinear_last_error() == q.QL_OK
    assert torch.equal(r_got.view(torch.int16), r_ref.view(torch.int16)), "stored residual"
    for i, (a, b) in enumerate(zip(got, ref)):
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), f"call {i} differs from the same call made alone"


@pytest.mark.parametrize("m", [100, 2100])
def test_multi_equals_separate_calls(q, m):
    # qlinear_pgemm_multi forms the split row sums of X once for all its weights; every
    # output must equal the weight's own qlinear_pgemm call bit for bit, below and above
    # the row count from which the codes are converted once per call, with weights of
    # other widths and sizes, and outputs with padded pitches.
    k = 2048
    specs = [(1024, 4), (256, 6), (320, 8), (1024, 4)]
    ws = [U.dev_weight(U.weight(n, k, b, config_id=68, tensor_id=i)) for i, (n, b) in enumerate(specs)]
    X = U.dev_x(synth.make_x(m, k, config_id=69))
    X2 = U.dev_x(synth.make_x(m, k, config_id=70))
    Ys = [torch.full((m, n + 8 * i), float("nan"), device=X.device)[:, :n] for i, (n, _) in enumerate(specs)]
    # below 2048 rows the GEMMs of one call run beside each other; a second call on
    # another X follows at once (its row sums replace the first call's)
    got = q.qlinear_pgemm_multi(ws, X, Ys)
    got2 = q.qlinear_pgemm_multi(ws[::-1], X2)
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    for i, w in enumerate(ws):
        ref = q.qlinear_pgemm(w, X)
        ref2 = q.qlinear_pgemm(w, X2)
        torch.cuda.synchronize()
        assert torch.equal(got[i], ref), f"weight {i} differs from its own call"
        assert torch.equal(got2[len(ws) - 1 - i], ref2), f"weight {i} of the second call differs"
    one = q.qlinear_pgemm_multi(ws[:1], X)[0]
    torch.cuda.synchronize()
    assert torch.equal(one, got[0])
    rows = np.array([0, m // 2, m - 1])
    y64, A = orc.pgemm(synth.make_x(m, k, config_id=69)[rows], U.weight(320, k, 8, config_id=68, tensor_id=2))
    U.assert_close(got[2][torch.from_numpy(rows).cuda()], y64, A, f"pgemm_multi m={m}")
