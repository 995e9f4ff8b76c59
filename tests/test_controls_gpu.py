"""Planted controls and cross-process determinism on the GPU.

TensorFold PR #1696 (later revision), "What it adds": every kernel is checked against
a float64 reference with a planted control that must fail; "Checks": the prompt GEMM's
window test uses the decode path's different summation order as its control, and the
RoPE kernels' compiled sub-group width once changed a reply from one process to the
next.  Here:

* a flipped nibble in the device weights must fail the oracle comparison, on exactly
  the row it sits in (decode and prompt GEMM): the parity check can see a one-code
  error;
* the decode matvec and the prompt GEMM sum in different orders: on the same rows
  both are within tolerance of the oracle, and the bit-for-bit comparison that the
  window-cut and N-row tests use tells them apart - it detects an order change;
* two fresh processes running every entry point on the same seeded inputs produce
  the same bytes.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from oracle import qlinear_oracle as orc
from tests import _util as U
from weight_only_bit_mlx_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q():
    from weight_only_bit_mlx_gb300 import qlinear
    assert torch.cuda.is_available()
    return qlinear


def _out_of_tol(y_gpu, y64, A):
    y = y_gpu.detach().float().cpu().numpy().astype(np.float64)
    return np.abs(y - y64) > U.tol(A)


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_flipped_code_fails_parity(q, bits):
    n, k = 256, 2048
    w = U.weight(n, k, bits, config_id=150, tensor_id=bits)
    x = synth.make_x(4, k, config_id=150)
    X = synth.make_x(40, k, config_id=151)
    # the planted mistake: one code of row 77 changed by 2^(bits-1), at the k where row 0
    # of x is largest, written into a copy of the device weights
    r, j = 77, int(np.argmax(np.abs(orc.bf16_bits_to_f64(x[0]))))
    bad = dict(w, wq=w["wq"].copy())
    word, off = (bits * j) // 32, (bits * j) % 32
    assert off + bits <= 32  # the chosen field does not straddle (j is such that it does not for 6 bits)
    bad["wq"][r, word] ^= np.uint32(1 << (off + bits - 1))
    good_d, bad_d = U.dev_weight(w), U.dev_weight(bad)
    y64, A = orc.qlinear_w(x, w)
    Y64, AY = orc.pgemm(X, w)
    # the control: the comparison passes on the true weights...
    assert not _out_of_tol(q.qlinear_mv_rows(good_d, U.dev_x(x)), y64, A).any()
    assert not _out_of_tol(q.qlinear_pgemm(good_d, U.dev_x(X)), Y64, AY).any()
    # ... and fails on exactly the planted row with the flipped code
    bad_mv = _out_of_tol(q.qlinear_mv_rows(bad_d, U.dev_x(x)), y64, A)
    bad_pg = _out_of_tol(q.qlinear_pgemm(bad_d, U.dev_x(X)), Y64, AY)
    assert bad_mv[0, r] and bad_pg[:, r].any()
    assert not np.delete(bad_mv, r, axis=1).any() and not np.delete(bad_pg, r, axis=1).any()


def test_different_order_is_detected_bit_for_bit(q):
    # the decode path's order against the prompt GEMM's: both within the oracle's
    # tolerance, most outputs different in their last bits
    n, k = 2048, 2048
    w = U.weight(n, k, 4, config_id=152)
    X = synth.make_x(16, k, config_id=152)
    wd, Xd = U.dev_weight(w), U.dev_x(X)
    y_mv = q.qlinear_mv_rows(wd, Xd)
    y_pg = q.qlinear_pgemm(wd, Xd)
    torch.cuda.synchronize()
    y64, A = orc.qlinear_w(X, w)
    U.assert_close(y_mv, y64, A, "decode order")
    U.assert_close(y_pg, y64, A, "prompt-GEMM order")
    assert not torch.equal(y_mv, y_pg)
    assert (y_mv != y_pg).float().mean().item() > 0.5


def test_two_processes_give_the_same_bytes():
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    runs = []
    for _ in range(2):
        res = subprocess.run([sys.executable, "-m", "tests._determinism_child"], cwd=ROOT, env=env,
                             capture_output=True, text=True, timeout=600)
        assert res.returncode == 0, res.stderr[-2000:]
        runs.append(json.loads(res.stdout.strip().splitlines()[-1]))
    assert runs[0]["status"] == 0
    assert len(runs[0]) == 9 * 3 + 4  # nine entry points at three widths, three more, the status
    assert runs[0] == runs[1], {k: (runs[0][k], runs[1].get(k)) for k in runs[0] if runs[0][k] != runs[1].get(k)}
