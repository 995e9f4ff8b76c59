"""qlinear_pgemm_noalloc: the prompt GEMM for callers that cannot allocate device
memory when they call (device memory owned by another allocator or held to a fixed
budget, or no tolerance for the device-wide synchronization of growing a scratch
buffer).  Its scratch is a fixed static device array, so its output is checked
against qlinear_pgemm (which uses the library's growable buffer) through the C ABI,
on two calls in a row that share the array.

Kept in a file that pytest collects last, so a run that stops at the first failure
has already run every other test; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from oracle import qlinear_oracle as orc
from tests import _util as U
from weight_only_bit_mlx_gb300 import synth

pytestmark = pytest.mark.gpu


def _noalloc(q, w, X, Y):
    return q.LIB.qlinear_pgemm_noalloc(ctypes.byref(w.c), X.data_ptr(), int(X.shape[0]), X.stride(0),
                                       Y.data_ptr(), Y.stride(0), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_pgemm_on_two_calls_in_a_row():
    from weight_only_bit_mlx_gb300 import qlinear as q

    cases = [(4, 300, 1000, 2048), (8, 2000, 512, 512)]
    data = []
    for i, (bits, m, n, k) in enumerate(cases):
        w = U.weight(n, k, bits, config_id=80, tensor_id=i)
        X = synth.make_x(m, k, config_id=80, tensor_id=100 + i)
        wd, Xd = U.dev_weight(w), U.dev_x(X)
        Y_ref = q.qlinear_pgemm(wd, Xd)
        data.append((w, X, wd, Xd, Y_ref))
    torch.cuda.synchronize()
    outs = []
    for w, X, wd, Xd, _ in data:  # two calls in a row, both through the fixed array
        Y = torch.full((Xd.shape[0], wd.n), float("nan"), device="cuda")
        assert _noalloc(q, wd, Xd, Y) == q.QL_OK
        outs.append(Y)
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    for (w, X, wd, Xd, Y_ref), Y in zip(data, outs):
        # the same kernels on the same inputs: the same bits as qlinear_pgemm
        assert torch.equal(Y, Y_ref)
        # and within the library's tolerance of the float64 oracle
        y64, A = orc.pgemm(X, w)
        U.assert_close(Y, y64, A, "qlinear_pgemm_noalloc")


def test_noalloc_rejects_problems_beyond_its_fixed_scratch():
    from weight_only_bit_mlx_gb300 import qlinear as q

    # k = 8192: 384 split-sum values per row, so m = 3000 needs 1,152,000 > 1,048,576
    w = U.dev_weight(U.weight(64, 8192, 4, config_id=81))
    X = torch.zeros(3000, 8192, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(3000, 64, device="cuda")
    assert _noalloc(q, w, X, Y) == q.QL_ERR_TOO_LARGE
    assert "fixed scratch" in q.qlinear_strerror(q.QL_ERR_TOO_LARGE)
    # the largest m that fits (2730 * 384 values), on seeded non-zero rows: the same bits
    # as qlinear_pgemm, so the scratch pitch holds at the size limit
    Xs = U.dev_x(synth.make_x(2730, 8192, config_id=81, tensor_id=100))
    Ys = torch.full((2730, 64), float("nan"), device="cuda")
    assert _noalloc(q, w, Xs, Ys) == q.QL_OK
    Y_ref = q.qlinear_pgemm(w, Xs)
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    assert torch.equal(Ys, Y_ref)
