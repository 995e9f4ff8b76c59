"""The bounded-wait failure path, exercised without a fault: a CTA waits on a
barrier that nothing completes, its wait gives up after a short budget, and the
status word reports QL_ERR_TIMEOUT while the context stays usable."""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_wait_probe_times_out_and_context_survives():
    from weight_only_bit_mlx_gb300 import qlinear as q
    from tests import _util as U
    from weight_only_bit_mlx_gb300 import synth

    assert q.qlinear_last_error() == q.QL_OK
    q.qlinear_wait_probe(2_000_000)  # 2 ms
    assert q.qlinear_last_error() == q.QL_ERR_TIMEOUT
    assert q.qlinear_last_error() == q.QL_OK  # read clears it
    # the context is still healthy
    w = U.dev_weight(U.weight(64, 128, 4, config_id=70))
    y = q.qlinear_mv(w, U.dev_x(synth.make_x(1, 128, config_id=70))[0])
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    assert q.qlinear_last_error() == q.QL_OK


def test_fused_resid_norm_after_timeout_status():
    """Reading a non-zero status also re-arms the fused post-add / next-norm epilogue
    (its tile counter is zeroed).  The fused call made after the timeout must give the
    same bits as the same call made before it, twice in a row; its stored residual is
    bit-equal to the unfused pair's (the same rounding decision in the same precision)."""
    import numpy as np
    from weight_only_bit_mlx_gb300 import qlinear as q
    from weight_only_bit_mlx_gb300 import synth

    n, k = 1024, 2048
    w = q.QWeight.from_numpy(synth.make_weight(n, k, 4, config_id=71, tensor_id=1))
    x = q.bf16_from_bits(synth.make_x(3, k, config_id=71, tensor_id=2))
    r0 = q.bf16_from_bits(synth.make_bf16((3, n), config_id=71, tensor_id=3))
    gamma = q.bf16_from_bits(synth.make_bf16((n,), 0.5, 1.5, config_id=71, tensor_id=4))
    rb = r0.clone()
    out_before = q.qlinear_mv_resid_norm(w, x, rb, gamma, 1e-5)
    torch.cuda.synchronize()
    assert q.qlinear_last_error() == q.QL_OK
    rs = r0.clone()
    q.qresid_rmsnorm(q.qlinear_mv_rows(w, x), rs, gamma, 1e-5)
    q.qlinear_wait_probe(1_000_000)  # 1 ms
    assert q.qlinear_last_error() == q.QL_ERR_TIMEOUT
    for _ in range(2):
        rf = r0.clone()
        out_f = q.qlinear_mv_resid_norm(w, x, rf, gamma, 1e-5)
        torch.cuda.synchronize()
        assert q.qlinear_last_error() == q.QL_OK
        assert torch.equal(rf.view(torch.int16), rs.view(torch.int16))
        assert torch.equal(rf.view(torch.int16), rb.view(torch.int16))
        assert np.array_equal(out_f.view(torch.int16).cpu().numpy(), out_before.view(torch.int16).cpu().numpy())
