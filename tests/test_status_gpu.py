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
