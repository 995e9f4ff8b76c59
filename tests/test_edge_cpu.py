"""CPU checks of the inputs the degenerate-weight GPU tests build: the vectorised
test packer agrees with the plain loop packer (and with the oracle's unpacker), and
every band of an edge weight dequantizes to what its name says."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import qlinear_oracle as orc
from tests import _util as U
from tests.test_edge_gpu import BAND, edge_weight
from tests.test_oracle_pins import pack_rows


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_vector_packer_matches_loop_packer(bits):
    g = np.random.default_rng(bits)
    q = g.integers(0, 1 << bits, size=(3, 192))
    packed = U.pack_codes(q, bits)
    assert np.array_equal(packed, pack_rows(q, bits))
    assert np.array_equal(orc.unpack_q(packed, bits, 192), q)


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_edge_weight_bands(bits):
    k = 256
    w = edge_weight(k, bits, 7, 1)
    wd = orc.dequant(w["wq"], w["scales"], w["biases"], bits, k)
    q = orc.unpack_q(w["wq"], bits, k)
    zero, cancel, half, rnd = (slice(i * BAND, (i + 1) * BAND) for i in range(4))
    assert not wd[zero].any() and not q[zero].any()
    assert not wd[cancel].any() and q[cancel].min() >= 1        # weights vanish, codes do not
    even = np.concatenate([np.arange(g * 64, g * 64 + 64) for g in range(0, k // 64, 2)])
    odd = np.setdiff1d(np.arange(k), even)
    assert not wd[half][:, even].any() and np.abs(wd[half][:, odd]).min() >= 0
    assert np.count_nonzero(wd[half][:, odd]) > 0.9 * wd[half][:, odd].size
    assert np.count_nonzero(wd[rnd]) > 0.9 * wd[rnd].size
