"""The CUDA path's decision uniforms against the oracle's, bit for bit
(isd_decision_uniforms, include/isd_debug.h): the two Philox4x64-10
implementations share no code, and the decisions of every kernel use the
device function this call exposes.  A sweep over sequences, positions and
purposes, under random 64-bit seeds and offsets and at the extremes of the
counter words."""
import numpy as np
import pytest
import torch

import oracle
from speculative_verify_accept_02_b300.api import isd_decision_uniforms

pytestmark = pytest.mark.gpu


def test_uniforms_equal_the_oracle():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    rng = np.random.default_rng(5)
    rows = [(i, k, t) for i in range(0, 300, 7) for k in range(1, 34, 4) for t in range(4)]
    rows += [(2**40 + 3, 1, 0), (2**62, 32, 3), (0, 0, 0), (5, 2**40, 2)]
    ctr = np.array(rows, dtype=np.int64)
    for seed, offset in [(0, 0), (1234, 5)] + [tuple(int(v) for v in rng.integers(0, 2**63, 2)) for _ in range(3)]:
        got = isd_decision_uniforms(seed, offset, torch.from_numpy(ctr).cuda()).cpu().numpy()
        want = np.array([oracle.uniform(seed, offset, int(i), int(k), int(t)) for i, k, t in rows], np.float32)
        assert np.array_equal(got, want), (seed, offset, np.flatnonzero(got != want)[:5])
