"""Failure detection on the GPU without a fault: a kernel's bounded mbarrier
wait runs out on a barrier nothing completes, the device error word reports
ITO_ERR_TIMEOUT to the host, and the context stays usable (a contraction
right after matches the oracle)."""
import time

import numpy as np
import pytest

import oracle as O
from gpu_util import import_ito

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    ito = import_ito()
    assert ito.ito_get_error() == 0
    t0 = time.monotonic()
    ito.ito_selftest_wait_timeout()
    waited = time.monotonic() - t0
    assert 1.5 < waited < 30.0
    assert ito.ito_get_error() == ito.ITO_ERR_TIMEOUT
    assert ito.ito_get_error() == 0            # the read clears the word
    rng = np.random.default_rng(11)
    x = rng.integers(-127, 128, (300, 700)).astype(np.int8)
    W = rng.integers(-127, 128, (260, 700)).astype(np.int8)
    y32, _, _, _ = ito.ito_linear_fwd(torch.from_numpy(x).cuda(), torch.from_numpy(W).cuda(), 1)
    assert np.array_equal(y32.cpu().numpy(), O.linear_fwd(x, W))
    assert ito.ito_get_error() == 0
