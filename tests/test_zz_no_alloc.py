"""ito_linear_fwd_noalloc, the forward Linear entry point for callers that
cannot allocate device memory while they run (it uses a scratch array built
into the library instead of a caller workspace), against ito_linear_fwd, the
workspace entry point, and against the CPU oracle: bit-identical outputs on two
calls in a row, and a clear rejection of sizes beyond the built-in scratch.

This file is collected last on purpose, so that a run that stops at the first
failure has already run every other test; it also passes on its own."""
import numpy as np
import pytest

import oracle as O
from gpu_util import import_ito

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _same(ref, got):
    for r, g in zip(ref, got):
        assert np.array_equal(r.cpu().numpy(), g.cpu().numpy())


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    ito = import_ito()
    import torch
    rng = np.random.default_rng(77)
    # two consecutive calls with different shapes and data: the second must not
    # see anything the first left in the shared scratch
    for (B, IC, OC, relu) in ((129, 300, 257, 1), (256, 784, 1024, 0)):
        x = rng.integers(-128, 128, (B, IC)).astype(np.int8)
        W = rng.integers(-127, 128, (OC, IC)).astype(np.int8)
        xd, Wd = _dev(x), _dev(W)
        ref = ito.ito_linear_fwd(xd, Wd, relu)
        out = (torch.empty((B, OC), dtype=torch.int32, device="cuda"),
               torch.zeros(1, dtype=torch.int32, device="cuda"),
               torch.zeros(1, dtype=torch.int32, device="cuda"),
               torch.empty((B, OC), dtype=torch.int8, device="cuda"))
        got = ito.ito_linear_fwd_noalloc(xd, Wd, relu, out=out)
        torch.cuda.synchronize()
        _same(ref, got)
        y32 = O.linear_fwd(x, W)
        y8, shift, mx = O.requant(y32, relu=bool(relu))
        assert np.array_equal(got[0].cpu().numpy(), y32)
        assert (int(got[1].cpu().numpy()[0]) & 0xFFFFFFFF) == mx
        assert int(got[2].cpu().numpy()[0]) == shift
        assert np.array_equal(got[3].cpu().numpy(), y8)
    assert ito.ito_get_error() == 0


def test_noalloc_rejects_sizes_beyond_the_scratch():
    ito = import_ito()
    import torch
    B, IC, OC = 4096, 4096, 8        # bf16 copy of x alone is 32 MiB > 16 MiB
    x = torch.zeros((B, IC), dtype=torch.int8, device="cuda")
    W = torch.zeros((OC, IC), dtype=torch.int8, device="cuda")
    with pytest.raises(ito.ItoError) as ei:
        ito.ito_linear_fwd_noalloc(x, W, 0)
    assert ei.value.code == ito.ITO_ERR_SHAPE
    assert "scratch" in str(ei.value)
