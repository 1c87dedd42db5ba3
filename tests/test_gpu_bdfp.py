"""Blocked-DFP on the GPU against the CPU oracle ("Mixed Precision Training of
Convolutional Neural Networks using Integer Operations", section 3:
Blocked-DFP; section 4: FP32 outputs): conversions block by block and the
blocked linear forward, compared bit for bit (mantissas, exponents, floats)."""
import numpy as np
import pytest

import oracle as O
from gpu_util import import_ito

pytestmark = pytest.mark.gpu

rng = np.random.default_rng(6060)


@pytest.fixture(scope="module")
def ito():
    return import_ito()


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _scaled(rows, cols, block):
    """Normal values whose scale changes from block to block by up to 2^40."""
    nb = (cols + block - 1) // block
    sc = np.exp2(rng.integers(-20, 21, (rows, nb))).astype(np.float32)
    return (rng.standard_normal((rows, cols)) * np.repeat(sc, block, axis=1)[:, :cols]).astype(np.float32)


@pytest.mark.parametrize("rows,cols,block", [(3, 200, 64), (5, 1000, 128), (2, 7, 3), (1, 4096, 512), (64, 33, 33)])
def test_bdfp_conversions(ito, rows, cols, block):
    f = _scaled(rows, cols, block)
    f[0, 0] = 0.0
    if cols > block:
        f[-1, :block] = 0.0        # an all-zero block gets exponent 0
    m, e = ito.ito_bdfp16_from_float(_dev(f), block)
    mref, eref = O.bdfp_from_float(f, block)
    assert np.array_equal(m.cpu().numpy(), mref)
    assert np.array_equal(e.cpu().numpy().astype(np.int32), eref)
    back = ito.ito_bdfp16_to_float(m, e, block)
    assert np.array_equal(back.cpu().numpy(), O.bdfp_to_float(mref, eref, block))
    assert ito.ito_get_error() == 0


@pytest.mark.parametrize("B,IC,OC,block", [(64, 512, 128, 64), (300, 1000, 130, 64), (129, 640, 257, 256),
                                           (2048, 2048, 2048, 512), (16, 100, 8, 128)])
def test_bdfp_linear_fwd(ito, B, IC, OC, block):
    nb = (IC + block - 1) // block
    x = rng.integers(-32767, 32768, (B, IC)).astype(np.int16)
    W = rng.integers(-32767, 32768, (OC, IC)).astype(np.int16)
    ex = rng.integers(-40, 0, (B, nb)).astype(np.int8)
    ew = rng.integers(-40, 0, (OC, nb)).astype(np.int8)
    y = ito.ito_bdfp16_linear_fwd_f32(_dev(x), _dev(ex), _dev(W), _dev(ew), block)
    yref = O.bdfp_linear_fwd_f32(x, ex.astype(np.int32), W, ew.astype(np.int32), block)
    assert np.array_equal(y.cpu().numpy(), yref)
    assert ito.ito_get_error() == 0


def test_bdfp_from_float_then_linear_matches_float64(ito):
    """End to end: float tensors whose blocks span 2^40 in scale, converted and
    contracted; within the relative error of 15-bit mantissas of a float64
    product (a sanity bound, the bit-exact pins are above)."""
    B, IC, OC, block = 96, 1024, 80, 128
    x = _scaled(B, IC, block)
    W = _scaled(OC, IC, block)
    xm, xe = ito.ito_bdfp16_from_float(_dev(x), block)
    wm, we = ito.ito_bdfp16_from_float(_dev(W), block)
    y = ito.ito_bdfp16_linear_fwd_f32(xm, xe, wm, we, block).cpu().numpy().astype(np.float64)
    ref = x.astype(np.float64) @ W.astype(np.float64).T
    scale = np.abs(x.astype(np.float64)) @ np.abs(W.astype(np.float64)).T
    assert (np.abs(y - ref) <= 2.0 ** -13 * scale + 1e-30).all()


def test_bdfp_bad_block(ito):
    import torch
    x = torch.zeros((4, 128), dtype=torch.int16, device="cuda")
    e = torch.zeros((4, 2), dtype=torch.int8, device="cuda")
    with pytest.raises(ito.ItoError) as ei:
        ito.ito_bdfp16_linear_fwd_f32(x, e, x, e, 100)
    assert ei.value.code == ito.ITO_ERR_ARG
