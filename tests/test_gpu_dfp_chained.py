"""The FP32 partial accumulation on the GPU ("Mixed Precision Training of
Convolutional Neural Networks using Integer Operations", section 4, "Handling
overflows") against the CPU oracle, bit for bit: ragged shapes over several
tiles, every chain length, with and without the one-bit input shift, chains
that overflow INT32 (and wrap) and the hand-worked cases."""
import numpy as np
import pytest

import oracle as O
from gpu_util import import_ito

pytestmark = pytest.mark.gpu

rng = np.random.default_rng(404)


@pytest.fixture(scope="module")
def ito():
    return import_ito()


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(ito, x, ex, W, ew, chain, shift):
    y = ito.ito_dfp16_linear_fwd_f32_chained(_dev(x), ito._i32dev(ex), _dev(W), ito._i32dev(ew), chain, shift)
    return y.cpu().numpy()


def _normal(shape, sigma=4096.0):
    return np.clip(np.rint(rng.normal(0, sigma, shape)), -32767, 32767).astype(np.int16)


@pytest.mark.parametrize("B,IC,OC", [(1, 64, 1), (3, 200, 70), (130, 1000, 129), (256, 2048, 300)])
@pytest.mark.parametrize("chain", [64, 128, 256, 512])
@pytest.mark.parametrize("shift", [0, 1])
def test_chained_matches_oracle(ito, B, IC, OC, chain, shift):
    x, W = _normal((B, IC)), _normal((OC, IC))
    got = _run(ito, x, -12, W, -17, chain, shift)
    want = O.dfp_linear_fwd_f32_chained(x, -12, W, -17, chain, input_shift=bool(shift))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert ito.ito_get_error() == 0


@pytest.mark.parametrize("shift", [0, 1])
def test_chained_overflowing_chains_wrap_like_the_oracle(ito, shift):
    """Saturated mantissas of mostly one sign: chains of 64 terms overflow INT32
    (with and without the shift) and wrap modulo 2^32 in both."""
    B, IC, OC = 64, 1100, 96
    x = np.where(rng.random((B, IC)) < 0.9, 32767, -32767).astype(np.int16)
    W = np.where(rng.random((OC, IC)) < 0.9, 32767, -32767).astype(np.int16)
    got = _run(ito, x, -12, W, -17, 64, shift)
    want = O.dfp_linear_fwd_f32_chained(x, -12, W, -17, 64, input_shift=bool(shift))
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_chained_hand_cases(ito):
    x = np.zeros((1, 128), np.int16)
    W = np.zeros((1, 128), np.int16)
    x[0, :4] = 32767
    W[0, :3] = 32767
    x[0, 64:68] = [1, 2, 3, 4]
    W[0, 64:68] = [5, 6, 7, 8]
    assert _run(ito, x, -20, W, -10, 64, 0)[0, 0] == np.float32(-8390143 / 2.0 ** 23)
    assert _run(ito, x, -20, W, -10, 64, 1)[0, 0] == np.float32(98301 / 2.0 ** 15)
    x = np.zeros((1, 192), np.int16)
    W = np.zeros((1, 192), np.int16)
    x[0, 0], W[0, 0] = 8191, 4096
    x[0, 64], W[0, 64] = 1, 1
    x[0, 128], W[0, 128] = 1, 1
    assert _run(ito, x, 0, W, 0, 64, 1)[0, 0] == np.float32(2.0 ** 25)


def test_chained_exponent_outside_int8_is_reported(ito):
    x, W = _normal((4, 64)), _normal((4, 64))
    _run(ito, x, 200, W, -17, 64, 1)
    assert ito.ito_get_error() == ito.ITO_ERR_EXPONENT
    assert ito.ito_get_error() == 0
