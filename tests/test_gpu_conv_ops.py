"""Single-layer 3x3 conv and global pooling on the GPU against the CPU
oracle's direct loops, element by element: the integer CNN's three conv shapes
at full batch, ragged shapes (odd spatial sizes, channel counts that are not a
multiple of 8, a one-pixel image), gated and ungated delta propagation, and the
pooling forward/backward."""
import numpy as np
import pytest

import oracle as O
import seeded_inputs as si
from gpu_util import import_ito

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ito():
    return import_ito()


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _host(t):
    return t.cpu().numpy()


def _u32(t):
    return int(_host(t)[0]) & 0xFFFFFFFF


rng = np.random.default_rng(7031)


def i8(shape, lo=-128, hi=127):
    return rng.integers(lo, hi + 1, shape).astype(np.int8)


# (B, H, W, IC, OC, stride): the CNN workload's convs at batch 128, then ragged cases
CNN = si.by_name(2)
FULL = [(CNN.batch, 32 // (1 if l == 0 else 2 ** (l - 1)), 32 // (1 if l == 0 else 2 ** (l - 1)), ic, oc, s)
        for l, (ic, oc, s) in enumerate(CNN.convs)]
RAGGED = [(1, 1, 1, 1, 1, 1), (2, 7, 5, 5, 12, 2), (3, 9, 11, 3, 70, 1), (2, 6, 6, 16, 130, 2),
          (1, 13, 4, 24, 8, 3), (5, 8, 8, 9, 257, 1)]


def test_full_shapes_are_the_workload():
    assert [f[3:] for f in FULL] == [(3, 64, 1), (64, 128, 2), (128, 256, 2)]
    assert [f[1] for f in FULL] == [32, 32, 16]


# Stride-2 shapes taken by the parity-plane kernels (even H and W, OW of 8, 16 or 32,
# channels in multiples of 64): a row tile of two images with one or three in the batch,
# 32 output columns, a 4 x 32 input (four images to a row tile), 512 delta channels (the
# four-tap delta phase sums 2048 terms: two exact chunks)
PHASE = [(1, 16, 16, 64, 64, 2), (3, 16, 16, 128, 64, 2), (2, 64, 64, 64, 64, 2), (2, 4, 32, 64, 128, 2),
         (2, 16, 16, 64, 512, 2)]

@pytest.mark.parametrize("B,H,W,IC,OC,stride", FULL + RAGGED + PHASE)
@pytest.mark.parametrize("relu", [0, 1])
def test_conv2d_fwd(ito, B, H, W, IC, OC, stride, relu):
    x, Wt = i8((B, H, W, IC), -127, 127), i8((OC, 3, 3, IC), -127, 127)
    y32, mx, sh, y = ito.ito_conv2d_fwd(_dev(x), _dev(Wt), stride, relu)
    Y = O.conv2d_fwd(x, Wt, stride)
    a, s, m = O.requant(Y, relu=bool(relu))
    assert np.array_equal(_host(y32), Y)
    assert (_u32(mx), int(_host(sh)[0])) == (m, s)
    assert np.array_equal(_host(y), a)
    assert ito.ito_get_error() == 0


@pytest.mark.parametrize("B,H,W,IC,OC,stride", FULL[1:] + RAGGED)
@pytest.mark.parametrize("gated", [False, True])
def test_conv2d_bwd_delta(ito, B, H, W, IC, OC, stride, gated):
    OH, OW = O.conv_out(H, 3, stride), O.conv_out(W, 3, stride)
    e, Wt = i8((B, OH, OW, OC)), i8((OC, 3, 3, IC), -127, 127)
    a_prev = i8((B, H, W, IC), -3, 127) if gated else None
    d32, mx, sh, dp = ito.ito_conv2d_bwd_delta(_dev(e), _dev(Wt), _dev(a_prev) if gated else None, (H, W), stride)
    D = O.conv2d_dgrad(e, Wt, (H, W), stride)
    ep, s, m = O.requant_mask(D, a_prev)
    assert np.array_equal(_host(d32), D)
    assert (_u32(mx), int(_host(sh)[0])) == (m, s)
    assert np.array_equal(_host(dp), ep)


@pytest.mark.parametrize("B,H,W,IC,OC,stride", PHASE)
@pytest.mark.parametrize("gated", [False, True])
def test_conv2d_bwd_delta_stride2_phases(ito, B, H, W, IC, OC, stride, gated):
    OH, OW = O.conv_out(H, 3, stride), O.conv_out(W, 3, stride)
    e, Wt = i8((B, OH, OW, OC)), i8((OC, 3, 3, IC), -127, 127)
    a_prev = i8((B, H, W, IC), -3, 127) if gated else None
    d32, mx, sh, dp = ito.ito_conv2d_bwd_delta(_dev(e), _dev(Wt), _dev(a_prev) if gated else None, (H, W), stride)
    D = O.conv2d_dgrad(e, Wt, (H, W), stride)
    ep, s, m = O.requant_mask(D, a_prev)
    assert np.array_equal(_host(d32), D)
    assert (_u32(mx), int(_host(sh)[0])) == (m, s)
    assert np.array_equal(_host(dp), ep)


def test_conv2d_bwd_delta_stride2_extreme(ito):
    """Every product (-128)(-127): the interior positions of the four-tap phase sum
    4 x 512 = 2048 of them, 1024 to an exact chunk."""
    B, H, W, IC, OC = 2, 16, 16, 64, 512
    e = np.full((B, 8, 8, OC), -128, np.int8)
    Wt = np.full((OC, 3, 3, IC), -127, np.int8)
    d32, mx, _, _ = ito.ito_conv2d_bwd_delta(_dev(e), _dev(Wt), None, (H, W), 2)
    D = O.conv2d_dgrad(e, Wt, (H, W), 2)
    assert int(D.max()) == 4 * OC * 128 * 127
    assert np.array_equal(_host(d32), D)
    assert _u32(mx) == int(np.abs(D).max())


@pytest.mark.parametrize("B,H,W,IC,OC,stride", FULL + RAGGED + PHASE)
def test_conv2d_wgrad(ito, B, H, W, IC, OC, stride):
    OH, OW = O.conv_out(H, 3, stride), O.conv_out(W, 3, stride)
    e, x = i8((B, OH, OW, OC)), i8((B, H, W, IC), 0, 127)
    G, mx = ito.ito_conv2d_wgrad(_dev(e), _dev(x), stride)
    Gref = O.conv2d_wgrad(e, x, 3, stride)
    assert np.array_equal(_host(G), Gref)
    assert _u32(mx) == O.absmax32(Gref)


def test_conv2d_stride2_planes_extreme(ito):
    """Every product (-127)(-127) or (-128)(-127) on the parity-plane kernels: the forward of
    the third conv sums 9 x 128 = 1152 terms at interior positions (two exact chunks);
    the second conv's weight gradient sums 128 x 16 x 16 = 32768 terms for the centre
    tap, over K slices added by the reduction."""
    B, H, W, IC, OC = 4, 16, 16, 128, 64
    x = np.full((B, H, W, IC), -127, np.int8)
    Wt = np.full((OC, 3, 3, IC), -127, np.int8)
    y32, mx, _, _ = ito.ito_conv2d_fwd(_dev(x), _dev(Wt), 2, 0)
    Y = O.conv2d_fwd(x, Wt, 2)
    assert int(Y.max()) == 9 * IC * 127 * 127
    assert np.array_equal(_host(y32), Y)
    assert _u32(mx) == int(np.abs(Y).max())
    B, H, W, IC, OC = 128, 32, 32, 64, 128
    e = np.full((B, 16, 16, OC), -128, np.int8)
    x = np.full((B, H, W, IC), -127, np.int8)
    G, mx = ito.ito_conv2d_wgrad(_dev(e), _dev(x), 2)
    Gr = O.conv2d_wgrad(e, x, 3, 2)
    assert int(Gr.max()) == B * 16 * 16 * 128 * 127
    assert np.array_equal(_host(G), Gr)
    assert _u32(mx) == int(np.abs(Gr).max())


def test_conv2d_wgrad_extreme_long_contraction(ito):
    """The first conv's weight gradient sums up to 131072 terms: with every
    product (-128)(-127) = 16256 the centre tap reaches 2130706432, just under
    2^31, exact through the chunked fp32 accumulation; edge taps sum fewer."""
    B, H, W, IC, OC = 128, 32, 32, 3, 64
    e = np.full((B, H, W, OC), -128, np.int8)
    x = np.full((B, H, W, IC), -127, np.int8)
    G, mx = ito.ito_conv2d_wgrad(_dev(e), _dev(x), 1)
    Gref = O.conv2d_wgrad(e, x, 3, 1)
    assert np.array_equal(_host(G), Gref)
    assert _u32(mx) == O.absmax32(Gref) == 128 * 32 * 32 * 128 * 127


@pytest.mark.parametrize("B,H,W,C", [(128, 8, 8, 256), (3, 5, 7, 10), (1, 1, 1, 1)])
def test_gap_fwd_bwd(ito, B, H, W, C):
    a = i8((B, H, W, C), -20, 127)
    P, mx, sh, pa = ito.ito_gap_fwd(_dev(a))
    Pref = O.gap_fwd(a)
    pref, s, m = O.requant(Pref, relu=False)
    assert np.array_equal(_host(P), Pref)
    assert (_u32(mx), int(_host(sh)[0])) == (m, s)
    assert np.array_equal(_host(pa), pref)
    dP = i8((B, C))
    d = ito.ito_gap_bwd(_dev(dP), _dev(a))
    assert np.array_equal(_host(d), O.gap_bwd(dP, a))


def test_conv_bad_arguments(ito):
    import torch
    x = torch.zeros((1, 4, 4, 3), dtype=torch.int8, device="cuda")
    Wt = torch.zeros((8, 3, 3, 3), dtype=torch.int8, device="cuda")
    with pytest.raises(ito.ItoError) as ei:
        ito.ito_conv2d_fwd(x, Wt, 5, 1)
    assert ei.value.code == ito.ITO_ERR_SHAPE
    assert ito._lib.ito_conv2d_workspace_size(1, 4, 4, 3, 8, 0) == 0
