"""Single-layer operations on the GPU against the CPU oracle, element by element:
ragged shapes spanning several tiles, adversarial values for the exactness of
the tensor-core contraction, every branch of the NITI update."""
import numpy as np
import pytest

import oracle as O
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


rng = np.random.default_rng(2024)

SHAPES = [(1, 1, 1), (3, 27, 10), (32, 64, 64), (129, 300, 257), (256, 784, 1024), (200, 2100, 130),
          (17, 1000, 1000), (300, 64, 520)]


def i8(shape, lo=-128, hi=127):
    return rng.integers(lo, hi + 1, shape).astype(np.int8)


@pytest.mark.parametrize("B,IC,OC", SHAPES)
@pytest.mark.parametrize("relu", [0, 1])
def test_linear_fwd(ito, B, IC, OC, relu):
    x, W = i8((B, IC)), i8((OC, IC), -127, 127)
    y32, mx, sh, y = ito.ito_linear_fwd(_dev(x), _dev(W), relu)
    Y = O.linear_fwd(x, W)
    a, s, m = O.requant(Y, relu=bool(relu))
    assert np.array_equal(_host(y32), Y)
    assert (_u32(mx), int(_host(sh)[0])) == (m, s)
    assert np.array_equal(_host(y), a)
    assert ito.ito_get_error() == 0


@pytest.mark.parametrize("B,IC,OC", SHAPES)
@pytest.mark.parametrize("gated", [False, True])
def test_linear_bwd_delta(ito, B, IC, OC, gated):
    e, W = i8((B, OC)), i8((OC, IC), -127, 127)
    a_prev = i8((B, IC), -3, 127) if gated else None
    d32, mx, sh, dp = ito.ito_linear_bwd_delta(_dev(e), _dev(W), _dev(a_prev) if gated else None)
    D = O.linear_dgrad(e, W)
    ep, s, m = O.requant_mask(D, a_prev)
    assert np.array_equal(_host(d32), D)
    assert (_u32(mx), int(_host(sh)[0])) == (m, s)
    assert np.array_equal(_host(dp), ep)


@pytest.mark.parametrize("B,IC,OC", SHAPES + [(8192, 72, 40), (3000, 130, 9)])
def test_linear_wgrad(ito, B, IC, OC):
    e, a = i8((B, OC)), i8((B, IC), 0, 127)
    G, mx = ito.ito_linear_wgrad(_dev(e), _dev(a))
    Gref = O.linear_wgrad(e, a)
    assert np.array_equal(_host(G), Gref)
    assert _u32(mx) == O.absmax32(Gref)


@pytest.mark.parametrize("K", [1, 63, 1023, 1024, 1025, 2048, 4096, 8192])
def test_exactness_all_extreme(ito, K):
    """Every product is (-128)(-128) = 2^14: chunk sums reach exactly 2^24."""
    x = np.full((130, K), -128, np.int8)
    W = np.full((260, K), -128, np.int8)
    y32, mx, sh, y = ito.ito_linear_fwd(_dev(x), _dev(W), 0)
    assert (_host(y32) == K * 16384).all()
    assert _u32(mx) == K * 16384


@pytest.mark.parametrize("K", [1024, 2048, 3000])
def test_exactness_large_then_small_terms(ito, K):
    """Large products next to +-1 products in the same chunk: a truncating
    accumulator would lose the small ones."""
    h = K // 2
    x = np.zeros((128, K), np.int8)
    W = np.zeros((256, K), np.int8)
    x[:, :h] = -128
    x[:, h:] = 1
    W[:, :h] = -128
    W[:, h:] = rng.choice([-1, 1], size=(256, K - h))
    x[1::2] = x[1::2, ::-1]        # odd rows: small terms first
    W[3::4, h:] = 0
    y32, _, _, _ = ito.ito_linear_fwd(_dev(x), _dev(W), 0)
    assert np.array_equal(_host(y32), O.linear_fwd(x, W))


def test_exactness_alternating_and_random_extremes(ito):
    K = 4096
    x = np.tile(np.array([127, -128], np.int8), (96, K // 2))
    W = i8((200, K))
    W[::3] = np.where(rng.random((len(W[::3]), K)) < 0.5, -128, 127)
    y32, _, _, _ = ito.ito_linear_fwd(_dev(x), _dev(W), 0)
    assert np.array_equal(_host(y32), O.linear_fwd(x, W))


@pytest.mark.parametrize("target_shift", [0, 1, 3, 9, 10, 12, 25])
@pytest.mark.parametrize("n", [7, 4096, 100003])
def test_niti_update_branches(ito, target_shift, n):
    if target_shift == 25:
        # max |G| = 2^31 needs INT32_MIN itself
        G = rng.integers(-(2**31) + 1, 2**31, n).astype(np.int32)
        G[0] = np.iinfo(np.int32).min
    else:
        lim = (1 << (target_shift + 7)) - 1
        G = rng.integers(-lim, lim + 1, n).astype(np.int32)
        G[0] = lim
    W = i8(n)
    W[:4] = [-128, 127, -128, 127]
    Wd = _dev(W)
    Gd = _dev(G)
    mx = _dev(np.array([O.absmax32(G)], dtype=np.uint32).view(np.int32))
    sh, ws, nz = ito.ito_niti_update(Wd, Gd, mx)
    Wn, s, wsh, m, nzo = O.niti_update(W, G)
    assert s == target_shift
    assert (int(_host(sh)[0]), int(_host(ws)[0]), int(_host(nz)[0])) == (s, wsh, nzo)
    assert np.array_equal(_host(Wd), Wn)


def test_top_error(ito):
    B, C = 300, 1000
    logits = i8((B, C))
    labels = rng.integers(0, C, B).astype(np.int32)
    logits[0, labels[0]] = 127
    logits[1, labels[1]] = -128
    d = ito.ito_top_error(_dev(logits), _dev(labels), 64)
    assert np.array_equal(_host(d), O.top_error(logits, labels, 64))


@pytest.mark.parametrize("C", [1000, 10])   # eight-class groups, and the per-element kernel
def test_top_error_bad_label_sets_error_word(ito, C):
    """The oracle rejects a label outside [0, C); the kernel reports it through
    the device error word (ITO_ERR_ARG) and leaves the valid rows right."""
    B = 64
    logits = i8((B, C))
    labels = rng.integers(0, C, B).astype(np.int32)
    assert ito.ito_get_error() == 0
    for bad in (C, -1):
        lab = labels.copy()
        lab[5] = bad
        d = _host(ito.ito_top_error(_dev(logits), _dev(lab), 64))
        assert ito.ito_get_error() == ito.ITO_ERR_ARG
        assert ito.ito_get_error() == 0                 # read and cleared
        ok = np.arange(B) != 5
        assert np.array_equal(d[ok], O.top_error(logits[ok], lab[ok], 64))


def test_wgrad_longest_contraction_extreme_values(ito):
    """K = 131072 terms of (-128) * 127 = -16256: the sum -2,130,706,432 is just
    inside int32 (split-K slices and chunk drains must add exactly)."""
    B, IC, OC = 131072, 27, 64
    e = np.full((B, OC), -128, np.int8)
    a = np.full((B, IC), 127, np.int8)
    e[:, 1] = 127                      # column 1: +16129 per term
    a[::2, 2] = -127                   # column 2 alternates sign: sums to 0 for column 0
    G, mx = ito.ito_linear_wgrad(_dev(e), _dev(a))
    Gh = _host(G)
    assert Gh[0, 0] == -128 * 127 * B and Gh[1, 0] == 127 * 127 * B
    assert Gh[0, 2] == 0
    assert _u32(mx) == 128 * 127 * B


def test_update_zero_gradient_leaves_weights(ito):
    W = i8(4096)
    Wd = _dev(W)
    sh, ws, nz = ito.ito_niti_update(Wd, _dev(np.zeros(4096, np.int32)), _dev(np.zeros(1, np.int32)))
    assert (int(_host(sh)[0]), int(_host(ws)[0]), int(_host(nz)[0])) == (0, 0, 0)
    assert np.array_equal(_host(Wd), W)


@pytest.mark.parametrize("B,IC,OC", [(8192, 2000, 3000), (8192, 4096, 4096)])
def test_wgrad_last_wave_split(ito, B, IC, OC):
    """Weight gradients whose last wave of 256 x 256 pair tiles is split along K
    (3000 x 2000 outputs: 96 tiles, ragged edges; 4096 x 4096: 256 tiles)
    against the oracle's exact float64 contraction."""
    e, a = i8((B, OC)), i8((B, IC), 0, 127)
    G, mx = ito.ito_linear_wgrad(_dev(e), _dev(a))
    Gref = O.linear_wgrad_f64(e, a)
    assert np.array_equal(_host(G), Gref)
    assert _u32(mx) == O.absmax32(Gref)
    assert ito.ito_get_error() == 0


def test_fwd_last_wave_split(ito):
    """A forward contraction (K-major operands) with a split last wave:
    3000 x 2000 outputs, K = 8192, ragged edges."""
    x, W = i8((3000, 8192)), i8((2000, 8192), -127, 127)
    y32, mx, sh, y = ito.ito_linear_fwd(_dev(x), _dev(W), 1)
    Y = O.linear_fwd_f64(x, W)
    assert np.array_equal(_host(y32), Y)
    a, s, m = O.requant(Y, relu=True)
    assert (_u32(mx), int(_host(sh)[0])) == (m, s)
    assert np.array_equal(_host(y), a)
