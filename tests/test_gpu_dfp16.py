"""DFP16 path on the GPU against the CPU oracle: exact int64 limb contractions
(ragged shapes, extreme mantissas, chunk boundaries), down-conversion with its
exponent, the integer update, and whole training steps in lockstep."""
import ctypes

import numpy as np
import pytest

import oracle as O
import seeded_inputs as si
from gpu_util import compare_records, digest, import_ito, load_digests

pytestmark = pytest.mark.gpu

rng = np.random.default_rng(4242)


@pytest.fixture(scope="module")
def ito():
    return import_ito()


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _h(t):
    return t.cpu().numpy()


def i16(shape, lim=32767):
    return rng.integers(-lim, lim + 1, shape).astype(np.int16)


SHAPES = [(1, 1, 1), (3, 27, 10), (16, 64, 48), (129, 513, 70), (200, 1025, 257), (64, 2048, 128)]


def _check_down(P_ref, e_in, out, e_out, rs, mx):
    m_ref, e_ref, rs_ref, mx_ref = O.dfp_down(P_ref, e_in)
    assert np.array_equal(_h(out), m_ref)
    assert int(_h(e_out)[0]) == e_ref and int(_h(rs)[0]) == rs_ref
    assert int(_h(mx)[0]) == mx_ref


@pytest.mark.parametrize("B,IC,OC", SHAPES)
def test_dfp_fwd(ito, B, IC, OC):
    x, W = i16((B, IC)), i16((OC, IC))
    x[0, :] = -32767
    W[0, :] = -32767
    ex, ew = -12, -17
    p64, mx, y, ey, rs = ito.ito_dfp16_linear_fwd(_dev(x), ito._i32dev(ex), _dev(W), ito._i32dev(ew))
    P = O.dfp_linear_fwd(x, W)
    assert np.array_equal(_h(p64), P)
    _check_down(P, ex + ew, y, ey, rs, mx)


@pytest.mark.parametrize("B,IC,OC", SHAPES)
def test_dfp_bwd_delta(ito, B, IC, OC):
    e, W = i16((B, OC)), i16((OC, IC))
    p64, mx, dp, ee, rs = ito.ito_dfp16_linear_bwd_delta(_dev(e), ito._i32dev(-20), _dev(W), ito._i32dev(-17))
    P = O.dfp_linear_dgrad(e, W)
    assert np.array_equal(_h(p64), P)
    _check_down(P, -37, dp, ee, rs, mx)


@pytest.mark.parametrize("B,IC,OC", SHAPES + [(2048, 40, 24)])
def test_dfp_wgrad(ito, B, IC, OC):
    e, x = i16((B, OC)), i16((B, IC))
    p64, mx, g, eg, rs = ito.ito_dfp16_linear_wgrad(_dev(e), ito._i32dev(-20), _dev(x), ito._i32dev(-12))
    P = O.dfp_linear_wgrad(e, x)
    assert np.array_equal(_h(p64), P)
    _check_down(P, -32, g, eg, rs, mx)


# at least 256 rows: the CTA-pair limb kernels, 1024-term chunks (the limb-stacked one with
# 128 x 128 tiles where the output has at least 128 columns, else 256 x 64 tiles); the last
# two shapes take the limb-stacked kernel in all three contractions, ragged in M, N and K
PAIR_SHAPES = [(256, 64, 64), (300, 1000, 130), (513, 2049, 200), (1024, 4096, 64), (2048, 1100, 96),
               (1100, 700, 300), (600, 520, 260)]


@pytest.mark.parametrize("B,IC,OC", PAIR_SHAPES)
def test_dfp_pair_fwd_dgrad_wgrad(ito, B, IC, OC):
    x, W = i16((B, IC)), i16((OC, IC))
    e = i16((B, OC))
    p64, _, _, _, _ = ito.ito_dfp16_linear_fwd(_dev(x), ito._i32dev(-12), _dev(W), ito._i32dev(-17))
    assert np.array_equal(_h(p64), O.dfp_linear_fwd(x, W))
    p64, _, _, _, _ = ito.ito_dfp16_linear_bwd_delta(_dev(e), ito._i32dev(-20), _dev(W), ito._i32dev(-17))
    assert np.array_equal(_h(p64), O.dfp_linear_dgrad(e, W))
    p64, _, _, _, _ = ito.ito_dfp16_linear_wgrad(_dev(e), ito._i32dev(-20), _dev(x), ito._i32dev(-12))
    assert np.array_equal(_h(p64), O.dfp_linear_wgrad(e, x))
    assert ito.ito_get_error() == 0


# The wide-tile kernel's result leaves through shared memory and TMA in 32 x 8 boxes, one
# at a time before a pair's last tile and all at once (staged in the idle pipeline
# stages) for it: a partial last wave, several tiles per pair, ragged M, N and K (boxes
# clipped at both edges), each contraction twice in a row
WIDE_SHAPES = [(1100, 1000, 2000), (2048, 1000, 1100), (2048, 2048, 2048), (512, 2048, 2048), (777, 3000, 1500)]


@pytest.mark.parametrize("B,IC,OC", WIDE_SHAPES)
def test_dfp_pair_wide_tile_stores(ito, B, IC, OC):
    x, W = i16((B, IC)), i16((OC, IC))
    e = i16((B, OC))
    for _ in range(2):
        p64, mx, _, _, _ = ito.ito_dfp16_linear_fwd(_dev(x), ito._i32dev(-12), _dev(W), ito._i32dev(-17))
        P = O.dfp_linear_fwd(x, W)
        assert np.array_equal(_h(p64), P)
        assert int(_h(mx)[0]) == int(np.abs(P).max())
    p64, _, _, _, _ = ito.ito_dfp16_linear_bwd_delta(_dev(e), ito._i32dev(-20), _dev(W), ito._i32dev(-17))
    assert np.array_equal(_h(p64), O.dfp_linear_dgrad(e, W))
    p64, _, _, _, _ = ito.ito_dfp16_linear_wgrad(_dev(e), ito._i32dev(-20), _dev(x), ito._i32dev(-12))
    assert np.array_equal(_h(p64), O.dfp_linear_wgrad(e, x))
    assert ito.ito_get_error() == 0


@pytest.mark.parametrize("OC", [70, 200])      # both pair kernels
def test_dfp_pair_extreme_chunks(ito, OC):
    """256+ rows, all products (-32767)^2: each of the pair kernels' limb
    accumulators reaches 2^24 exactly at a 1024-term chunk."""
    for K in (1023, 1024, 1025, 2048, 4096):
        x = np.full((300, K), -32767, np.int16)
        W = np.full((OC, K), -32767, np.int16)
        W[1::2] = 32767
        p64, _, _, _, _ = ito.ito_dfp16_linear_fwd(_dev(x), ito._i32dev(0), _dev(W), ito._i32dev(0))
        P = _h(p64)
        assert (P[:, 0::2] == K * 32767 * 32767).all() and (P[:, 1::2] == -K * 32767 * 32767).all()


def test_dfp_extreme_chunks(ito):
    """All products (-32767)^2: every limb accumulator reaches its chunk bound."""
    for K in (511, 512, 513, 1024, 2048):
        x = np.full((128, K), -32767, np.int16)
        W = np.full((64, K), -32767, np.int16)
        W[1::2] = 32767
        p64, _, _, _, _ = ito.ito_dfp16_linear_fwd(_dev(x), ito._i32dev(0), _dev(W), ito._i32dev(0))
        P = _h(p64)
        assert (P[:, 0::2] == K * 32767 * 32767).all() and (P[:, 1::2] == -K * 32767 * 32767).all()


@pytest.mark.parametrize("k_target", [-20, -3, 0, 5, 8, 15, 40])
def test_dfp_update(ito, k_target):
    n = 10007
    W, g = i16(n), i16(n)
    W[:3] = [32767, -32767, 0]
    ew, eta = -17, 8
    eg = ew + eta - k_target
    Wd = _dev(W)
    k, nz = ito.ito_dfp16_update(Wd, _dev(g), ito._i32dev(eg), ew, eta)
    Wn, nzo = O.dfp_update(W, g, k_target)
    assert int(_h(k)[0]) == k_target and int(_h(nz)[0]) == nzo
    assert np.array_equal(_h(Wd), Wn)


def test_dfp_exponent_overflow_is_reported(ito):
    x, W = i16((8, 64)), i16((8, 64))
    ito.ito_dfp16_linear_fwd(_dev(x), ito._i32dev(120), _dev(W), ito._i32dev(100))
    assert ito.ito_get_error() == ito.ITO_ERR_EXPONENT
    assert ito.ito_get_error() == 0          # read clears the word


class DfpRun:
    def __init__(self, w):
        import torch
        self.torch = torch
        self.ito = import_ito()
        self.w = w
        self.m = self.ito.Dfp16Model(list(w.dims), w.batch, w.exp_w, w.eta)
        for l, W in enumerate(si.make_weights(w)):
            self.m.set_weights(l, W)

    def step(self, t):
        x, _ = si.make_batch(self.w, t)
        self.m.train_step(self.torch.from_numpy(x).cuda(), self.w.exp_x)
        self.torch.cuda.synchronize()
        return x

    def record(self, kinds=("p", "y", "e", "pd", "pg", "g", "w")):
        r = {}
        L = self.m.n_layers
        for l in range(L):
            for k in kinds:
                if k == "pd" and l == 0:
                    continue
                r["%s%d" % (k, l)] = self.m.tensor("%s%d" % (k, l)).cpu().numpy()
        st = self.m.stats()
        for k, v in st.items():
            if (k.startswith("rsd") or k.startswith("pdmax")) and k.endswith("0") and len(k) in (4, 6):
                continue
            r[k] = v
        return r


def test_dfp_model_small_lockstep():
    w = si.Workload(97, "dfp16_small", "dfp16", 16, dims=(64, 48, 32), sigma=4096.0, lim=32767,
                    exp_x=-12, exp_w=-17, eta=8)
    g = DfpRun(w)
    weights = si.make_weights(w)
    for t in range(5):
        x, _ = si.make_batch(w, t)
        rec = O.dfp16_step(weights, w.exp_w, x, w.exp_x, eta=w.eta)
        g.step(t)
        compare_records(rec, g.record(), t)
        weights = [rec["w%d" % l] for l in range(len(weights))]


def test_dfp_model_full_size_live_step():
    w = si.by_name(4)
    g = DfpRun(w)
    weights = si.make_weights(w)
    x, _ = si.make_batch(w, 0)
    rec = O.dfp16_step(weights, w.exp_w, x, w.exp_x, eta=w.eta, route="f64")
    g.step(0)
    compare_records(rec, g.record(), 0)


def test_dfp_model_100_steps_digests():
    w = si.by_name(4)
    ref = load_digests(w)
    assert ref is not None and len(ref) == 100
    g = DfpRun(w)
    for t, d in enumerate(ref):
        x = g.step(t)
        assert digest(x) == d["in.x"], "input generator diverged"
        kinds = ("p", "y", "e", "pd", "pg", "g", "w") if t < 3 else ("y", "e", "g", "w")
        r = g.record(kinds)
        bad = [k for k, v in r.items() if k in d and
               (digest(v) if isinstance(v, np.ndarray) else int(v)) != d[k]]
        assert not bad, "step %d differs from the oracle in %s" % (t, bad)


def test_dfp_from_to_float_parity(ito):
    import torch
    for scale in (1e-30, 1e-3, 1.0, 3.7e5, 1e30):
        f = (rng.standard_normal(10001) * scale).astype(np.float32)
        f[5] = 0.0
        f[6] = np.float32(1e-42) * np.sign(scale)        # a subnormal input
        mant, e = ito.ito_dfp16_from_float(torch.from_numpy(f).cuda())
        m_ref, e_ref = O.dfp_from_float(f)
        assert int(_h(e)[0]) == e_ref and np.array_equal(_h(mant), m_ref), scale
        back = ito.ito_dfp16_to_float(mant, e)
        assert np.array_equal(_h(back).view(np.int32), O.dfp_to_float(m_ref, e_ref).view(np.int32))
    assert ito.ito_get_error() == 0


def test_dfp_linear_fwd_f32_parity(ito):
    B, IC, OC = 130, 1025, 70
    x, W = i16((B, IC)), i16((OC, IC))
    p64, y = ito.ito_dfp16_linear_fwd_f32(_dev(x), ito._i32dev(-12), _dev(W), ito._i32dev(-17))
    P = O.dfp_linear_fwd(x, W)
    assert np.array_equal(_h(p64), P)
    assert np.array_equal(_h(y).view(np.int32), O.p64_to_float(P, -29).view(np.int32))
    # the FP32 output re-quantised for the next layer (float -> DFP16)
    mant, e = ito.ito_dfp16_from_float(y)
    m_ref, e_ref = O.dfp_from_float(O.p64_to_float(P, -29))
    assert int(_h(e)[0]) == e_ref and np.array_equal(_h(mant), m_ref)


def test_dfp_model_pipelined_host_steps():
    """ito_dfp16_train_step_host_async (input copies on the model's copy stream into two
    alternating buffers, overlapping the previous step) trains as steps on device inputs:
    the same tensors after the last step, and the statistics copied back (in the layout
    of ito_dfp16_model_read_stats) are the step's."""
    import torch
    w = si.Workload(97, "dfp16_small", "dfp16", 256, dims=(512, 384, 256), sigma=4096.0, lim=32767,
                    exp_x=-12, exp_w=-17, eta=8)
    a, b = DfpRun(w), DfpRun(w)
    stream = torch.cuda.Stream()
    xs = [torch.from_numpy(np.ascontiguousarray(si.make_batch(w, t)[0])).pin_memory() for t in range(5)]
    st = torch.zeros(a.m.num_stats(), dtype=torch.int64).pin_memory()
    for t in range(len(xs)):
        a.m.train_step_host_async(xs[t], w.exp_x, st, stream=stream)
        if t == 2:
            stream.synchronize()
    stream.synchronize()
    for t in range(len(xs)):
        b.step(t)
    ra, rb = a.record(), b.record()
    assert ra.keys() == rb.keys()
    for k in ra:
        assert np.array_equal(np.asarray(ra[k]), np.asarray(rb[k])), k
    n = a.m.num_stats()
    want = (ctypes.c_int64 * n)()
    assert a.ito._lib.ito_dfp16_model_read_stats(a.m._h, want, n) == 0
    assert list(st.numpy()) == list(want)
