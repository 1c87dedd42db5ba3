"""Adaptive precision training on the GPU against the CPU oracle ("Adaptive
Precision Training for Resource Constrained Devices", section III, on the DFP16
model): the k-bit saturating update and the precision change element by
element, a small run in lockstep (every tensor, every step scalar, the
epoch-end Gavg means compared as float64 values, the precision trajectory), and
the full 2048-wide workload against the oracle's 100-step digests."""
import numpy as np
import pytest

import oracle as O
import seeded_inputs as si
from gpu_util import compare_records, digest, import_ito, load_digests

pytestmark = pytest.mark.gpu

rng = np.random.default_rng(4451)


@pytest.fixture(scope="module")
def ito():
    return import_ito()


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("bits", [2, 6, 11, 16])
@pytest.mark.parametrize("k", [-3, 0, 5])
@pytest.mark.parametrize("n", [1, 7, 4096, 100003])
def test_update_bits(ito, bits, k, n):
    lim = (1 << (bits - 1)) - 1
    W = rng.integers(-lim, lim + 1, n).astype(np.int16)
    g = rng.integers(-32767, 32768, n).astype(np.int16)
    ew, eta = -9, 6
    eg = ew + eta - k
    Wd = _dev(W)
    kd, nz = ito.ito_dfp16_update_bits(Wd, _dev(g), ito._i32dev(eg), ew, eta, bits)
    Wref, nzref = O.dfp_update(W, g, k, bits)
    assert np.array_equal(Wd.cpu().numpy(), Wref)
    assert int(kd.cpu()[0]) == k and int(nz.cpu()[0]) == nzref


@pytest.mark.parametrize("old,new", [(6, 9), (9, 6), (16, 2), (2, 16), (12, 12), (16, 15), (3, 2)])
@pytest.mark.parametrize("n", [1, 4099])
def test_set_bits(ito, old, new, n):
    lim = (1 << (old - 1)) - 1
    W = rng.integers(-lim, lim + 1, n).astype(np.int16)
    W[: min(n, 2)] = [lim, -lim][: min(n, 2)]
    Wd = _dev(W)
    ito.ito_dfp_set_bits(Wd, old, new)
    Wref, _ = O.dfp_set_bits(W, old, new)
    assert np.array_equal(Wd.cpu().numpy(), Wref)


class AptRun:
    """The CUDA DFP16 model of an APT workload, stepped with Algorithm 2."""

    def __init__(self, w):
        import torch
        self.torch = torch
        self.ito = import_ito()
        self.w = w
        self.m = self.ito.Dfp16Model(list(w.dims), w.batch, w.exp_w, w.eta)
        for l, W in enumerate(si.make_weights(w)):
            self.m.set_weights(l, W)
        a = w.apt
        self.m.apt_enable(a.k_init, a.k_min, a.k_max, a.t_min, a.t_max, a.eval_every)

    def step(self, t):
        """-> (x, epoch-end result (gavg, bits) or None)"""
        x, _ = si.make_batch(self.w, t)
        self.m.train_step(self.torch.from_numpy(x).cuda(), self.w.exp_x)
        end = None
        if t % self.w.apt.epoch == self.w.apt.epoch - 1:
            end = self.m.apt_epoch_end()
        self.torch.cuda.synchronize()
        return x, end

    def precision(self):
        bits, exps = zip(*[self.m.precision(l) for l in range(self.m.n_layers)])
        return list(bits), list(exps)

    def record(self, kinds=("p", "y", "e", "pd", "pg", "g", "w")):
        r = {}
        for l in range(self.m.n_layers):
            for k in kinds:
                if k == "pd" and l == 0:
                    continue
                r["%s%d" % (k, l)] = self.m.tensor("%s%d" % (k, l)).cpu().numpy()
        for k, v in self.m.stats().items():
            if k in ("rsd0", "pdmax0"):
                continue
            r[k] = v
        return r


SMALL = si.Workload(96, "dfp16_apt_small", "dfp16", 16, dims=(64, 48, 32, 24), sigma=4096.0, lim=32767,
                    exp_x=-12, exp_w=-17, eta=8,
                    apt=si.AptSetting(k_init=6, k_min=3, k_max=12, t_min=0.015, t_max=0.018, epoch=4,
                                      eval_every=2))


def test_apt_small_lockstep():
    g = AptRun(SMALL)
    states = []
    recs = []
    O.apt_run(SMALL, 12, callback=lambda t, r, st: (recs.append(r), states.append(st)))
    moved = 0
    for t in range(12):
        _, end = g.step(t)
        # the weights in the record are after the epoch-end precision change; compare
        # the step's own tensors before it by comparing everything but w at epoch ends
        r = g.record(("p", "y", "e", "pd", "pg", "g") + (("w",) if end is None else ()))
        compare_records(recs[t], r, t)
        bits, exps = g.precision()
        assert bits == states[t]["bits"] and exps == states[t]["exp_w"], t
        if end is not None:
            gavg, nb = end
            assert gavg == states[t]["gavg"], "epoch-end Gavg differs at step %d" % t
            assert nb == states[t]["bits"]
            before = states[t - 1]["bits"]
            for l in range(3):
                want, _ = O.dfp_set_bits(recs[t]["w%d" % l], before[l], nb[l])
                assert np.array_equal(g.m.tensor("w%d" % l).cpu().numpy(), want.ravel()), (t, l)
            moved += 1
    assert moved == 3


def test_apt_full_size_digests():
    w = si.by_name(7)
    ref = load_digests(w)
    assert ref is not None and len(ref) == 100
    g = AptRun(w)
    for t, d in enumerate(ref):
        x, end = g.step(t)
        assert digest(x) == d["in.x"], "input generator diverged"
        kinds = ("p", "y", "e", "pd", "pg", "g") if t < 3 else ("y", "e", "g")
        r = g.record(kinds)
        bad = [k for k, v in r.items() if k in d and
               (digest(v) if isinstance(v, np.ndarray) else int(v)) != d[k]]
        assert not bad, "step %d differs from the oracle in %s" % (t, bad)
        bits, exps = g.precision()
        assert bits == [d["apt.bits%d" % l] for l in range(3)], t
        assert exps == [d["apt.exp_w%d" % l] for l in range(3)], t
        for l in range(3):
            assert digest(g.m.tensor("w%d" % l).cpu().numpy()) == d["w%d" % l] or end is not None, (t, l)
        if end is not None:
            assert end[0] == [d["apt.gavg%d" % l] for l in range(3)], t
