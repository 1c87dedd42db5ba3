"""Pins of the oracle's adaptive-precision pieces ("Adaptive Precision Training
for Resource Constrained Devices", section III, on DFP weights): the Gavg value
of a hand-worked gradient, the precision change against exact rational
rounding, Algorithm 1 on hand cases, the k-bit saturating update, and the
invariants of a whole run (Algorithm 2)."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
import seeded_inputs as si


def test_gavg_hand_worked():
    # g mantissas [3, -5, 0, 8, -16, 4] (sum |g| = 36), N = 6 weights, batch B = 3,
    # E_G = -10, E_W = -12: mean |g| over weights = 6 per unit of 2^-10 in batch-sum
    # terms; the batch-mean gradient is 2 * 2^-10 = 2^-9 per weight on average;
    # eps = 2^-12, so Gavg = 2^-9 / 2^-12 = 8.
    g = np.array([3, -5, 0, 8, -16, 4], np.int16)
    assert O.abs_sum16(g) == 36
    assert O.apt_gavg(36, 6, 3, -10, -12) == 8.0
    # a plausible slip, the exponents swapped, gives 1/8: the pin tells them apart
    assert math.ldexp(36.0, -12 + 10) / 18 != 8.0


def test_abs_sum_extremes():
    assert O.abs_sum16(np.array([-32768, 32767, -1, 0], np.int16)) == 65536


@pytest.mark.parametrize("old,new", [(6, 9), (2, 16), (15, 16), (7, 7)])
def test_set_bits_up_keeps_every_value(old, new):
    lim = (1 << (old - 1)) - 1
    W = np.arange(-lim, lim + 1, dtype=np.int16)
    Wn, de = O.dfp_set_bits(W, old, new)
    assert de == old - new
    # value m * 2^E is unchanged: m' * 2^(E + de) == m * 2^E
    assert all(int(a) * 2 ** (new - old) == int(b) for a, b in zip(W, Wn))


@pytest.mark.parametrize("old,new", [(10, 9), (10, 6), (16, 2), (12, 5), (3, 2)])
def test_set_bits_down_is_rounded_and_saturated(old, new):
    lim_o, lim_n = (1 << (old - 1)) - 1, (1 << (new - 1)) - 1
    W = np.arange(-lim_o, lim_o + 1, dtype=np.int16)
    Wn, de = O.dfp_set_bits(W, old, new)
    assert de == old - new
    for a, b in zip(W.tolist(), Wn.tolist()):
        exact = Fraction(a, 2 ** (old - new))
        want = math.floor(exact + Fraction(1, 2))          # round half up
        want = max(-lim_n, min(lim_n, want))
        assert b == want, (a, b, want)


def test_policy_hand_cases():
    bits = [6, 6, 6, 16, 2, 6]
    gavg = [0.5, 1.0, 5.0, 0.1, 200.0, 200.0]
    assert O.apt_policy(bits, gavg, 1.0, 100.0, 2, 16) == [7, 6, 6, 16, 2, 5]
    # T_max = infinity (the page's Figure 1 demonstration): never lowered
    assert O.apt_policy([6], [1e300], 1.0, float("inf"), 2, 16) == [6]


def test_update_saturates_to_the_precision():
    # 6 bits: |W| <= 31; k = 0 applies G unchanged, k = 1 rounds half up
    W = np.array([30, -30, 31, -31, 0, 5], np.int16)
    G = np.array([-5, 5, 0, 0, 100, -3], np.int16)
    Wn, nz = O.dfp_update(W, G, 0, bits=6)
    assert Wn.tolist() == [31, -31, 31, -31, -31, 8] and nz == 4
    Wn, nz = O.dfp_update(W, G, 1, bits=6)
    # rhu(-5,1) = -2, rhu(5,1) = 3, rhu(100,1) = 50, rhu(-3,1) = -1
    assert Wn.tolist() == [31, -31, 31, -31, -31, 6] and nz == 4
    # 16 bits is the plain DFP16 update
    W16 = np.array([32760, -32760], np.int16)
    assert O.dfp_update(W16, np.array([-100, 100], np.int16), 0)[0].tolist() == [32767, -32767]


SMALL = si.Workload(96, "dfp16_apt_small", "dfp16", 16, dims=(64, 48, 32, 24), sigma=4096.0, lim=32767,
                    exp_x=-12, exp_w=-17, eta=8,
                    apt=si.AptSetting(k_init=6, k_min=3, k_max=12, t_min=0.015, t_max=0.018, epoch=4,
                                      eval_every=2))


def test_apt_run_follows_algorithms_1_and_2():
    """A whole run: weights stay inside their precision; precision changes only
    at epoch ends, by Algorithm 1 applied to the mean of that epoch's Gavg
    evaluations (recomputed here from the step records); an increase keeps
    every weight value, a decrease rounds; raises and lowers both occur."""
    w, a = SMALL, SMALL.apt
    seen = {"up": 0, "down": 0}
    state = {"bits": [a.k_init] * 3, "exp": [w.exp_w + 16 - a.k_init] * 3, "evals": [[], [], []]}

    def cb(t, rec, st):
        te = t % a.epoch
        for l in range(3):
            lim = (1 << (state["bits"][l] - 1)) - 1
            assert np.abs(rec["w%d" % l].astype(np.int32)).max() <= lim
            if te % a.eval_every == 0:
                state["evals"][l].append(
                    math.ldexp(float(np.abs(rec["g%d" % l].astype(np.int64)).sum()), rec["eg%d" % l] - state["exp"][l])
                    / (rec["w%d" % l].size * w.batch))
        if te == a.epoch - 1:
            means = [sum(v) / len(v) for v in state["evals"]]
            assert st["gavg"] == means
            for l in range(3):
                k = state["bits"][l]
                want = k + 1 if means[l] < a.t_min and k < a.k_max else (
                    k - 1 if means[l] > a.t_max and k > a.k_min else k)
                assert st["bits"][l] == want
                assert st["exp_w"][l] == state["exp"][l] - (want - k)
                seen["up"] += want > k
                seen["down"] += want < k
            state["bits"], state["exp"] = list(st["bits"]), list(st["exp_w"])
            state["evals"] = [[], [], []]
        else:
            assert st["bits"] == state["bits"] and st["exp_w"] == state["exp"]

    O.apt_run(w, 12, callback=cb)
    assert seen["up"] > 0 and seen["down"] > 0


def test_apt_planted_policy_inversion_is_caught():
    """Inverting Algorithm 1's comparison (a plausible slip) changes the
    precision trajectory of the same run."""
    w, a = SMALL, SMALL.apt
    good = []
    O.apt_run(w, 8, callback=lambda t, r, st: good.append(list(st["bits"])))
    orig = O.apt_policy
    try:
        O.apt_policy = lambda bits, g, tmin, tmax, kmin, kmax: orig(bits, g, tmax, tmin, kmin, kmax)
        bad = []
        O.apt_run(w, 8, callback=lambda t, r, st: bad.append(list(st["bits"])))
    finally:
        O.apt_policy = orig
    assert good != bad
