"""Pins of the oracle's training-step order: hand-worked steps (tests/golden),
invariants that hold at any size, agreement of the two contraction routes, and
planted mistakes that the pins must catch."""
import numpy as np
import pytest

import oracle as O
import seeded_inputs as si
from conftest import load_golden


def test_tiny_mlp_step_hand_worked():
    g = load_golden("tiny_mlp_step.txt")
    W0 = np.array(g["W0"], np.int8).reshape(2, 2)
    W1 = np.array(g["W1"], np.int8).reshape(2, 2)
    x = np.array([g["x"]], np.int8)
    r = O.mlp_step([W0, W1], x, np.array(g["label"], np.int32))
    for k in ("y0", "a0", "y1", "a1", "e1", "d1", "e0", "g1", "w1", "g0", "w0"):
        assert r[k].ravel().tolist() == g[k], k
    for k in ("ys0", "ys1", "ds1", "gs1", "ws1", "gs0", "ws0"):
        assert r[k] == g[k][0], k


def test_tiny_mlp_planted_order_mistake_is_caught():
    """Delta propagation with the already-updated weight (a plausible order
    mistake) gives a different e0 than the hand-worked step."""
    g = load_golden("tiny_mlp_step.txt")
    W1_new = np.array(g["w1"], np.int8).reshape(2, 2)
    e1 = np.array([g["e1"]], np.int8)
    a0 = np.array([g["a0"]], np.int8)
    wrong, _, _ = O.requant_mask(O.linear_dgrad(e1, W1_new), a0)
    assert wrong.ravel().tolist() != g["e0"]


def test_tiny_dfp16_step_hand_worked():
    g = load_golden("tiny_dfp16_step.txt")
    W0 = np.array(g["W0"], np.int16).reshape(1, 2)
    x = np.array([g["x"]], np.int16)
    r = O.dfp16_step([W0], g["exp_w"][0], x, g["exp_x"][0], eta=g["eta"][0])
    for k in ("p0", "y0", "pg0", "g0", "w0"):
        assert r[k].ravel().tolist() == g[k], k
    for k in ("rs0", "ey0", "rsg0", "eg0", "k0"):
        assert r[k] == g[k][0], k


def _check_nitI_invariants(rec, n_layers):
    for k, v in rec.items():
        if isinstance(v, np.ndarray) and v.dtype == np.int8:
            assert v.min() >= -128 and v.max() <= 127
        if k[:2] in ("ys", "ds", "gs", "ws"):
            assert v >= 0
    for l in range(n_layers - 1):
        if "a%d" % l in rec:
            assert rec["a%d" % l].min() >= 0            # ReLU outputs
    for l in range(n_layers - 1):
        a, e = rec.get("a%d" % l), rec.get("e%d" % l)
        if a is not None and e is not None and a.shape == e.shape:
            assert not e[a <= 0].any()                  # gated deltas
    for l in range(n_layers):
        s, m = rec["gs%d" % l], rec["gmax%d" % l]
        assert s == max(0, int(m).bit_length() - 7)
        assert rec["ws%d" % l] == max(0, s - 2)


def test_mlp_small_100_steps_invariants():
    w = si.by_name(0)
    O.run_steps(w, 100, callback=lambda t, r: _check_nitI_invariants(r, 2))


def test_mlp_routes_agree_one_step():
    w = si.by_name(1)
    weights = si.make_weights(w)
    x, labels = si.make_batch(w, 0)
    a = O.mlp_step(weights, x, labels, route="loops")
    b = O.mlp_step(weights, x, labels, route="f64")
    assert a.keys() == b.keys()
    for k in a:
        assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), k
    _check_nitI_invariants(a, 4)


def test_cnn_small_step_invariants():
    # the CNN workload's structure on a 2-image batch
    w = si.by_name(2)
    weights = si.make_weights(w)
    x, labels = si.make_batch(w, 0)
    r = O.cnn_step(weights, x[:2], labels[:2], w.convs)
    assert r["y0"].shape == (2, 32, 32, 64) and r["y1"].shape == (2, 16, 16, 128)
    assert r["y2"].shape == (2, 8, 8, 256) and r["p"].shape == (2, 256)
    assert r["pa"].min() >= 0
    _check_nitI_invariants(r, 4)
    # pooled-delta broadcast gated by conv3's ReLU
    e2 = r["e2"]
    assert (e2 == np.where(r["a2"] > 0, r["pe"][:, None, None, :], 0)).all()


def test_dfp16_small_steps_exponents_track():
    w = si.Workload(99, "dfp16_small", "dfp16", 16, dims=(64, 48, 32), sigma=4096.0,
                    lim=32767, exp_x=-12, exp_w=-17, eta=8)
    seen = []

    def cb(t, r):
        for l in range(2):
            assert r["ey%d" % l] == (w.exp_x if l == 0 else r["ey%d" % (l - 1)]) + w.exp_w + r["rs%d" % l]
            assert np.abs(r["y%d" % l]).max() <= 32767
        seen.append(r["nz0"] + r["nz1"])
    O.run_steps(w, 5, callback=cb)
    assert sum(seen) > 0


def test_dfp16_routes_agree():
    w = si.Workload(98, "dfp16_mid", "dfp16", 64, dims=(256, 128, 96), sigma=4096.0,
                    lim=32767, exp_x=-12, exp_w=-17)
    weights = si.make_weights(w)
    x, _ = si.make_batch(w, 0)
    a = O.dfp16_step(weights, w.exp_w, x, w.exp_x, route="loops")
    b = O.dfp16_step(weights, w.exp_w, x, w.exp_x, route="f64")
    for k in a:
        assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), k


def test_partial_training_equals_training_the_suffix():
    """Training with the first k layers frozen ("trainable_layers_from_last")
    equals training the remaining layers on the frozen prefix's output; the
    frozen weights do not change."""
    w = si.by_name(5)
    weights = si.make_weights(w)
    x, labels = si.make_batch(w, 0)
    k = w.trainable_from
    r = O.mlp_step(weights, x, labels, trainable_from=k)
    for l in range(k):
        assert np.array_equal(r["w%d" % l], weights[l])
        assert "g%d" % l not in r and "d%d" % (l + 1) not in r
    prefix_out = r["a%d" % (k - 1)]
    s = O.mlp_step(weights[k:], prefix_out, labels)
    for name in ("y", "a", "e", "d", "g", "w"):
        for l in range(len(weights) - k):
            key = "%s%d" % (name, l)
            if key in s:
                assert np.array_equal(s[key], r["%s%d" % (name, l + k)]), key


def test_partial_planted_leak_into_frozen_layer_is_caught():
    """A backward that does not stop at the frozen boundary (planted here by
    moving the boundary one layer down) propagates a delta into the last frozen
    layer and computes its weight gradient: exactly the records the identity
    above requires to be absent."""
    w = si.by_name(5)
    weights = si.make_weights(w)
    x, labels = si.make_batch(w, 0)
    k = w.trainable_from
    good = O.mlp_step(weights, x, labels, trainable_from=k)
    leaked = O.mlp_step(weights, x, labels, trainable_from=k - 1)
    for key in ("d%d" % k, "g%d" % (k - 1)):
        assert key in leaked and key not in good
    assert np.array_equal(good["w%d" % k], leaked["w%d" % k])   # the boundary layer itself agrees
