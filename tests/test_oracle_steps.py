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


def _tiny_cnn():
    g = load_golden("tiny_cnn_step.txt")
    x = np.array(g["x"], np.int8).reshape(1, 4, 4, 1)
    W0 = np.array(g["W0"], np.int8).reshape(1, 3, 3, 1)
    W1 = np.array(g["W1"], np.int8).reshape(2, 3, 3, 1)
    W2 = np.array(g["W2"], np.int8).reshape(2, 2)
    convs = [(1, 1, 1), (1, 2, 2)]
    return g, x, [W0, W1, W2], np.array(g["label"], np.int32), convs


def test_tiny_cnn_step_hand_worked():
    g, x, weights, labels, convs = _tiny_cnn()
    r = O.cnn_step(weights, x, labels, convs)
    for k in ("y0", "a0", "y1", "a1", "p", "pa", "y2", "a2", "e2", "d2", "pe", "g2", "w2",
              "e1", "d1", "e0", "g1", "w1", "g0", "w0"):
        assert r[k].ravel().tolist() == g[k], k
    for k in ("ys0", "ys1", "ps", "ys2", "ds2", "gs2", "ws2", "nz2", "ds1", "gs1", "ws1", "nz1",
              "gs0", "ws0", "nz0"):
        assert r[k] == g[k][0], k


def test_tiny_cnn_planted_post_update_conv_dgrad_is_caught():
    """Conv delta propagation with the already-updated conv1 weights gives a
    different e0 than the hand-worked step."""
    g, x, weights, labels, convs = _tiny_cnn()
    e1 = np.array(g["e1"], np.int8).reshape(1, 2, 2, 2)
    a0 = np.array(g["a0"], np.int8).reshape(1, 4, 4, 1)
    w1_new = np.array(g["w1"], np.int8).reshape(2, 3, 3, 1)
    wrong, _, _ = O.requant_mask(O.conv2d_dgrad(e1, w1_new, (4, 4), 2), a0)
    assert wrong.ravel().tolist() != g["e0"]
    right, _, _ = O.requant_mask(O.conv2d_dgrad(e1, weights[1], (4, 4), 2), a0)
    assert right.ravel().tolist() == g["e0"]


def test_tiny_cnn_planted_pooled_delta_gate_is_caught():
    """Gating the pooled delta by the pooled activation (pa > 0) zeroes the
    channel whose pooled value rounded to 0 although some of its positions are
    active; the hand-worked e1 keeps it."""
    g, _, _, _, _ = _tiny_cnn()
    pe = np.array([g["pe"]], np.int8)
    pa = np.array([g["pa"]], np.int8)
    a1 = np.array(g["a1"], np.int8).reshape(1, 2, 2, 2)
    wrong = O.gap_bwd(np.where(pa > 0, pe, 0), a1)
    assert wrong.ravel().tolist() != g["e1"]
    assert O.gap_bwd(pe, a1).ravel().tolist() == g["e1"]


def _tiny_dfp2():
    g = load_golden("tiny_dfp16_2layer_step.txt")
    W0 = np.array(g["W0"], np.int16).reshape(2, 2)
    W1 = np.array(g["W1"], np.int16).reshape(1, 2)
    x = np.array([g["x"]], np.int16)
    return g, x, [W0, W1]


def test_tiny_dfp16_two_layer_step_hand_worked():
    g, x, weights = _tiny_dfp2()
    r = O.dfp16_step(weights, g["exp_w"][0], x, g["exp_x"][0], eta=g["eta"][0])
    for k in ("p0", "y0", "p1", "y1", "pd1", "e0", "pg1", "g1", "w1", "pg0", "g0", "w0"):
        assert r[k].ravel().tolist() == g[k], k
    for k in ("rs0", "ey0", "rs1", "ey1", "rsd1", "ee0", "rsg1", "eg1", "k1", "nz1",
              "rsg0", "eg0", "k0", "nz0"):
        assert r[k] == g[k][0], k
    assert r["ee1"] == g["ey1"][0]


def test_tiny_dfp16_planted_post_update_dgrad_is_caught():
    """DFP delta propagation with layer 1's already-updated weights gives a
    different e0 than the hand-worked step."""
    g, x, weights = _tiny_dfp2()
    e1 = np.array([g["y1"]], np.int16)
    w1_new = np.array(g["w1"], np.int16).reshape(1, 2)
    wrong, _, _, _ = O.dfp_down(O.dfp_linear_dgrad(e1, w1_new), g["ey1"][0] + g["exp_w"][0])
    assert wrong.ravel().tolist() != g["e0"]


def test_tiny_dfp16_planted_delta_exponent_mistake_is_caught():
    """Giving the propagated delta the activation's exponent (E_e + E_y0)
    instead of the weight's (E_e + E_W) changes E_G0 and so the update shift
    and the updated layer-0 weights."""
    g, x, weights = _tiny_dfp2()
    e0 = np.array([g["e0"]], np.int16)
    ee0_wrong = g["ey1"][0] + g["ey0"][0] + g["rsd1"][0]
    assert ee0_wrong != g["ee0"][0]
    gm, eg, _, _ = O.dfp_down(O.dfp_linear_wgrad(e0, x), ee0_wrong + g["exp_x"][0])
    w_wrong, _ = O.dfp_update(weights[0], gm, g["exp_w"][0] + g["eta"][0] - eg)
    assert w_wrong.ravel().tolist() != g["w0"]


def _tiny_static():
    g = load_golden("tiny_static_step.txt")
    x = np.array(g["x"], np.int8).reshape(2, 2)
    weights = [np.array(g["W0"], np.int8).reshape(2, 2), np.array(g["W1"], np.int8).reshape(2, 2)]
    static_q = [dict(offset=np.array(g["off%d" % l], np.int32), mult=np.array(g["mult%d" % l], np.int32),
                     k=np.array(g["k%d" % l], np.int32)) for l in range(2)]
    return g, x, weights, np.array(g["labels"], np.int32), static_q


def test_tiny_static_step_hand_worked():
    g, x, weights, labels, static_q = _tiny_static()
    r = O.mlp_step(weights, x, labels, static_q=static_q)
    for k in ("y0", "a0", "y1", "a1", "e1", "d1", "e0", "g1", "w1", "og1", "g0", "w0", "og0"):
        assert r[k].ravel().tolist() == g[k], k
    for k in ("ds1", "gs1", "ws1", "ogs1", "ows1", "gs0", "ws0", "ogs0", "ows0"):
        assert r[k] == g[k][0], k
    for l in range(2):
        assert r["off%d" % l].tolist() == g["new_off%d" % l]
        assert "ys%d" % l not in r               # no dynamic forward shift on a static layer


def test_tiny_static_planted_offset_gradient_from_propagated_delta_is_caught():
    """An offset gradient read after the layer's delta buffer was reused for
    the propagated delta (e0 instead of e1) gives a different layer-1 offset
    gradient than the hand-worked step."""
    g, _, _, _, _ = _tiny_static()
    wrong = O.offset_grad(np.array(g["e0"], np.int8).reshape(2, 2))
    assert wrong.tolist() != g["og1"]
    assert O.offset_grad(np.array(g["e1"], np.int8).reshape(2, 2)).tolist() == g["og1"]


def test_tiny_static_planted_offset_after_multiply_is_caught():
    """Adding the offset after the multiply (y*mult + off) instead of before it
    changes the hand-worked layer-0 activations."""
    g, x, weights, _, static_q = _tiny_static()
    y0 = O.linear_fwd(x, weights[0])
    q = static_q[0]
    wrong = np.clip(np.floor_divide(y0.astype(np.int64) * q["mult"] + q["offset"], 1 << q["k"].astype(np.int64)),
                    0, 127)
    assert wrong.ravel().tolist() != g["a0"]


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
