"""Partial-model training on the GPU ("Integer On-Device Training: Overview",
section 5): UINT8 input from a frozen prefix, the first layers frozen, the last
ones trained; bit-packed ReLU masks (section 8). Checked against the oracle."""
import numpy as np
import pytest

import oracle as O
import seeded_inputs as si
from gpu_util import GpuRun, compare_records, digest, import_ito, load_digests

pytestmark = pytest.mark.gpu


def test_partial_u8_lockstep_live():
    w = si.by_name(5)
    g = GpuRun(w)
    weights = si.make_weights(w)
    for t in range(3):
        x, labels = si.make_batch(w, t)
        rec = O.mlp_step(weights, x, labels, trainable_from=w.trainable_from)
        g.step(t)
        compare_records(rec, g.record(), t)
        weights = [rec["w%d" % l] for l in range(len(weights))]
    for l in range(w.trainable_from):
        assert np.array_equal(g.tensor("w%d" % l).reshape(weights[l].shape), si.make_weights(w)[l])
    assert g.ito.ito_get_error() == 0


def test_partial_u8_100_steps_digests():
    w = si.by_name(5)
    ref = load_digests(w)
    assert ref is not None and len(ref) == 100
    g = GpuRun(w)
    for t, d in enumerate(ref):
        x, labels = g.step(t)
        assert digest(x) == d["in.x"] and digest(labels) == d["in.labels"]
        r = g.record(("y", "a", "e", "d", "g", "w") if t < 3 else ("a", "e", "w"))
        bad = [k for k, v in r.items() if k in d and
               (digest(v) if isinstance(v, np.ndarray) else int(v)) != d[k]]
        assert not bad, "step %d differs from the oracle in %s" % (t, bad)


@pytest.mark.parametrize("index", [1, 2])
def test_packed_masks_lockstep(index):
    """The backward gate read from bit-packed masks gives the same step; the
    mask bits equal the oracle's packing of the ReLU outputs."""
    w = si.by_name(index)
    g = GpuRun(w, packed_masks=True)
    weights = si.make_weights(w)
    for t in range(2):
        x, labels = si.make_batch(w, t)
        rec = O.mlp_step(weights, x, labels) if w.kind == "mlp" else O.cnn_step(weights, x, labels, w.convs)
        g.step(t)
        compare_records(rec, g.record(), t)
        n_relu = len(weights) - 1
        for l in range(n_relu):
            a = rec["a%d" % l]
            a2 = a.reshape(-1, a.shape[-1])
            assert np.array_equal(g.tensor("m%d" % l).view(np.uint8), O.pack_relu_mask(a2).ravel()), "m%d" % l
        weights = [rec["w%d" % l] for l in range(len(weights))]


def test_u8_contraction_exact_at_extremes():
    """All inputs 255 and all first-layer weights -128: every 512-term chunk
    reaches 512 * 32640 (just under 2^24) and y0 = 784 * 255 * -128 exactly."""
    import torch
    ito = import_ito()
    layers = [ito.LayerDesc(ito.ITO_LAYER_LINEAR_RELU, 784, 1024, 0, 0, 0),
              ito.LayerDesc(ito.ITO_LAYER_LINEAR, 1024, 16, 0, 0, 0)]
    m = ito.Model(layers, 64, input_uint8=True)
    W0 = np.full((1024, 784), -128, np.int8)
    W0[1::2] = 127
    m.set_weights(0, W0)
    m.set_weights(1, np.ones((16, 1024), np.int8))
    x = np.full((64, 784), 255, np.uint8)
    labels = np.zeros(64, np.int32)
    m.train_step(torch.from_numpy(x).cuda(), torch.from_numpy(labels).cuda())
    torch.cuda.synchronize()
    y0 = m.tensor("y0").cpu().numpy().reshape(64, 1024)
    assert (y0[:, 0::2] == 784 * 255 * -128).all() and (y0[:, 1::2] == 784 * 255 * 127).all()
    assert np.array_equal(y0, O.linear_fwd_u8(x, W0))
    assert ito.ito_get_error() == 0


@pytest.mark.parametrize("index", [1, 2, 5])
def test_pingpong_grads_lockstep(index):
    """Deltas in two shared buffers ("Grad Buffers", section 8): the steps equal
    the oracle's (every tensor still readable, the weights of every layer over
    several steps); the buffers really are shared (e2 aliases e0)."""
    w = si.by_name(index)
    g = GpuRun(w, pingpong_grads=True)
    weights = si.make_weights(w)
    for t in range(3):
        x, labels = si.make_batch(w, t)
        if w.kind == "mlp":
            rec = O.mlp_step(weights, x, labels, trainable_from=w.trainable_from)
        else:
            rec = O.cnn_step(weights, x, labels, w.convs)
        g.step(t)
        compare_records(rec, g.record(), t)
        weights = [rec["w%d" % l] for l in range(len(weights))]
    if g.n_layers > 2:
        assert g.model.tensor("e2").data_ptr() == g.model.tensor("e0").data_ptr()
