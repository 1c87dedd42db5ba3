"""Whole training steps of the CUDA model against the CPU oracle: every int8
and int32 tensor and every shift/max scalar after every step.

Short runs are compared tensor by tensor with the oracle run live; the
100-step runs are compared against per-step digests of the oracle's tensors
(tests/golden/digests_*.jsonl, written by tests/golden/make_digests.py from
the oracle alone)."""
import numpy as np
import pytest

import oracle as O
import seeded_inputs as si
from gpu_util import GpuRun, compare_records, digest, load_digests

pytestmark = pytest.mark.gpu


def _oracle_step(w, weights, t, route):
    x, labels = si.make_batch(w, t)
    if w.kind == "mlp":
        return O.mlp_step(weights, x, labels, route=route)
    return O.cnn_step(weights, x, labels, w.convs)


@pytest.mark.parametrize("index,steps,route", [(0, 100, "loops"), (1, 3, "loops"), (2, 2, "loops"),
                                               (3, 1, "f64")])
def test_model_lockstep_live(index, steps, route):
    w = si.by_name(index)
    g = GpuRun(w)
    weights = si.make_weights(w)
    for t in range(steps):
        rec = _oracle_step(w, weights, t, route)
        g.step(t)
        compare_records(rec, g.record(), t)
        weights = [rec["w%d" % l] for l in range(len(weights))]
    assert g.ito.ito_get_error() == 0


@pytest.mark.parametrize("index", [1, 2, 3])
def test_model_100_steps_digests(index):
    w = si.by_name(index)
    ref = load_digests(w)
    assert ref is not None, "digest file for %s missing" % w.name
    g = GpuRun(w)
    full_steps = 3                       # int32 tensors too for the first steps
    for t, d in enumerate(ref):
        x, labels = g.step(t)
        assert digest(x) == d["in.x"] and digest(labels) == d["in.labels"], "input generator diverged"
        kinds = ("y", "a", "e", "d", "g", "w") if t < full_steps else ("a", "e", "w")
        r = g.record(kinds)
        bad = []
        for k, v in r.items():
            want = d.get(k)
            if want is None:
                continue
            got = digest(v) if isinstance(v, np.ndarray) else int(v)
            if got != want:
                bad.append(k)
        assert not bad, "step %d differs from the oracle in %s" % (t, bad)
    assert len(ref) == 100


@pytest.mark.parametrize("index,steps", [(0, 100), (2, 3)])
def test_model_graph_replay_lockstep(index, steps):
    """Steps replayed from captured CUDA graphs (side stream, two fixed input
    buffers) match the oracle step by step."""
    import torch
    w = si.by_name(index)
    g = GpuRun(w)
    g.model.use_graphs(True)
    stream = torch.cuda.Stream()
    bufs = [(torch.empty(si.input_shape(w), dtype=torch.int8, device="cuda"),
             torch.empty(w.batch, dtype=torch.int32, device="cuda")) for _ in range(2)]
    weights = si.make_weights(w)
    for t in range(steps):
        x, labels = si.make_batch(w, t)
        xb, lb = bufs[t % 2]
        with torch.cuda.stream(stream):
            xb.copy_(torch.from_numpy(x))
            lb.copy_(torch.from_numpy(labels))
            g.model.train_step(xb, lb, stream=stream)
        stream.synchronize()
        rec = _oracle_step(w, weights, t, "loops")
        compare_records(rec, g.record(), t)
        weights = [rec["w%d" % l] for l in range(len(weights))]
    assert g.ito.ito_get_error() == 0


@pytest.mark.parametrize("index,pingpong", [(1, False), (6, True), (2, True)])
def test_overlap_modes_give_identical_steps(index, pingpong):
    """The backward overlap moves bandwidth passes to a second stream; every
    tensor and statistic after three steps is the same in all three modes
    (one stream, requantisation + updates overlapped, updates only). The
    default, overlapped mode is the one the lockstep and digest tests compare
    with the oracle."""
    w = si.by_name(index)
    results = []
    for mode in (0, 1, 2):
        g = GpuRun(w, pingpong_grads=pingpong)
        g.model.set_overlap(mode)
        for t in range(3):
            g.step(t)
        results.append(g.record())
    for mode, r in zip((1, 2), results[1:]):
        assert r.keys() == results[0].keys()
        for k in r:
            assert np.array_equal(np.asarray(r[k]), np.asarray(results[0][k])), (mode, k)
