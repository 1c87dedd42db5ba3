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


@pytest.mark.parametrize("index,steps,route,speculate", [(0, 100, "loops", True), (1, 3, "loops", True),
                                                         (1, 3, "loops", False), (2, 2, "loops", True),
                                                         (3, 1, "f64", True)])
def test_model_lockstep_live(index, steps, route, speculate):
    """Every step's tensors and scalars against the oracle run live. With
    speculative requantisation on (the default) the int32 results of the
    speculating contractions are not written; the run with it off compares
    them too."""
    w = si.by_name(index)
    g = GpuRun(w)
    g.model.set_speculation(speculate)
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


@pytest.mark.parametrize("index,pingpong,spec_min", [(1, False, 0), (6, True, 0), (2, True, 0), (1, False, 1),
                                                    (2, False, 0), (0, False, 0), (3, False, 0)])
def test_overlap_modes_give_identical_steps(index, pingpong, spec_min):
    """The backward overlap moves work to a second stream; every tensor and
    statistic after three steps is the same in every mode (one stream,
    requantisation + updates overlapped, updates only, and, without ping-pong
    delta buffers or static requantisation, weight gradients + updates beside
    the delta chain), also with speculative requantisation (whose checks and
    re-launches stay on the caller's stream). A new model's default mode is the
    one the lockstep and digest tests compare with the oracle."""
    w = si.by_name(index)
    modes = (0, 1, 2) if pingpong or w.static_requant else (0, 1, 2, 3)
    results = []
    for mode in modes:
        # spec_min = 1: every eligible contraction requantises speculatively
        g = GpuRun(w, pingpong_grads=pingpong, speculate_min_elems=spec_min)
        g.model.set_overlap(mode)
        for t in range(3):
            g.step(t)
        results.append(g.record())
    for mode, r in zip(modes[1:], results[1:]):
        assert r.keys() == results[0].keys()
        for k in r:
            assert np.array_equal(np.asarray(r[k]), np.asarray(results[0][k])), (mode, k)


def test_overlap_mode_3_refused_with_shared_delta_buffers():
    g = GpuRun(si.by_name(1), pingpong_grads=True)
    with pytest.raises(g.ito.ItoError):
        g.model.set_overlap(3)


@pytest.mark.parametrize("index,steps", [(0, 6), (1, 4), (5, 3), (3, 3)])
def test_speculation_gives_identical_steps(index, steps):
    """Speculative requantisation in the contraction epilogues changes no
    result: with it on and off every tensor and statistic is the same after
    each step. The predictions of step t are the shifts of step t-1 on the
    slots whose contraction plan took the fused epilogue, and the model's
    counters score each step's predictions at the start of the next."""
    w = si.by_name(index)
    runs = []
    for on in (False, True):
        # every contraction that can speculate does, however small its output
        g = GpuRun(w, speculate_min_elems=1)
        g.model.set_speculation(on)
        runs.append(g)
    nl = runs[0].n_layers
    hits = misses = 0
    for t in range(steps):
        recs = []
        for g in runs:
            g.step(t)
            recs.append(g.record())
        # the speculating contractions write no int32 result; everything else is identical
        assert set(recs[1].keys()) == set(recs[0].keys()) - runs[1].unwritten_int32()
        for k in recs[1]:
            assert np.array_equal(np.asarray(recs[0][k]), np.asarray(recs[1][k])), (t, k)
        spec = runs[1].model.tensor("spec").cpu().numpy()
        pred, last, used = spec[: 2 * nl], spec[2 * nl: 4 * nl], spec[4 * nl: 6 * nl]
        off = runs[0].model.tensor("spec").cpu().numpy()
        assert (off[: 2 * nl] == -1).all()
        assert np.array_equal(off[2 * nl: 6 * nl], spec[2 * nl: 6 * nl]), t
        # re-launch words of the speculating slots: 0 where the prediction held, else the
        # step's shift + 1 (a missed prediction, or none yet: the re-launch wrote the outputs)
        redo = spec[6 * nl: 8 * nl]
        u = used != 0
        held = u & (pred >= 0) & (pred == last)
        assert np.array_equal(redo[u], np.where(held[u], 0, last[u] + 1)), t
        assert (redo[~u] == 0).all(), t
        assert (pred[used == 0] == -1).all()
        # the counters hold the steps before this one
        cnt = runs[1].model.tensor("spec_count").cpu().numpy()
        assert (int(cnt[0]), int(cnt[1])) == (hits, misses), t
        assert (runs[0].model.tensor("spec_count").cpu().numpy() == 0).all()
        act = (used != 0) & (pred >= 0)
        hits += int((pred[act] == last[act]).sum())
        misses += int((pred[act] != last[act]).sum())
        if t == 0:
            assert not act.any()
    if index in (1, 3, 5):
        # the hidden layers' forward and delta-propagation contractions speculate
        assert used.sum() > 0 and hits > 0
    assert runs[0].ito.ito_get_error() == 0


@pytest.mark.parametrize("index,steps,route", [(1, 4, "loops"), (3, 2, "f64")])
def test_mispredicted_shift_relaunch_matches_oracle(index, steps, route):
    """Forced mispredictions: before steps 1, 2, ... every speculating slot's
    prediction is set one or more off the true previous shift. The epilogue
    then requantises with the wrong shift, the check records the step's shift
    in the re-launch word, and the contraction's re-launch rewrites the int8
    and bf16 outputs; every tensor and scalar still matches the oracle."""
    import torch
    w = si.by_name(index)
    g = GpuRun(w, speculate_min_elems=1)
    assert g.model.speculation()
    nl = g.n_layers
    weights = si.make_weights(w)
    for t in range(steps):
        spec = g.model.tensor("spec")
        used = spec[4 * nl: 6 * nl] != 0
        if t > 0:
            # the step's predictions are read from the previous step's shifts (the "last" block)
            last = spec[2 * nl: 4 * nl]
            last.copy_(torch.where(used, last + (1 if t % 2 else 3), last))
            torch.cuda.synchronize()
        rec = _oracle_step(w, weights, t, route)
        g.step(t)
        compare_records(rec, g.record(), t)
        weights = [rec["w%d" % l] for l in range(len(weights))]
        spec = g.model.tensor("spec").cpu().numpy()
        pred, last, used, redo = (spec[i * 2 * nl: (i + 1) * 2 * nl] for i in range(4))
        if t > 0:
            act = (used != 0) & (pred >= 0)
            assert act.any()
            # (a shift that itself moved by the offset makes a prediction hold by chance)
            assert (pred[act] != last[act]).any(), t
            assert np.array_equal(redo[act], np.where(pred[act] == last[act], 0, last[act] + 1)), t
    assert g.ito.ito_get_error() == 0


def test_moving_weights_at_4096_width_with_speculation():
    """The 4096-wide MLP at batch 1024 with inputs in [-7, 7]: the first layer's
    weights move every step (its gradient shift is 8, weight shift 6), while the
    forward and delta-propagation contractions of 2^22 outputs run on the CTA
    pair with a speculating epilogue (the default threshold). Three steps in
    lockstep with the oracle: from the second step on, the speculating forward
    of layer 0 predicts from a step whose weights have since changed."""
    w = si.by_name(8)
    g = GpuRun(w)
    assert g.model.speculation()
    nl = g.n_layers
    weights = si.make_weights(w)
    for t in range(3):
        rec = _oracle_step(w, weights, t, "f64")
        g.step(t)
        compare_records(rec, g.record(), t)
        assert rec["nz0"] > 0 and g.model.stats()["nz0"] == rec["nz0"]
        assert not np.array_equal(rec["w0"], weights[0])
        weights = [rec["w%d" % l] for l in range(len(weights))]
        used = g.model.tensor("spec").cpu().numpy()[4 * nl: 6 * nl]
        assert used[0] != 0 and used[nl + 1] != 0      # layer 0 forward, layer 1 delta propagation
    assert g.ito.ito_get_error() == 0


def test_speculation_covers_large_contractions_only():
    """By default only contractions with at least 2^22 output elements
    speculate: none of the 784-1024x3-10 MLP (batch 256), all the 4096-wide
    forward and delta-propagation ones of the batch-8192 MLP (not its
    1000-wide logits, whose row is not a multiple of 16 bytes). Every delta
    propagation of the latter speculates, so it takes overlap mode 3."""
    g = GpuRun(si.by_name(1))
    nl = g.n_layers
    assert (g.model.tensor("spec").cpu().numpy()[4 * nl: 6 * nl] == 0).all()
    assert g.model.overlap() == 1
    g = GpuRun(si.by_name(3))
    nl = g.n_layers
    used = g.model.tensor("spec").cpu().numpy()[4 * nl: 6 * nl]
    assert list(used[:nl]) == [1, 1, 1, 1, 0]
    assert list(used[nl:]) == [0, 1, 1, 1, 1]
    assert g.model.overlap() == 3


@pytest.mark.parametrize("index,graphs", [(1, True), (0, False), (3, True)])
def test_pipelined_host_steps_match_device_steps(index, graphs):
    """ito_train_step_host_async (input copies on the model's copy stream into two
    alternating buffers, overlapping the previous step) trains exactly as steps on device
    inputs: the same weights and activations after every step, and the stats copied back
    are the step's."""
    import torch
    w = si.by_name(index)
    a, b = GpuRun(w), GpuRun(w)
    stream = torch.cuda.Stream()
    a.model.use_graphs(graphs)
    batches = [si.make_batch(w, t) for t in range(5)]
    xs_h = [torch.from_numpy(np.ascontiguousarray(x)).pin_memory() for x, _ in batches]
    ls_h = [torch.from_numpy(np.ascontiguousarray(lab)).pin_memory() for _, lab in batches]
    st_h = torch.zeros(a.model.num_stats(), dtype=torch.int32).pin_memory()
    for t in range(len(batches)):
        a.model.train_step_host_async(xs_h[t], ls_h[t], st_h, stream=stream)
        if t % 2 == 1:
            stream.synchronize()    # sometimes wait, sometimes queue two steps
    stream.synchronize()
    for t in range(len(batches)):
        b.step(t)
    names = [n for n in a.names(("a", "e", "w")) if n in b.names(("a", "e", "w"))]
    for n in names:
        assert np.array_equal(a.tensor(n), b.tensor(n)), n
    stats_b = b.model.tensor("stats").cpu().numpy()
    assert np.array_equal(st_h.numpy(), stats_b)
    assert a.ito.ito_get_error() == 0


@pytest.mark.parametrize("spec_min", [0, 1])
def test_infer_matches_oracle_forward(spec_min):
    """ito_infer (the forward pass alone, "INTODT_Infer") after a few training steps
    gives the oracle's logits for the current weights, with the speculating forward
    contractions (spec_min = 1: every eligible one, however small) and without."""
    import torch
    w = si.by_name(1)
    g = GpuRun(w, speculate_min_elems=spec_min)
    weights = si.make_weights(w)
    for t in range(3):
        rec = _oracle_step(w, weights, t, "loops")
        g.step(t)
        weights = [rec["w%d" % l] for l in range(len(weights))]
    x, labels = si.make_batch(w, 7)
    logits = torch.empty((w.batch, w.dims[-1]), dtype=torch.int8, device="cuda")
    g.model.infer(torch.from_numpy(np.ascontiguousarray(x)).cuda(), logits)
    torch.cuda.synchronize()
    ref = O.mlp_step(weights, x, labels, route="loops")
    nl = len(weights)
    assert np.array_equal(logits.cpu().numpy(), ref["a%d" % (nl - 1)])
    for l in range(nl):
        assert np.array_equal(g.tensor("a%d" % l).ravel(), ref["a%d" % l].ravel()), l
    assert g.ito.ito_get_error() == 0


@pytest.mark.parametrize("index", [0, 3])
def test_model_step_bad_label_sets_error_word(index):
    """A label outside [0, C) in a training step (where the oracle's top error aborts)
    records ITO_ERR_ARG in the device error word: the logits' requantisation, which
    computes the top error, checks every row's label (the 10-class scalar pass and the
    1000-class vectorised one)."""
    import torch
    w = si.by_name(index)
    g = GpuRun(w)
    x, labels = si.make_batch(w, 0)
    labels = labels.copy()
    labels[len(labels) // 2] = w.classes
    assert g.ito.ito_get_error() == 0
    g.model.train_step(torch.from_numpy(np.ascontiguousarray(x)).cuda(),
                       torch.from_numpy(np.ascontiguousarray(labels)).cuda())
    torch.cuda.synchronize()
    assert g.ito.ito_get_error() == g.ito.ITO_ERR_ARG
    assert g.ito.ito_get_error() == 0


@pytest.mark.parametrize("index", [1, 2])
def test_overlap_mode_3_in_graphs(index):
    """Overlap mode 3 captured into a CUDA graph (cross-stream events as graph edges) on a
    non-default stream trains exactly as mode 1 stepping directly: every tensor and
    statistic after four steps (one direct step, the capture and its launch, two replays;
    the same input buffers, refilled each step)."""
    import torch
    w = si.by_name(index)
    a, b = GpuRun(w), GpuRun(w)
    a.model.set_overlap(1)
    b.model.set_overlap(3)
    b.model.use_graphs(True)
    stream = torch.cuda.Stream()
    x0, l0 = si.make_batch(w, 0)
    xd = torch.empty(x0.shape, dtype=torch.int8, device="cuda")
    ld = torch.empty(l0.shape, dtype=torch.int32, device="cuda")
    for t in range(4):
        a.step(t)
        x, labels = si.make_batch(w, t)
        xd.copy_(torch.from_numpy(np.ascontiguousarray(x)))
        ld.copy_(torch.from_numpy(np.ascontiguousarray(labels)))
        torch.cuda.synchronize()
        b.model.train_step(xd, ld, stream=stream)
        torch.cuda.synchronize()
    ra, rb = a.record(), b.record()
    assert ra.keys() == rb.keys()
    for k in ra:
        assert np.array_equal(np.asarray(ra[k]), np.asarray(rb[k])), k
    assert a.ito.ito_get_error() == 0
