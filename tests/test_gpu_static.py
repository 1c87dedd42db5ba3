"""The TI library's own forward on the GPU: static per-channel
requantisation with INT32 offsets trained by the backward pass, against the
oracle; and the checkpoint round trip."""
import os
import tempfile

import numpy as np
import pytest

import oracle as O
import seeded_inputs as si
from gpu_util import GpuRun, compare_records, digest, load_digests

pytestmark = pytest.mark.gpu


def test_static_requant_lockstep_live():
    w = si.by_name(6)
    g = GpuRun(w)
    weights = si.make_weights(w)
    static_q = si.make_static_requant(w)
    for t in range(3):
        x, labels = si.make_batch(w, t)
        rec = O.mlp_step(weights, x, labels, static_q=static_q)
        g.step(t)
        compare_records(rec, g.record(), t)
        weights = [rec["w%d" % l] for l in range(len(weights))]
        static_q = [dict(q, offset=rec["off%d" % l]) for l, q in enumerate(static_q)]
    assert g.ito.ito_get_error() == 0


def _check_digest_steps(g, ref, steps):
    for t in steps:
        d = ref[t]
        x, labels = g.step(t)
        assert digest(x) == d["in.x"] and digest(labels) == d["in.labels"]
        r = g.record(("y", "a", "e", "d", "g", "w") if t < 3 else ("a", "e", "w"))
        bad = [k for k, v in r.items() if k in d and
               (digest(v) if isinstance(v, np.ndarray) else int(v)) != d[k]]
        assert not bad, "step %d differs from the oracle in %s" % (t, bad)


def test_static_requant_100_steps_digests():
    w = si.by_name(6)
    ref = load_digests(w)
    assert ref is not None and len(ref) == 100
    _check_digest_steps(GpuRun(w), ref, range(100))


@pytest.mark.parametrize("index", [1, 6])
def test_checkpoint_resume_matches_straight_run(index):
    """50 steps, save, load into a fresh model, 50 more steps: every step of
    the resumed run matches the oracle's 100-step digests (weights, offsets
    and the step's tensors)."""
    w = si.by_name(index)
    ref = load_digests(w)
    g = GpuRun(w)
    _check_digest_steps(g, ref, range(50))
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "ckpt.ito")
        g.model.save(path)
        g2 = GpuRun(w)                     # fresh model with the initial weights
        g2.model.load(path)
    _check_digest_steps(g2, ref, range(50, 100))
