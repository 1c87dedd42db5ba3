"""Helpers shared by the GPU tests: run the CUDA model on a seeded workload and
read its tensors back as numpy arrays under the oracle's record names."""
import hashlib
import json
import os

import numpy as np

import seeded_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def digest(a: np.ndarray) -> str:
    # identical to tests/golden/make_digests.py
    a = np.ascontiguousarray(a)
    return hashlib.sha256(a.astype(a.dtype.newbyteorder("<"), copy=False).tobytes()).hexdigest()[:24]


def load_digests(workload):
    path = os.path.join(ROOT, "tests", "golden", "digests_%s.jsonl" % workload.name)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        return [json.loads(line) for line in f]


def import_ito():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need a CUDA device")
    import integer_only_nn_gb300 as ito   # raises if the library is not built
    return ito


class GpuRun:
    """A CUDA model of a seeded mlp/cnn workload, stepped one batch at a time."""

    def __init__(self, workload, batch=None, packed_masks=False, pingpong_grads=False, speculate_min_elems=0):
        import torch
        self.torch = torch
        self.ito = import_ito()
        self.w = workload
        self.batch = batch or workload.batch
        self.model = self.ito.Model(self.ito.layers_for(workload), self.batch, input_uint8=workload.input_uint8,
                                    trainable_from=workload.trainable_from, packed_masks=packed_masks,
                                    pingpong_grads=pingpong_grads, speculate_min_elems=speculate_min_elems)
        self.pingpong = pingpong_grads
        self.n_layers = self.model.n_weight_layers
        for l, W in enumerate(si.make_weights(workload)):
            self.model.set_weights(l, W)
        self.static_q = si.make_static_requant(workload) if workload.kind == "mlp" else None
        if self.static_q:
            for l, q in enumerate(self.static_q):
                if q is not None:
                    self.model.set_static_requant(l, q["offset"], q["mult"], q["k"])

    def step(self, t):
        x, labels = si.make_batch(self.w, t)
        x, labels = x[: self.batch], labels[: self.batch]
        xd = self.torch.from_numpy(np.ascontiguousarray(x)).cuda()
        ld = self.torch.from_numpy(np.ascontiguousarray(labels)).cuda()
        self.model.train_step(xd, ld)
        self.torch.cuda.synchronize()
        return x, labels

    def unwritten_int32(self):
        """The int32 contraction results the model does not write: with
        speculative requantisation on, those of the contractions whose epilogue
        requantises ("y<l>" forward, "d<l>" delta propagation)."""
        if not self.model.speculation():
            return set()
        nl = self.n_layers
        used = self.model.tensor("spec").cpu().numpy()[4 * nl: 6 * nl]
        return {"y%d" % l for l in range(nl) if used[l]} | {"d%d" % l for l in range(nl) if used[nl + l]}

    def names(self, kinds=("y", "a", "e", "d", "g", "w")):
        out = []
        first = self.w.trainable_from
        skip = self.unwritten_int32()
        for l in range(self.n_layers):
            for k in kinds:
                if "%s%d" % (k, l) in skip:
                    continue
                if k == "d" and l <= first:
                    continue
                if k in ("e", "g") and l < first:
                    continue
                if k == "e" and self.pingpong and l >= 2:
                    continue    # aliases the buffer of layer l % 2
                out.append("%s%d" % (k, l))
        if self.w.kind == "cnn":
            out += ["p", "pa", "pe"]
        if self.static_q:
            out += ["off%d" % l for l in range(self.n_layers)]
            if "g" in kinds:
                out += ["og%d" % l for l in range(self.w.trainable_from, self.n_layers)]
        return out

    def tensor(self, name):
        return self.model.tensor(name).cpu().numpy()

    def record(self, kinds=("y", "a", "e", "d", "g", "w")):
        r = {n: self.tensor(n) for n in self.names(kinds)}
        r.update(self.model.stats())
        if self.w.kind != "cnn":
            r.pop("pmax", None)
            r.pop("ps", None)
        return r


def compare_records(oracle_rec, gpu_rec, step):
    """Element-by-element comparison of every tensor and scalar the GPU record holds."""
    bad = []
    for k, v in gpu_rec.items():
        if k not in oracle_rec:
            continue
        o = oracle_rec[k]
        if isinstance(o, np.ndarray):
            if o.size != np.asarray(v).size or not np.array_equal(o.ravel(), np.asarray(v).ravel()):
                n = int((o.ravel() != np.asarray(v).ravel()).sum()) if o.size == np.asarray(v).size else -1
                bad.append("%s (%d elements differ)" % (k, n))
        elif int(o) != int(v):
            bad.append("%s: oracle %d gpu %d" % (k, int(o), int(v)))
    assert not bad, "step %d: %s" % (step, "; ".join(bad))
