"""Write per-step digests of every tensor of an oracle training run.

Usage: python tests/golden/make_digests.py <workload index> [steps]

Calls only the CPU oracle (oracle/) and the seeded input generator. Output:
tests/golden/digests_<workload name>.jsonl, one JSON object per step: tensor
names map to the first 24 hex digits of the SHA-256 of the tensor's
little-endian, row-major bytes in its own dtype (int8, int16, int32 or int64);
scalar names map to their integer value. The inputs of each step are digested
too ("in.x", "in.labels") so that a generator divergence between machines shows
up apart from a training-step divergence.
"""
import hashlib
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as O          # noqa: E402
import seeded_inputs as si  # noqa: E402


def digest(a: np.ndarray) -> str:
    a = np.ascontiguousarray(a)
    return hashlib.sha256(a.astype(a.dtype.newbyteorder("<"), copy=False).tobytes()).hexdigest()[:24]


def record_digests(rec: dict) -> dict:
    out = {}
    for k, v in sorted(rec.items()):
        out[k] = digest(v) if isinstance(v, np.ndarray) else int(v)
    return out


def main():
    w = si.by_name(int(sys.argv[1]))
    steps = int(sys.argv[2]) if len(sys.argv) > 2 else 100
    path = os.path.join(ROOT, "tests", "golden", "digests_%s.jsonl" % w.name)
    route = "f64" if w.kind in ("mlp", "dfp16") else "loops"
    tmp = path + ".tmp"
    t0 = time.time()
    with open(tmp, "w") as f:
        def cb(t, rec, extra=None):
            x, labels = si.make_batch(w, t)
            d = {"step": t, "in.x": digest(x)}
            if labels is not None:
                d["in.labels"] = digest(labels)
            d.update(record_digests(rec))
            d.update(extra or {})
            f.write(json.dumps(d, sort_keys=True) + "\n")
            f.flush()
            print("step %d  %.1fs" % (t, time.time() - t0), flush=True)
        if w.apt is not None:
            # adaptive precision: also the precision state after each step, and the
            # epoch's mean Gavg per layer (float64, exact in JSON) when an epoch ends
            def cb_apt(t, rec, st):
                cb(t, rec, extra={**{"apt.bits%d" % l: b for l, b in enumerate(st["bits"])},
                                  **{"apt.exp_w%d" % l: e for l, e in enumerate(st["exp_w"])},
                                  **({"apt.gavg%d" % l: g for l, g in enumerate(st["gavg"])}
                                     if st["gavg"] is not None and t % w.apt.epoch == w.apt.epoch - 1 else {})})
            O.apt_run(w, steps, callback=cb_apt, route=route)
        else:
            O.run_steps(w, steps, callback=cb, route=route)
    os.replace(tmp, path)


if __name__ == "__main__":
    main()
