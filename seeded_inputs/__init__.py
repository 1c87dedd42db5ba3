"""Seeded synthetic inputs for the integer training workloads.

This module is shared by the CPU oracle tests, the GPU tests and the benchmark.
It holds random draws and workload shapes only: none of the training method's
arithmetic (no contraction, shift, rounding or saturation rule) lives here.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the finaliser constants are Vigna's), used in
counter form: output ``i`` of stream ``s`` under seed ``S`` is
``mix64(S + GAMMA * (s * 2**40 + i + 1))``. Every value depends only on
(seed, stream, index), so any slice can be regenerated independently and the
result is identical on every platform.

Draws:

* uniform integers in ``[lo, hi]``: Lemire's multiply-shift method on the top
  32 bits of a draw, with the unbiased rejection step ("Fast random integer
  generation in an interval", ACM TOMACS 2019). A rejected element ``i`` tries
  counters ``i + n, i + 2n, ...`` of the same stream.
* normals: Box-Muller (cosine branch) on two 53-bit uniforms taken from
  counters ``2i`` and ``2i + 1``; ``round_clamp_normal`` scales by sigma, rounds
  half away from zero and clamps to ``[-lim, lim]``.

Stream layout per workload: the weights of layer ``l`` use stream ``8 + l``
(drawn once, before step 0); step ``t`` draws its input batch from stream
``64 * (t + 1)`` and its labels from stream ``64 * (t + 1) + 1``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_SPAN = 1 << 40


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def u64(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    """Outputs ``start .. start+n-1`` of one SplitMix64 stream, as uint64."""
    if n < 0 or start < 0 or start + n > _STREAM_SPAN:
        raise ValueError("counter range outside the stream")
    base = (seed + int(GAMMA) * (stream * _STREAM_SPAN + start + 1)) & 0xFFFFFFFFFFFFFFFF
    idx = np.arange(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(base) + idx * GAMMA
        return _mix64(z)


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """``n`` integers uniform in ``[lo, hi]`` (int64)."""
    r = hi - lo + 1
    if r <= 0 or r > (1 << 32):
        raise ValueError("range must hold 1 .. 2**32 values")
    thresh = ((1 << 32) - r) % r
    out = np.empty(n, dtype=np.int64)
    todo = np.arange(n, dtype=np.int64)
    attempt = 0
    while todo.size:
        # counter for element i on attempt j is i + j*n; draw the whole block once per attempt
        block = u64(seed, stream, attempt * n, n)[todo]
        x = block >> np.uint64(32)
        m = x * np.uint64(r)
        low = m & np.uint64(0xFFFFFFFF)
        ok = low >= np.uint64(thresh)
        out[todo[ok]] = (m[ok] >> np.uint64(32)).astype(np.int64) + lo
        todo = todo[~ok]
        attempt += 1
    return out


def std_normal(seed: int, stream: int, n: int) -> np.ndarray:
    """``n`` standard normals (float64) by Box-Muller, cosine branch."""
    z = u64(seed, stream, 0, 2 * n)
    scale = 1.0 / float(1 << 53)
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * scale  # (0, 1]
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * scale          # [0, 1)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def round_clamp_normal(seed: int, stream: int, n: int, sigma: float, lim: int) -> np.ndarray:
    """round(N(0, sigma)) with ties away from zero, clamped to [-lim, lim] (int64)."""
    v = std_normal(seed, stream, n) * sigma
    r = np.sign(v) * np.floor(np.abs(v) + 0.5)
    return np.clip(r, -lim, lim).astype(np.int64)


# --------------------------------------------------------------------------
# Workloads. Shapes and distributions of the five training workloads.
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class AptSetting:
    """Adaptive precision training (Algorithms 1-2 of "Adaptive Precision
    Training for Resource Constrained Devices"): initial weight precision,
    precision limits, Gavg thresholds, epoch length in steps and the step
    interval of Gavg evaluations within an epoch."""
    k_init: int = 6
    k_min: int = 2
    k_max: int = 16
    t_min: float = 1.0
    t_max: float = float("inf")
    epoch: int = 10
    eval_every: int = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    name: str
    kind: str                 # "mlp", "cnn" or "dfp16"
    batch: int
    dims: tuple = ()          # mlp / dfp16: feature sizes, input first
    classes: int = 0
    image: tuple = ()         # cnn: (H, W, C)
    convs: tuple = ()         # cnn: (IC, OC, stride) per 3x3 conv, pad 1
    fc: tuple = ()            # cnn: (IC, OC) of the final Linear
    sigma: float = 32.0       # weight normal sigma
    lim: int = 127            # clamp for weights and inputs
    in_lim: int = 127         # mlp/cnn: int8 inputs uniform in [-in_lim, in_lim]
    exp_x: int = 0            # dfp16 shared exponents of input and weights
    exp_w: int = 0
    eta: int = 20             # dfp16 integer SGD learning rate 2^-eta (on the batch-summed gradient)
    input_uint8: bool = False # mlp: UINT8 input in [0, 255] (partial-model training)
    trainable_from: int = 0   # mlp: layers before this one are frozen
    static_requant: tuple = ()  # mlp: per layer (k_lo, k_hi) of a static requantisation, () = dynamic
    apt: AptSetting = None    # dfp16: adaptive per-layer weight precision

    @property
    def seed(self) -> int:
        return 0x1A7E0000 + self.index


WORKLOADS = (
    Workload(0, "mlp64-64-10_b32", "mlp", 32, dims=(64, 64, 10), classes=10),
    Workload(1, "mlp784-1024x3-10_b256", "mlp", 256, dims=(784, 1024, 1024, 1024, 10), classes=10),
    Workload(2, "cnn3-64-128-256_gap_fc10_b128", "cnn", 128, classes=10, image=(32, 32, 3),
             convs=((3, 64, 1), (64, 128, 2), (128, 256, 2)), fc=(256, 10)),
    Workload(3, "mlp4096x4-1000_b8192", "mlp", 8192, dims=(4096, 4096, 4096, 4096, 4096, 1000),
             classes=1000),
    Workload(4, "dfp16_2048x3_b2048", "dfp16", 2048, dims=(2048, 2048, 2048, 2048),
             sigma=4096.0, lim=32767, exp_x=-12, exp_w=-17),
    # partial-model training: UINT8 input, the last two of four layers trainable
    Workload(5, "mlp784-1024x3-10_b256_u8_last2", "mlp", 256, dims=(784, 1024, 1024, 1024, 10),
             classes=10, input_uint8=True, trainable_from=2),
    # the TI library's forward: static per-channel requantisation with trained INT32 offsets
    Workload(6, "mlp784-1024x3-10_b256_static", "mlp", 256, dims=(784, 1024, 1024, 1024, 10), classes=10,
             static_requant=((24, 25), (24, 25), (24, 25), (22, 23))),
    # adaptive precision training on the DFP16 stack: weights start at 6 bits
    Workload(7, "dfp16_2048x3_b2048_apt6", "dfp16", 2048, dims=(2048, 2048, 2048, 2048),
             sigma=4096.0, lim=32767, exp_x=-12, exp_w=-17,
             apt=AptSetting(k_init=6, k_min=2, k_max=16, t_min=100.0, t_max=float("inf"), epoch=10, eval_every=1)),
    # the 4096-wide MLP at batch 1024 with inputs in [-7, 7]: the first layer's weight
    # gradient is small enough for its weights to move (the wider-input workloads' do not)
    Workload(8, "mlp4096x4-1000_b1024_x7", "mlp", 1024, dims=(4096, 4096, 4096, 4096, 4096, 1000),
             classes=1000, in_lim=7),
)


def weight_stream(layer: int) -> int:
    return 8 + layer


def batch_stream(step: int, which: int) -> int:
    return 64 * (step + 1) + which


def weight_shapes(w: Workload) -> list:
    """Weight tensor shapes, row-major: Linear [OC, IC]; conv [OC, 3, 3, IC]."""
    if w.kind in ("mlp", "dfp16"):
        return [(w.dims[i + 1], w.dims[i]) for i in range(len(w.dims) - 1)]
    shapes = [(oc, 3, 3, ic) for (ic, oc, _s) in w.convs]
    shapes.append((w.fc[1], w.fc[0]))
    return shapes


def make_weights(w: Workload) -> list:
    """Initial weights: int8 for mlp/cnn, int16 mantissas for dfp16."""
    dt = np.int16 if w.kind == "dfp16" else np.int8
    out = []
    for l, shp in enumerate(weight_shapes(w)):
        n = int(np.prod(shp))
        v = round_clamp_normal(w.seed, weight_stream(l), n, w.sigma, w.lim)
        out.append(v.astype(dt).reshape(shp))
    return out


def make_static_requant(w: Workload):
    """Per layer None, or dict(offset int32 [OC] = round(N(0, 2^14)), mult
    int32 [OC] uniform in [2^14, 2^15), k int32 [OC] uniform in [k_lo, k_hi])
    for a workload with a static requantisation (streams 40 + 3l .. 42 + 3l)."""
    if not w.static_requant:
        return None
    out = []
    for l, (klo, khi) in enumerate(w.static_requant):
        oc = w.dims[l + 1]
        off = round_clamp_normal(w.seed, 40 + 3 * l, oc, 16384.0, 1 << 30).astype(np.int32)
        mult = uniform_int(w.seed, 41 + 3 * l, oc, 1 << 14, (1 << 15) - 1).astype(np.int32)
        k = uniform_int(w.seed, 42 + 3 * l, oc, klo, khi).astype(np.int32)
        out.append(dict(offset=off, mult=mult, k=k))
    return out


def input_shape(w: Workload) -> tuple:
    if w.kind == "cnn":
        return (w.batch,) + tuple(w.image)
    return (w.batch, w.dims[0])


def make_batch(w: Workload, step: int):
    """(x, labels) for one step. mlp/cnn: int8 x uniform in [-in_lim, in_lim]
    (uint8 in [0, 255] for a UINT8-input workload), int32 labels uniform in
    [0, classes). dfp16: int16 x = round(N(0, sigma)) clamped, labels None."""
    shp = input_shape(w)
    n = int(np.prod(shp))
    if w.kind == "dfp16":
        x = round_clamp_normal(w.seed, batch_stream(step, 0), n, w.sigma, w.lim)
        return x.astype(np.int16).reshape(shp), None
    if w.input_uint8:
        x = uniform_int(w.seed, batch_stream(step, 0), n, 0, 255).astype(np.uint8).reshape(shp)
    else:
        x = uniform_int(w.seed, batch_stream(step, 0), n, -w.in_lim, w.in_lim).astype(np.int8).reshape(shp)
    labels = uniform_int(w.seed, batch_stream(step, 1), w.batch, 0, w.classes - 1).astype(np.int32)
    return x, labels


def by_name(name_or_index) -> Workload:
    for w in WORKLOADS:
        if name_or_index in (w.index, w.name, str(w.index)):
            return w
    raise KeyError(name_or_index)
