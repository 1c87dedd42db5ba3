"""The seeded input generator: SplitMix64's published outputs, determinism,
ranges and distribution shape of the workloads' draws."""
import numpy as np

import seeded_inputs as si


def test_splitmix64_reference_outputs():
    # SplitMix64 from state 1234567: the first five outputs of the published
    # reference generator (Vigna's splitmix64.c, as used to seed xoshiro).
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert si.u64(1234567, 0, 0, 5).tolist() == want


def test_counter_slices_are_consistent():
    a = si.u64(7, 3, 0, 100)
    b = si.u64(7, 3, 40, 20)
    assert (a[40:60] == b).all()
    assert not (si.u64(7, 4, 0, 100) == a).any()


def test_uniform_int_range_and_balance():
    v = si.uniform_int(5, 1, 200000, -127, 127)
    assert v.min() == -127 and v.max() == 127
    counts = np.bincount(v + 127)
    assert counts.min() > 0.8 * counts.mean() and counts.max() < 1.2 * counts.mean()
    assert (si.uniform_int(5, 1, 1000, -127, 127) == v[:1000]).all()


def test_normal_moments_and_clamp():
    v = si.round_clamp_normal(9, 2, 400000, 32.0, 127)
    assert abs(v.mean()) < 0.3 and abs(v.std() - 32.0) < 0.3
    assert v.min() >= -127 and v.max() <= 127
    w = si.round_clamp_normal(9, 2, 10000, 4096.0, 32767)
    assert w.max() <= 32767 and w.min() >= -32767


def test_workload_shapes():
    w = si.by_name(3)
    shapes = si.weight_shapes(w)
    assert shapes == [(4096, 4096)] * 4 + [(1000, 4096)]
    x, labels = si.make_batch(si.by_name(0), 0)
    assert x.shape == (32, 64) and x.dtype == np.int8 and labels.dtype == np.int32
    assert labels.min() >= 0 and labels.max() <= 9
    x, labels = si.make_batch(si.by_name(2), 1)
    assert x.shape == (128, 32, 32, 3)
    ws = si.make_weights(si.by_name(2))
    assert [a.shape for a in ws] == [(64, 3, 3, 3), (128, 3, 3, 64), (256, 3, 3, 128), (10, 256)]
    x, labels = si.make_batch(si.by_name(4), 0)
    assert x.dtype == np.int16 and labels is None


def test_narrow_input_workload():
    w = si.by_name(8)
    x, labels = si.make_batch(w, 0)
    assert x.shape == (1024, 4096) and x.min() == -7 and x.max() == 7
    assert labels.max() <= 999
    assert si.weight_shapes(w) == si.weight_shapes(si.by_name(3))
