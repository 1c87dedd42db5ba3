"""Pins of the oracle's Blocked-DFP pieces ("Mixed Precision Training of
Convolutional Neural Networks using Integer Operations", section 3: several
fine-grained exponents per tensor; section 4: FP32 outputs): each block is a
DFP-16 tensor of its own; one block per row reduces to the per-tensor
conversion; the blocked linear forward equals the exact rational result
rounded once when no double rounding can occur, and the unblocked DFP FP32
path when all exponents agree."""
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

rng = np.random.default_rng(9090)


def test_blocks_are_independent_dfp_tensors():
    scales = np.repeat([1e-3, 1e3, 1.0, 7.5e-6], 64)[:200]
    f = (rng.standard_normal((3, 200)) * scales).astype(np.float32)
    m, ex = O.bdfp_from_float(f, 64)
    assert ex.shape == (3, 4)
    for r in range(3):
        for j in range(4):
            mm, e = O.dfp_from_float(f[r:r + 1, j * 64:(j + 1) * 64])
            assert e == ex[r, j] and np.array_equal(mm.ravel(), m[r, j * 64:(j + 1) * 64])
    # one block per row is the per-tensor conversion row by row
    m1, e1 = O.bdfp_from_float(f, 200)
    for r in range(3):
        mm, e = O.dfp_from_float(f[r:r + 1])
        assert e == e1[r, 0] and np.array_equal(mm.ravel(), m1[r])


def test_blocked_range_beats_one_exponent():
    """The point of several exponents: a block of tiny values next to a block
    of huge ones keeps its precision (a single exponent flushes it to 0)."""
    f = np.concatenate([np.full(64, 3e-4, np.float32), np.full(64, 5e3, np.float32)])[None, :]
    m, ex = O.bdfp_from_float(f, 64)
    back = O.bdfp_to_float(m, ex, 64)
    assert np.allclose(back, f, rtol=2 ** -14)
    ms, e = O.dfp_from_float(f)
    assert (ms[0, :64] == 0).all()


def _exact_linear(x, ex, W, ew, block):
    B, IC = x.shape
    OC = W.shape[0]
    nb = (IC + block - 1) // block
    y = np.empty((B, OC), np.float32)
    for b in range(B):
        for o in range(OC):
            s = Fraction(0)
            for j in range(nb):
                p = sum(int(x[b, k]) * int(W[o, k]) for k in range(j * block, min(IC, (j + 1) * block)))
                s += Fraction(p) * Fraction(2) ** int(ex[b, j] + ew[o, j])
            y[b, o] = np.float32(float(s))
    return y


@pytest.mark.parametrize("IC,block", [(64, 64), (200, 64), (128, 128)])
def test_blocked_linear_exact_when_no_double_rounding(IC, block):
    """Small mantissas and exponents within a few bits: every double sum is
    exact, so the result is the exact rational value rounded once to float."""
    B, OC = 3, 5
    nb = (IC + block - 1) // block
    x = rng.integers(-300, 301, (B, IC)).astype(np.int16)
    W = rng.integers(-300, 301, (OC, IC)).astype(np.int16)
    ex = rng.integers(-20, -10, (B, nb)).astype(np.int32)
    ew = rng.integers(-20, -10, (OC, nb)).astype(np.int32)
    y = O.bdfp_linear_fwd_f32(x, ex, W, ew, block)
    assert np.array_equal(y, _exact_linear(x, ex, W, ew, block))


def test_blocked_linear_with_equal_exponents_is_the_dfp_path():
    x = rng.integers(-32767, 32768, (4, 1000)).astype(np.int16)
    W = rng.integers(-32767, 32768, (6, 1000)).astype(np.int16)
    ex = np.full((4, 8), -9, np.int32)
    ew = np.full((6, 8), -21, np.int32)
    y = O.bdfp_linear_fwd_f32(x, ex, W, ew, 128)
    P = O.dfp_linear_fwd(x, W)
    # the block sums add exactly in double (|P| < 2^53), so one rounding: float(P * 2^-30)
    assert np.array_equal(y, O.p64_to_float(P, -30))


def test_planted_block_misalignment_is_caught():
    """Pairing x's block j with W's block j + 1 (a plausible indexing slip)
    changes the result."""
    x = rng.integers(-100, 101, (2, 128)).astype(np.int16)
    W = rng.integers(-100, 101, (3, 128)).astype(np.int16)
    ex = np.array([[-4, -12], [-6, -2]], np.int32)
    ew = np.array([[-3, -9], [0, -5], [-7, -1]], np.int32)
    good = O.bdfp_linear_fwd_f32(x, ex, W, ew, 64)
    bad = O.bdfp_linear_fwd_f32(x, ex, W, ew[:, ::-1].copy(), 64)
    assert not np.array_equal(good, bad)
    assert np.array_equal(good, _exact_linear(x, ex, W, ew, 64))
