"""Pins of the oracle's FP32 partial accumulation ("Mixed Precision Training of
Convolutional Neural Networks using Integer Operations", section 4, "Handling
overflows"): hand-worked cases of the INT32 chain overflow that the one-bit
input shift prevents and of the rounding at chain boundaries, and reductions
to the pinned exact DFP contraction and its FP32 conversion."""
import numpy as np
import pytest

import oracle as O


def _hand_case_overflow():
    # one output, 128 terms, chains of 64:
    #   chain 0: x = 32767 at k = 0..3, W = 32767 at k = 0..2 (0 at k = 3)
    #   chain 1: x = 1, 2, 3, 4 and W = 5, 6, 7, 8 at k = 64..67
    x = np.zeros((1, 128), np.int16)
    W = np.zeros((1, 128), np.int16)
    x[0, :4] = 32767
    W[0, :3] = 32767
    x[0, 64:68] = [1, 2, 3, 4]
    W[0, 64:68] = [5, 6, 7, 8]
    return x, W


def test_chain_overflow_hand_case_without_shift_wraps():
    """Without the shift, chain 0 is 3 * 32767^2 = 3221028867 > 2^31 - 1: the
    INT32 accumulator wraps to 3221028867 - 2^32 = -1073938429. To float (24
    bits: a multiple of 2^7 at this size): -1073938429 = -(8390144 * 128 - 3)
    -> -8390144 * 128; times 2^(-20 - 10) = -8390144 * 2^-23. Chain 1 is
    5 + 12 + 21 + 32 = 70 -> 70 * 2^-30, 70/128 = 0.546875 of an ulp (2^-23)
    toward zero: -8390143.453125 * 2^-23 rounds to -8390143 * 2^-23."""
    x, W = _hand_case_overflow()
    y = O.dfp_linear_fwd_f32_chained(x, -20, W, -10, 64, input_shift=False)
    assert y[0, 0] == np.float32(-8390143 / 2.0 ** 23)


def test_chain_overflow_hand_case_with_shift_fits():
    """With the shift, x' = rhu(32767, 1) = 16384 and rhu(1..4, 1) = 1, 1, 2, 2;
    E_inp = -20 + 1. Chain 0 = 3 * 16384 * 32767 = 1610563584 = 98301 * 2^14
    (fits int32, exact in float) -> 98301 * 2^14 * 2^-29 = 98301 * 2^-15.
    Chain 1 = 5 + 6 + 14 + 16 = 41 -> 41 * 2^-29, a third of an ulp (2^-22) of
    the running sum: the sum stays 98301 * 2^-15 = 2.999908447265625."""
    x, W = _hand_case_overflow()
    y = O.dfp_linear_fwd_f32_chained(x, -20, W, -10, 64, input_shift=True)
    assert y[0, 0] == np.float32(98301 / 2.0 ** 15)


def _hand_case_rounding():
    x = np.zeros((1, 192), np.int16)
    W = np.zeros((1, 192), np.int16)
    x[0, 0], W[0, 0] = 8191, 4096        # shifted: 4096 * 4096 = 2^24
    x[0, 64], W[0, 64] = 1, 1            # shifted: rhu(1, 1) = 1 -> 1
    x[0, 128], W[0, 128] = 1, 1
    return x, W


def test_rounding_at_chain_boundaries_hand_case():
    """Chains 2^24, 1, 1 scaled by 2^(0 + 1 + 0): terms 2^25, 2, 2. In chain
    order: 2^25 + 2 is a tie between 2^25 and 2^25 + 4 (ulp 4) -> the even
    significand 2^25; + 2 again -> 2^25. The exact sum 2^25 + 4 is a float,
    and adding in reverse order (2 + 2 + 2^25) gives it: the order and the
    rounding at every chain boundary are what the hand value pins."""
    x, W = _hand_case_rounding()
    y = O.dfp_linear_fwd_f32_chained(x, 0, W, 0, 64, input_shift=True)
    assert y[0, 0] == np.float32(2.0 ** 25)
    assert y[0, 0] != np.float32(2.0 ** 25 + 4)     # the exact (or reverse-order) value


def test_single_chain_reduces_to_the_exact_contraction_rounded_once():
    """One chain over the whole contraction, no overflow: the result is the
    exact sum of the shifted inputs' products rounded to float and scaled
    (the pinned p64_to_float of the pinned exact contraction)."""
    rng = np.random.default_rng(3)
    x = np.clip(np.rint(rng.normal(0, 4096, (5, 64))), -32767, 32767).astype(np.int16)
    W = np.clip(np.rint(rng.normal(0, 4096, (7, 64))), -32767, 32767).astype(np.int16)
    xs = np.vectorize(lambda v: O.rhu(int(v), 1))(x).astype(np.int16)
    P = O.dfp_linear_fwd(xs, W)
    assert np.abs(P).max() < 2 ** 31
    want = O.p64_to_float(P, -12 + 1 - 17)
    got = O.dfp_linear_fwd_f32_chained(x, -12, W, -17, 64, input_shift=True)
    assert np.array_equal(got, want)
    got = O.dfp_linear_fwd_f32_chained(x, -12, W, -17, 1000, input_shift=True)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("chain", [1, 3, 64, 100, 512])
def test_small_values_sum_exactly_for_any_chain(chain):
    """Every chain and running sum below 2^24 is an exact float: the result
    is the exact integer sum whatever the chain length."""
    rng = np.random.default_rng(chain)
    x = rng.integers(-7, 8, (4, 1000)).astype(np.int16)
    W = rng.integers(-7, 8, (3, 1000)).astype(np.int16)
    got = O.dfp_linear_fwd_f32_chained(x, 0, W, 0, chain, input_shift=False)
    assert np.array_equal(got, O.dfp_linear_fwd(x, W).astype(np.float32))
