"""Pins of the oracle's tensor primitives: hand-worked cases of the NITI steps,
brute force on tiny inputs, independent float64 matmul, transposition and
adjoint identities that a swapped index or operand breaks."""
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle as O

rng = np.random.default_rng(12345)


# ------------------------------------------------------------- requantise

def test_requant_shift1_saturates_and_rounds():
    Y = np.array([255, -255, 3, -3, 1, -1, 128, -128], np.int32)
    a, s, m = O.requant(Y, relu=False)
    assert (m, s) == (255, 1)
    assert a.tolist() == [127, -127, 2, -1, 1, 0, 64, -64]
    a, s, _ = O.requant(Y, relu=True)
    assert a.tolist() == [127, 0, 2, 0, 1, 0, 64, 0]


def test_requant_shift2_negative_saturation():
    Y = np.array([-511, 511, -2, 2, -6], np.int32)
    a, s, _ = O.requant(Y, relu=False)
    assert s == 2
    assert a.tolist() == [-128, 127, 0, 1, -1]


def test_requant_zero_tensor_and_int32_min():
    a, s, m = O.requant(np.zeros(7, np.int32), relu=True)
    assert (m, s) == (0, 0) and not a.any()
    Y = np.array([np.iinfo(np.int32).min, 1 << 24, -(1 << 24) - 1], np.int32)
    a, s, m = O.requant(Y, relu=False)
    assert m == 1 << 31 and s == 25
    assert a.tolist() == [-64, 1, -1]


def test_requant_fits_without_shift():
    Y = np.array([127, -128, 0, 5], np.int32)
    a, s, m = O.requant(Y, relu=False)
    # max|Y| = 128 needs 8 bits, so shift 1
    assert (m, s) == (128, 1) and a.tolist() == [64, -64, 0, 3]
    a, s, m = O.requant(np.array([127, -127], np.int32), relu=False)
    assert s == 0 and a.tolist() == [127, -127]


def test_requant_mask_gates_on_positive_activation():
    D = np.array([10, -10, 300, -300], np.int32)      # max 300 -> 9 bits -> shift 2
    a_prev = np.array([1, 0, -3, 127], np.int8)
    out, s, m = O.requant_mask(D, a_prev)
    assert (m, s) == (300, 2)
    assert out.tolist() == [3, 0, 0, -75]
    out, _, _ = O.requant_mask(D, None)
    assert out.tolist() == [3, -2, 75, -75]


# -------------------------------------------------------------- top error

def test_top_error_cases():
    logits = np.array([[127, 5, -128], [-128, 0, 64]], np.int8)
    labels = np.array([0, 0], np.int32)
    e = O.top_error(logits, labels, 64)
    assert e.tolist() == [[63, 5, -128], [-128, 0, 64]]
    e = O.top_error(logits, np.array([2, 2], np.int32), 64)
    assert e.tolist() == [[127, 5, -128], [-128, 0, 0]]


# ----------------------------------------------------------- NITI update

def _g_for(gq_values, s):
    """int32 gradient whose shift is s (a leading element sets max|G|) and
    whose later elements round to the requested Gq values at that shift."""
    lead = (1 << (s + 7)) - 1           # bitlen = s + 7 exactly
    return np.array([lead] + [v << s for v in gq_values], np.int32)


def test_update_weight_shift_7_cases():
    s = 9                                # ws = 7
    G = _g_for([64, 63, -64, -65], s)
    W = np.zeros(G.size, np.int8)
    Wn, shift, ws, m, nz = O.niti_update(W, G)
    assert (shift, ws) == (9, 7)
    # lead: Gq = rhu(65535, 9) = 128 -> sat 127 -> rhu(127, 7) = 1
    assert (-Wn).tolist() == [1, 1, 0, 0, -1]
    assert nz == 3


def test_update_weight_shift_8_vanishes():
    s = 10                               # ws = 8: every int8 Gq rounds to 0
    G = _g_for([127, -127, 100, -1], s)
    Wn, shift, ws, m, nz = O.niti_update(np.full(G.size, 9, np.int8), G)
    assert (shift, ws) == (10, 8) and nz == 0
    assert Wn.tolist() == [9] * G.size


def test_update_saturates_both_ends():
    # shift 0 (max 100 < 128), ws 0: dW = G
    G = np.array([1, -1, 100, -100], np.int32)
    W = np.array([-128, 127, -100, 100], np.int8)
    Wn, shift, ws, m, nz = O.niti_update(W, G)
    assert (shift, ws) == (0, 0)
    assert Wn.tolist() == [-128, 127, -128, 127]


def test_update_max_zero_leaves_weights():
    W = rng.integers(-128, 128, 50).astype(np.int8)
    Wn, shift, ws, m, nz = O.niti_update(W, np.zeros(50, np.int32))
    assert (shift, ws, m, nz) == (0, 0, 0, 0) and (Wn == W).all()


def test_update_double_shift_reading():
    # s = 3 (max 512 -> 10 bits), ws = 1: dW = rhu(rhu(G, 3) sat8, 1)
    G = np.array([512, 12, -12, 20, -20], np.int32)
    Wn, shift, ws, m, nz = O.niti_update(np.zeros(5, np.int8), G)
    assert (shift, ws) == (3, 1)
    # Gq = [64, 2 (1.5 -> 2), -1 (-1.5 -> -1), 3 (2.5 -> 3), -2 (-2.5 -> -2)]
    # dW = rhu(Gq, 1) = [32, 1, 0, 2, -1]
    assert (-Wn).tolist() == [32, 1, 0, 2, -1]


# ------------------------------------------------------- int8 contractions

def brute_fwd(X, W):
    B, IC = X.shape
    OC = W.shape[0]
    return np.array([[sum(int(X[b, i]) * int(W[o, i]) for i in range(IC)) for o in range(OC)]
                     for b in range(B)], np.int64)


def brute_dgrad(E, W):
    B, OC = E.shape
    IC = W.shape[1]
    return np.array([[sum(int(E[b, o]) * int(W[o, i]) for o in range(OC)) for i in range(IC)]
                     for b in range(B)], np.int64)


def brute_wgrad(E, A):
    B, OC = E.shape
    IC = A.shape[1]
    return np.array([[sum(int(E[b, o]) * int(A[b, i]) for b in range(B)) for i in range(IC)]
                     for o in range(OC)], np.int64)


@pytest.mark.parametrize("B,IC,OC", [(1, 1, 1), (2, 3, 4), (4, 4, 2), (3, 1, 5)])
def test_contractions_brute_force_tiny(B, IC, OC):
    for lo, hi in ((-2, 3), (-128, 128)):
        X = rng.integers(lo, hi, (B, IC)).astype(np.int8)
        W = rng.integers(lo, hi, (OC, IC)).astype(np.int8)
        E = rng.integers(lo, hi, (B, OC)).astype(np.int8)
        assert (O.linear_fwd(X, W) == brute_fwd(X, W)).all()
        assert (O.linear_dgrad(E, W) == brute_dgrad(E, W)).all()
        assert (O.linear_wgrad(E, X) == brute_wgrad(E, X)).all()


def test_contractions_vs_float64_matmul_medium():
    B, IC, OC = 67, 300, 45
    X = rng.integers(-128, 128, (B, IC)).astype(np.int8)
    W = rng.integers(-128, 128, (OC, IC)).astype(np.int8)
    E = rng.integers(-128, 128, (B, OC)).astype(np.int8)
    f = lambda a, b: np.rint(a.astype(np.float64) @ b.astype(np.float64)).astype(np.int64)
    assert (O.linear_fwd(X, W) == f(X, W.T)).all()
    assert (O.linear_dgrad(E, W) == f(E, W)).all()
    assert (O.linear_wgrad(E, X) == f(E.T, X)).all()
    # the exact-float64 route of the oracle agrees with its C loops
    assert (O.linear_fwd_f64(X, W) == O.linear_fwd(X, W)).all()
    assert (O.linear_dgrad_f64(E, W) == O.linear_dgrad(E, W)).all()
    assert (O.linear_wgrad_f64(E, X) == O.linear_wgrad(E, X)).all()


def test_contraction_transposition_identities():
    B, IC, OC = 9, 13, 7
    X = rng.integers(-128, 128, (B, IC)).astype(np.int8)
    W = rng.integers(-128, 128, (OC, IC)).astype(np.int8)
    E = rng.integers(-128, 128, (B, OC)).astype(np.int8)
    # dgrad is the forward contraction with the transposed weight
    assert (O.linear_dgrad(E, W) == O.linear_fwd(E, np.ascontiguousarray(W.T))).all()
    # wgrad is the forward contraction of E^T against X^T
    assert (O.linear_wgrad(E, X) == O.linear_fwd(np.ascontiguousarray(E.T),
                                                  np.ascontiguousarray(X.T))).all()


def test_contraction_extreme_values_exact():
    K = 8192
    X = np.full((2, K), -128, np.int8)
    W = np.full((3, K), -128, np.int8)
    assert (O.linear_fwd(X, W) == K * 16384).all()
    X[1, ::2] = 127
    y = O.linear_fwd(X, W)
    assert y[1, 0] == (K // 2) * (127 * -128) + (K // 2) * 16384


def test_int32_overflow_aborts():
    code = textwrap.dedent("""
        import numpy as np, oracle as O
        K = 140000
        O.linear_fwd(np.full((1, K), -128, np.int8), np.full((1, K), -128, np.int8))
    """)
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       cwd=O._HERE + "/..")
    assert p.returncode != 0 and "int32 overflow" in p.stderr


# --------------------------------------------------------------- conv NHWC

def im2col_conv(X, Wt, stride, pad=1):
    B, H, Wd, IC = X.shape
    OC, KH, KW, _ = Wt.shape
    Xp = np.zeros((B, H + 2 * pad, Wd + 2 * pad, IC), np.int64)
    Xp[:, pad:pad + H, pad:pad + Wd, :] = X
    OH, OW = O.conv_out(H, KH, stride, pad), O.conv_out(Wd, KW, stride, pad)
    cols = np.empty((B, OH, OW, KH, KW, IC), np.int64)
    for kh in range(KH):
        for kw in range(KW):
            cols[:, :, :, kh, kw, :] = Xp[:, kh:kh + stride * OH:stride, kw:kw + stride * OW:stride, :]
    return np.einsum("bhwk,ok->bhwo", cols.reshape(B, OH, OW, -1), Wt.reshape(OC, -1).astype(np.int64))


@pytest.mark.parametrize("stride,H,Wd", [(1, 5, 6), (2, 7, 8), (2, 8, 8), (1, 1, 1), (2, 3, 2)])
def test_conv_fwd_vs_im2col(stride, H, Wd):
    X = rng.integers(-128, 128, (2, H, Wd, 3)).astype(np.int8)
    Wt = rng.integers(-128, 128, (4, 3, 3, 3)).astype(np.int8)
    assert (O.conv2d_fwd(X, Wt, stride) == im2col_conv(X, Wt, stride)).all()


def test_conv_delta_kernel_reproduces_input():
    X = rng.integers(-128, 128, (2, 6, 5, 3)).astype(np.int8)
    Wt = np.zeros((3, 3, 3, 3), np.int8)
    for c in range(3):
        Wt[c, 1, 1, c] = 1 if c != 1 else -1
    Y = O.conv2d_fwd(X, Wt, 1)
    assert (Y[..., 0] == X[..., 0]).all() and (Y[..., 1] == -X[..., 1].astype(np.int32)).all()
    assert (Y[..., 2] == X[..., 2]).all()


@pytest.mark.parametrize("stride,H,Wd", [(1, 5, 6), (2, 7, 8), (2, 8, 8), (2, 3, 2)])
def test_conv_adjoint_identities(stride, H, Wd):
    """<conv(x, W), e> = <x, dgrad(e, W)> = <W, wgrad(e, x)> for every x, W, e."""
    B, IC, OC = 2, 3, 4
    X = rng.integers(-128, 128, (B, H, Wd, IC)).astype(np.int8)
    Wt = rng.integers(-128, 128, (OC, 3, 3, IC)).astype(np.int8)
    OH, OW = O.conv_out(H, 3, stride), O.conv_out(Wd, 3, stride)
    E = rng.integers(-128, 128, (B, OH, OW, OC)).astype(np.int8)
    lhs = int((O.conv2d_fwd(X, Wt, stride).astype(np.int64) * E).sum())
    D = O.conv2d_dgrad(E, Wt, (H, Wd), stride)
    G = O.conv2d_wgrad(E, X, 3, stride)
    assert lhs == int((D.astype(np.int64) * X).sum())
    assert lhs == int((G.astype(np.int64) * Wt).sum())


def test_conv_dgrad_scatter_vs_gather():
    # gather form: D[b,ih,iw,ic] = sum over (kh,kw,oc) with oh*s-1+kh = ih, ...
    B, H, Wd, IC, OC, s = 1, 5, 4, 2, 3, 2
    Wt = rng.integers(-128, 128, (OC, 3, 3, IC)).astype(np.int8)
    OH, OW = O.conv_out(H, 3, s), O.conv_out(Wd, 3, s)
    E = rng.integers(-128, 128, (B, OH, OW, OC)).astype(np.int8)
    D = O.conv2d_dgrad(E, Wt, (H, Wd), s)
    for ih in range(H):
        for iw in range(Wd):
            for ic in range(IC):
                acc = 0
                for kh in range(3):
                    for kw in range(3):
                        if (ih + 1 - kh) % s or (iw + 1 - kw) % s:
                            continue
                        oh, ow = (ih + 1 - kh) // s, (iw + 1 - kw) // s
                        if 0 <= oh < OH and 0 <= ow < OW:
                            acc += int(E[0, oh, ow, :].astype(np.int64) @ Wt[:, kh, kw, ic].astype(np.int64))
                assert D[0, ih, iw, ic] == acc


def test_gap_fwd_bwd():
    A = rng.integers(-128, 128, (3, 4, 2, 5)).astype(np.int8)
    P = O.gap_fwd(A)
    assert (P == A.astype(np.int64).sum(axis=(1, 2))).all()
    dP = np.array([[1, -2, 3, -4, 5]] * 3, np.int8)
    A2 = np.zeros((3, 4, 2, 5), np.int8)
    A2[0, 1, 1, 2] = 7
    A2[2, 3, 0, 4] = 1
    A2[1, 0, 0, 0] = -5
    D = O.gap_bwd(dP, A2)
    assert D[0, 1, 1, 2] == 3 and D[2, 3, 0, 4] == 5 and np.count_nonzero(D) == 2


# --------------------------------------------------------------------- DFP16

@pytest.mark.parametrize("vals,rs,want", [
    ([32767], 0, [32767]), ([32768], 1, [16384]), ([65535], 1, [32767]),
    ([-65535], 1, [-32767]), ([-32767, 3], 0, [-32767, 3]), ([0, 0], 0, [0, 0]),
    ([1 << 40, -3 << 30], 26, [16384, -48]),
])
def test_dfp_down_cases(vals, rs, want):
    out, e, r, m = O.dfp_down(np.array(vals, np.int64), exp_in=-20)
    assert r == rs and out.tolist() == want and e == -20 + rs


def test_dfp_down_value_within_half_ulp():
    P = rng.integers(-(1 << 40), 1 << 40, 1000)
    out, e, rs, m = O.dfp_down(P, exp_in=-30)
    # i * 2^(E_in + Rs) approximates P * 2^E_in within half a step, unless saturated
    err = np.abs(out.astype(np.int64) * (1 << rs) - P)
    unsat = np.abs(out) < 32767
    assert (err[unsat] <= (1 << rs) // 2).all()


def test_dfp_exponent_range_error():
    with pytest.raises(OverflowError):
        O.dfp_down(np.array([1 << 40], np.int64), exp_in=120)


def test_dfp_contractions_vs_brute_and_float64():
    B, IC, OC = 3, 5, 4
    X = rng.integers(-32767, 32768, (B, IC)).astype(np.int16)
    W = rng.integers(-32767, 32768, (OC, IC)).astype(np.int16)
    E = rng.integers(-32767, 32768, (B, OC)).astype(np.int16)
    assert (O.dfp_linear_fwd(X, W) == brute_fwd(X, W)).all()
    assert (O.dfp_linear_dgrad(E, W) == brute_dgrad(E, W)).all()
    assert (O.dfp_linear_wgrad(E, X) == brute_wgrad(E, X)).all()
    B, IC, OC = 40, 2048, 33
    X = np.full((B, IC), -32767, np.int16)
    X[1:] = rng.integers(-32767, 32768, (B - 1, IC))
    W = rng.integers(-32767, 32768, (OC, IC)).astype(np.int16)
    W[0] = -32767
    E = rng.integers(-32767, 32768, (B, OC)).astype(np.int16)
    assert (O.dfp_linear_fwd(X, W) == O.dfp_linear_fwd_f64(X, W)).all()
    assert O.dfp_linear_fwd(X, W)[0, 0] == IC * 32767 * 32767
    assert (O.dfp_linear_dgrad(E, W) == O.dfp_linear_dgrad_f64(E, W)).all()
    assert (O.dfp_linear_wgrad(E, X) == O.dfp_linear_wgrad_f64(E, X)).all()


def test_dfp_update_cases():
    W = np.array([0, 100, -32767, 32767, 5], np.int16)
    G = np.array([256, -384, 1, -1, 0], np.int16)
    Wn, nz = O.dfp_update(W, G, 8)          # dW = rhu(G, 8) = [1, -1 (-1.5 -> -1), 0, 0, 0]
    assert Wn.tolist() == [-1, 101, -32767, 32767, 5] and nz == 2
    Wn, nz = O.dfp_update(W, G, -3)         # dW = G * 8
    assert Wn.tolist() == [-2048, 3172, -32767, 32767, 5]
    Wn, _ = O.dfp_update(W, G, -40)         # any left shift past 17 bits saturates the same way
    assert Wn.tolist() == [-32767, 32767, -32767, 32767, 5]


# ------------------------------------------------- partial-model (UINT8 input)

@pytest.mark.parametrize("B,IC,OC", [(1, 1, 1), (2, 5, 3), (4, 3, 4)])
def test_u8_contractions_brute_force(B, IC, OC):
    X = rng.integers(0, 256, (B, IC)).astype(np.uint8)
    X[0, 0] = 255
    W = rng.integers(-128, 128, (OC, IC)).astype(np.int8)
    E = rng.integers(-128, 128, (B, OC)).astype(np.int8)
    assert (O.linear_fwd_u8(X, W) == brute_fwd(X, W)).all()
    assert (O.linear_wgrad_u8(E, X) == brute_wgrad(E, X)).all()
    # a uint8 value is not its int8 bit pattern: 255 must not read as -1
    assert O.linear_fwd_u8(np.array([[255]], np.uint8), np.array([[2]], np.int8))[0, 0] == 510


def test_u8_contractions_vs_float64_medium():
    X = rng.integers(0, 256, (70, 513)).astype(np.uint8)
    W = rng.integers(-128, 128, (33, 513)).astype(np.int8)
    E = rng.integers(-128, 128, (70, 33)).astype(np.int8)
    assert (O.linear_fwd_u8(X, W) == O.linear_fwd_f64(X, W)).all()
    assert (O.linear_wgrad_u8(E, X) == O.linear_wgrad_f64(E, X)).all()


def test_pack_relu_mask_hand_case():
    A = np.array([[1, 0, -1, 5, 0, 0, 0, 127, 3, -128],
                  [0, 0, 0, 0, 0, 0, 0, 0, 0, 1]], np.int8)
    m = O.pack_relu_mask(A)
    assert m.shape == (2, 2)
    assert m[0].tolist() == [0b10001001, 0b00000001]
    assert m[1].tolist() == [0, 0b00000010]


# ------------------------------------- static requantisation with INT32 offsets

def test_requant_static_hand_cases():
    Y = np.array([[100, -100, 5, -7, 1000]], np.int32)
    off = np.array([10, 0, -5, 0, 0], np.int32)
    mult = np.array([3, 2, 1, 1, 1], np.int32)
    k = np.array([2, 1, 0, 1, 0], np.int32)
    # (110*3)/4 = 82.5 -> 82; (-200)/2 = -100; 0; -7/2 = -3.5 -> floor -4; 1000 -> clip 127
    assert O.requant_static(Y, off, mult, k, relu=False).tolist() == [[82, -100, 0, -4, 127]]
    assert O.requant_static(Y, off, mult, k, relu=True).tolist() == [[82, 0, 0, 0, 127]]
    big = np.array([[-(1 << 30)]], np.int32)
    assert O.requant_static(big, np.array([0], np.int32), np.array([1 << 14], np.int32),
                            np.array([30], np.int32), relu=False).tolist() == [[-128]]   # -2^44 >> 30 = -2^14, clip


def test_requant_static_identity_case_is_plain_clip():
    Y = rng.integers(-400, 400, (7, 9)).astype(np.int32)
    z = np.zeros(9, np.int32)
    one = np.ones(9, np.int32)
    assert (O.requant_static(Y, z, one, z, relu=False) == np.clip(Y, -128, 127)).all()
    assert (O.requant_static(Y, z, one, z, relu=True) == np.clip(Y, 0, 127)).all()


def test_offset_grad_and_update():
    d = np.array([[1, -128, 5], [2, -128, -5], [3, -128, 0]], np.int8)
    g = O.offset_grad(d)
    assert g.tolist() == [6, -384, 0]
    # max 384 -> 9 bits -> shift 2, weight shift 0: Gq = [2 (1.5 -> 2), -96, 0]
    on, s, ws, m, nz = O.offset_update(np.array([0, np.iinfo(np.int32).max, 7], np.int32), g)
    assert (s, ws, m, nz) == (2, 0, 384, 2)
    assert on.tolist() == [-2, np.iinfo(np.int32).max, 7]       # +96 saturates at INT32_MAX
    on, *_ = O.offset_update(np.array([np.iinfo(np.int32).min + 1], np.int32), np.array([100], np.int32))
    assert on.tolist() == [np.iinfo(np.int32).min]


# ------------------------------------------------------- float <-> DFP16

def test_dfp_from_float_hand_cases():
    m, e = O.dfp_from_float(np.array([1.0, -0.5, 0.75, 3.0], np.float32))
    assert e == -13 and m.tolist() == [8192, -4096, 6144, 24576]        # 3.0 = 0.75 * 2^2
    assert O.dfp_to_float(m, e).tolist() == [1.0, -0.5, 0.75, 3.0]
    # max 32768 = 0.5 * 2^16: E = 1; x / 2 rounds to nearest, ties to even
    m, e = O.dfp_from_float(np.array([32768.0, 3.0, 5.0, 7.0, -5.0, -7.0], np.float32))
    assert e == 1 and m.tolist() == [16384, 2, 2, 4, -2, -4]
    # just below 2^15 with E = 0: 32767.75 rounds to 32768 and saturates
    m, e = O.dfp_from_float(np.array([32767.75, -1.25], np.float32))
    assert e == 0 and m.tolist() == [32767, -1]
    m, e = O.dfp_from_float(np.zeros(5, np.float32))
    assert e == 0 and not m.any()


def test_dfp_from_float_error_bound():
    f = (rng.standard_normal(5000) * 1e-3).astype(np.float32)
    m, e = O.dfp_from_float(f)
    back = m.astype(np.float64) * 2.0 ** e
    assert np.abs(back - f.astype(np.float64)).max() <= 2.0 ** (e - 1)
    assert np.abs(m).max() >= 16384                  # the exponent uses the full 15 bits


def test_p64_to_float_rounds_once_then_scales():
    P = np.array([(1 << 24) + 1, (1 << 24) + 3, -(1 << 40) - 1, 7], np.int64)
    out = O.p64_to_float(P, -3)
    # 2^24 + 1 is a tie between 2^24 and 2^24 + 2: to even (2^24); 2^24 + 3 -> 2^24 + 4
    assert out.tolist() == [2.0 ** 21, (2.0 ** 24 + 4) / 8, -(2.0 ** 37), 7 / 8]
