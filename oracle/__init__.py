"""CPU oracle for integer-only training: plain C primitives (oracle.c) plus the
order of one training step, written out here.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package's smoke check
and by the benchmark's CPU-baseline leg, never by the product path. It shares no
code with the CUDA library and never imports it.

Sources:
  "Integer On-Device Training: Overview" (TI C2000 MCU AI user guide):
    section 3, NITI dynamic shifts, Steps 1-5 and the delta-propagation note;
    section 4, the training loop (forward, compute_loss writes dy, backward
    reads it and updates weights).
  "Mixed Precision Training of Convolutional Neural Networks using Integer
    Operations": section 3 and 3.1, DFP tensors and primitives.
  "Adaptive Precision Training for Resource Constrained Devices": section III,
    the Gavg metric (Equation 4), Algorithm 1 (precision adjustment) and
    Algorithm 2 (adjustment between epochs), applied to DFP weights.

Step order (one reading, stated): forward through all layers; top error;
then for each layer from the top down: delta propagation with the weights as
they were before this step's update (not for the first layer), weight
gradient, weight update.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

TARGET_BITS = 7      # NITI target_bits, for forward, delta and weight gradient
MU_WEIGHT = 2        # NITI mu_weight
TARGET_MAG = 64      # integer target on the true class
DFP_BITS = 15        # DFP-16 mantissa: 15 magnitude bits plus sign
DFP_ETA = 20         # DFP16 integer SGD: learning rate 2^-eta on the batch-summed gradient


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, OpenMP over output rows)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-Wall", "-Wextra", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def set_threads(n: int) -> None:
    """Threads of the C loops' OpenMP regions (timing only; results are the same)."""
    lib().ora_set_threads(int(n))


def max_threads() -> int:
    return lib().ora_max_threads()


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, u32, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
        sig = {
            "ora_set_threads": (None, [ctypes.c_int]),
            "ora_max_threads": (ctypes.c_int, []),
            "ora_bitlen": (i32, [u64]),
            "ora_shift_from_max": (i32, [u64, i32]),
            "ora_rhu": (i64, [i64, i32]),
            "ora_sat8": (i64, [i64]),
            "ora_sat16": (i64, [i64]),
            "ora_absmax32": (u32, [P, i64]),
            "ora_absmax64": (u64, [P, i64]),
            "ora_requant": (i32, [P, i64, i32, ctypes.c_int, P, P]),
            "ora_requant_mask": (i32, [P, P, i64, i32, P, P]),
            "ora_top_error": (None, [P, P, ctypes.c_int, ctypes.c_int, i32, P]),
            "ora_niti_update": (i64, [P, P, i64, i32, i32, P, P, P]),
            "ora_linear_fwd": (None, [P, P] + [ctypes.c_int] * 3 + [P]),
            "ora_linear_dgrad": (None, [P, P] + [ctypes.c_int] * 3 + [P]),
            "ora_linear_wgrad": (None, [P, P] + [ctypes.c_int] * 3 + [P]),
            "ora_linear_fwd_u8": (None, [P, P] + [ctypes.c_int] * 3 + [P]),
            "ora_linear_wgrad_u8": (None, [P, P] + [ctypes.c_int] * 3 + [P]),
            "ora_pack_relu_mask": (None, [P, ctypes.c_int, ctypes.c_int, P]),
            "ora_requant_static": (None, [P, ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_int, P]),
            "ora_offset_grad": (None, [P, ctypes.c_int, ctypes.c_int, P]),
            "ora_offset_update": (i64, [P, P, ctypes.c_int, i32, i32, P, P, P]),
            "ora_conv2d_fwd": (None, [P, P] + [ctypes.c_int] * 9 + [P]),
            "ora_conv2d_dgrad": (None, [P, P] + [ctypes.c_int] * 9 + [P]),
            "ora_conv2d_wgrad": (None, [P, P] + [ctypes.c_int] * 9 + [P]),
            "ora_gap_fwd": (None, [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]),
            "ora_gap_bwd": (None, [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]),
            "ora_dfp_linear_fwd": (None, [P, P] + [ctypes.c_int] * 3 + [P]),
            "ora_dfp_linear_dgrad": (None, [P, P] + [ctypes.c_int] * 3 + [P]),
            "ora_dfp_linear_wgrad": (None, [P, P] + [ctypes.c_int] * 3 + [P]),
            "ora_dfp_down": (i32, [P, i64, i32, P, P]),
            "ora_dfp_update": (i64, [P, P, i64, i32, i32]),
            "ora_dfp_set_bits": (i32, [P, i64, i32, i32]),
            "ora_bdfp_from_float": (None, [P, i64, i64, i32, P, P]),
            "ora_bdfp_to_float": (None, [P, P, i64, i64, i32, P]),
            "ora_bdfp_linear_fwd_f32": (None, [P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]),
            "ora_abs_sum16": (i64, [P, i64]),
            "ora_dfp_from_float": (i32, [P, i64, P]),
            "ora_dfp_to_float": (None, [P, i64, i32, P]),
            "ora_p64_to_float": (None, [P, i64, i32, P]),
            "ora_dfp_linear_fwd_f32_chained": (None, [P, i32, P, i32] + [ctypes.c_int] * 5 + [P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ------------------------------------------------------------------ scalars

def bitlen(m: int) -> int:
    return lib().ora_bitlen(m)


def shift_from_max(m: int, target_bits: int = TARGET_BITS) -> int:
    return lib().ora_shift_from_max(m, target_bits)


def rhu(x: int, s: int) -> int:
    return lib().ora_rhu(x, s)


def sat8(v: int) -> int:
    return lib().ora_sat8(v)


def sat16(v: int) -> int:
    return lib().ora_sat16(v)


# ---------------------------------------------------------- tensor primitives

def absmax32(v) -> int:
    v = _c(v, np.int32)
    return lib().ora_absmax32(_p(v), v.size)


def requant(Y, relu: bool, target_bits: int = TARGET_BITS):
    """-> (int8 tensor, shift, max|Y|)"""
    Y = _c(Y, np.int32)
    out = np.empty(Y.shape, np.int8)
    m = ctypes.c_uint32()
    s = lib().ora_requant(_p(Y), Y.size, target_bits, int(relu), _p(out), ctypes.byref(m))
    return out, s, m.value


def requant_mask(D, a_prev, target_bits: int = TARGET_BITS):
    """-> (int8 delta, shift, max|D|); a_prev None means no ReLU gate."""
    D = _c(D, np.int32)
    out = np.empty(D.shape, np.int8)
    m = ctypes.c_uint32()
    if a_prev is None:
        ap = None
    else:
        a_prev = _c(a_prev, np.int8)
        assert a_prev.size == D.size
        ap = _p(a_prev)
    s = lib().ora_requant_mask(_p(D), ap, D.size, target_bits, _p(out), ctypes.byref(m))
    return out, s, m.value


def top_error(logits, labels, target_mag: int = TARGET_MAG):
    logits = _c(logits, np.int8)
    labels = _c(labels, np.int32)
    B, C = logits.shape
    out = np.empty((B, C), np.int8)
    lib().ora_top_error(_p(logits), _p(labels), B, C, target_mag, _p(out))
    return out


def niti_update(W, G, target_bits: int = TARGET_BITS, mu_weight: int = MU_WEIGHT):
    """Returns (new W, shift, weight_shift, max|G|, nonzero count); W is not modified."""
    Wn = np.array(W, dtype=np.int8, copy=True, order="C")
    G = _c(G, np.int32)
    assert G.size == Wn.size
    s, ws, m = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_uint32()
    nz = lib().ora_niti_update(_p(Wn), _p(G), G.size, target_bits, mu_weight,
                               ctypes.byref(s), ctypes.byref(ws), ctypes.byref(m))
    return Wn, s.value, ws.value, m.value, nz


def linear_fwd(X, W):
    X, W = _c(X, np.int8), _c(W, np.int8)
    B, IC = X.shape
    OC = W.shape[0]
    assert W.shape == (OC, IC)
    Y = np.empty((B, OC), np.int32)
    lib().ora_linear_fwd(_p(X), _p(W), B, IC, OC, _p(Y))
    return Y


def linear_dgrad(delta, W):
    delta, W = _c(delta, np.int8), _c(W, np.int8)
    B, OC = delta.shape
    IC = W.shape[1]
    assert W.shape == (OC, IC)
    D = np.empty((B, IC), np.int32)
    lib().ora_linear_dgrad(_p(delta), _p(W), B, IC, OC, _p(D))
    return D


def linear_wgrad(delta, A):
    delta, A = _c(delta, np.int8), _c(A, np.int8)
    B, OC = delta.shape
    IC = A.shape[1]
    assert A.shape[0] == B
    G = np.empty((OC, IC), np.int32)
    lib().ora_linear_wgrad(_p(delta), _p(A), B, IC, OC, _p(G))
    return G


def linear_fwd_u8(X, W):
    X, W = _c(X, np.uint8), _c(W, np.int8)
    B, IC = X.shape
    OC = W.shape[0]
    assert W.shape == (OC, IC)
    Y = np.empty((B, OC), np.int32)
    lib().ora_linear_fwd_u8(_p(X), _p(W), B, IC, OC, _p(Y))
    return Y


def linear_wgrad_u8(delta, A):
    delta, A = _c(delta, np.int8), _c(A, np.uint8)
    B, OC = delta.shape
    IC = A.shape[1]
    assert A.shape[0] == B
    G = np.empty((OC, IC), np.int32)
    lib().ora_linear_wgrad_u8(_p(delta), _p(A), B, IC, OC, _p(G))
    return G


def requant_static(Y, offset, mult, k, relu: bool):
    Y = _c(Y, np.int32)
    B, C = Y.shape
    offset, mult, k = _c(offset, np.int32), _c(mult, np.int32), _c(k, np.int32)
    assert offset.size == mult.size == k.size == C
    out = np.empty((B, C), np.int8)
    lib().ora_requant_static(_p(Y), B, C, _p(offset), _p(mult), _p(k), int(relu), _p(out))
    return out


def offset_grad(delta):
    delta = _c(delta, np.int8)
    B, C = delta.shape
    g = np.empty(C, np.int32)
    lib().ora_offset_grad(_p(delta), B, C, _p(g))
    return g


def offset_update(offset, g, target_bits: int = TARGET_BITS, mu_weight: int = MU_WEIGHT):
    """-> (new offsets, shift, weight_shift, max|g|, nonzero count)"""
    on = np.array(offset, dtype=np.int32, copy=True, order="C")
    g = _c(g, np.int32)
    s, ws, m = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_uint32()
    nz = lib().ora_offset_update(_p(on), _p(g), g.size, target_bits, mu_weight, ctypes.byref(s), ctypes.byref(ws),
                                 ctypes.byref(m))
    return on, s.value, ws.value, m.value, nz


def pack_relu_mask(A):
    A = _c(A, np.int8)
    B, F = A.shape
    out = np.empty((B, (F + 7) // 8), np.uint8)
    lib().ora_pack_relu_mask(_p(A), B, F, _p(out))
    return out


# Exact float64 route for large contractions. Every product of two integers
# is exact in float64, and every partial sum is an integer bounded by
# K * max|A| * max|B|; below 2^53 all of them are exactly representable, so the
# BLAS result is the exact integer sum whatever order or fused multiply-add the
# library uses. The bound is checked before the call.

def _exact_matmul(A, B_T):
    """A [M, K] @ B_T [K, N] over integers, exact in float64 (bound checked)."""
    K = A.shape[1]
    ma = int(np.abs(A.astype(np.int64)).max(initial=0))
    mb = int(np.abs(B_T.astype(np.int64)).max(initial=0))
    if K * ma * mb >= (1 << 53):
        raise OverflowError("float64 route not exact for this contraction")
    r = A.astype(np.float64) @ B_T.astype(np.float64)
    return np.rint(r).astype(np.int64)


def _to_i32(v):
    if v.size and (v.max() > np.iinfo(np.int32).max or v.min() < np.iinfo(np.int32).min):
        raise OverflowError("int32 overflow in a contraction result")
    return v.astype(np.int32)


def linear_fwd_f64(X, W):
    return _to_i32(_exact_matmul(np.asarray(X), np.asarray(W).T))


def linear_dgrad_f64(delta, W):
    return _to_i32(_exact_matmul(np.asarray(delta), np.asarray(W)))


def linear_wgrad_f64(delta, A):
    return _to_i32(_exact_matmul(np.asarray(delta).T, np.asarray(A)))


def dfp_linear_fwd_f64(X, W):
    return _exact_matmul(np.asarray(X), np.asarray(W).T)


def dfp_linear_dgrad_f64(delta, W):
    return _exact_matmul(np.asarray(delta), np.asarray(W))


def dfp_linear_wgrad_f64(delta, A):
    return _exact_matmul(np.asarray(delta).T, np.asarray(A))


def conv_out(n: int, k: int = 3, stride: int = 1, pad: int = 1) -> int:
    return (n + 2 * pad - k) // stride + 1


def conv2d_fwd(X, Wt, stride: int, pad: int = 1):
    X, Wt = _c(X, np.int8), _c(Wt, np.int8)
    B, H, Wd, IC = X.shape
    OC, KH, KW, IC2 = Wt.shape
    assert IC == IC2
    OH, OW = conv_out(H, KH, stride, pad), conv_out(Wd, KW, stride, pad)
    Y = np.empty((B, OH, OW, OC), np.int32)
    lib().ora_conv2d_fwd(_p(X), _p(Wt), B, H, Wd, IC, OC, KH, KW, stride, pad, _p(Y))
    return Y


def conv2d_dgrad(delta, Wt, in_hw, stride: int, pad: int = 1):
    delta, Wt = _c(delta, np.int8), _c(Wt, np.int8)
    B = delta.shape[0]
    OC, KH, KW, IC = Wt.shape
    H, Wd = in_hw
    assert delta.shape == (B, conv_out(H, KH, stride, pad), conv_out(Wd, KW, stride, pad), OC)
    D = np.empty((B, H, Wd, IC), np.int32)
    lib().ora_conv2d_dgrad(_p(delta), _p(Wt), B, H, Wd, IC, OC, KH, KW, stride, pad, _p(D))
    return D


def conv2d_wgrad(delta, X, k: int, stride: int, pad: int = 1):
    delta, X = _c(delta, np.int8), _c(X, np.int8)
    B, H, Wd, IC = X.shape
    OC = delta.shape[3]
    assert delta.shape == (B, conv_out(H, k, stride, pad), conv_out(Wd, k, stride, pad), OC)
    G = np.empty((OC, k, k, IC), np.int32)
    lib().ora_conv2d_wgrad(_p(delta), _p(X), B, H, Wd, IC, OC, k, k, stride, pad, _p(G))
    return G


def gap_fwd(A):
    A = _c(A, np.int8)
    B, H, Wd, C = A.shape
    P = np.empty((B, C), np.int32)
    lib().ora_gap_fwd(_p(A), B, H * Wd, C, _p(P))
    return P


def gap_bwd(dP, A):
    dP, A = _c(dP, np.int8), _c(A, np.int8)
    B, H, Wd, C = A.shape
    assert dP.shape == (B, C)
    D = np.empty(A.shape, np.int8)
    lib().ora_gap_bwd(_p(dP), _p(A), B, H * Wd, C, _p(D))
    return D


def dfp_linear_fwd(X, W):
    X, W = _c(X, np.int16), _c(W, np.int16)
    B, IC = X.shape
    OC = W.shape[0]
    assert W.shape == (OC, IC)
    P = np.empty((B, OC), np.int64)
    lib().ora_dfp_linear_fwd(_p(X), _p(W), B, IC, OC, _p(P))
    return P


def dfp_linear_dgrad(delta, W):
    delta, W = _c(delta, np.int16), _c(W, np.int16)
    B, OC = delta.shape
    IC = W.shape[1]
    assert W.shape == (OC, IC)
    P = np.empty((B, IC), np.int64)
    lib().ora_dfp_linear_dgrad(_p(delta), _p(W), B, IC, OC, _p(P))
    return P


def dfp_linear_wgrad(delta, A):
    delta, A = _c(delta, np.int16), _c(A, np.int16)
    B, OC = delta.shape
    IC = A.shape[1]
    P = np.empty((OC, IC), np.int64)
    lib().ora_dfp_linear_wgrad(_p(delta), _p(A), B, IC, OC, _p(P))
    return P


def dfp_down(P, exp_in: int, target_bits: int = DFP_BITS):
    """-> (int16 mantissas, new exponent, Rs, max|P|). Raises if the new
    exponent leaves the signed 8-bit range the DFP format stores it in."""
    P = _c(P, np.int64)
    out = np.empty(P.shape, np.int16)
    m = ctypes.c_uint64()
    rs = lib().ora_dfp_down(_p(P), P.size, target_bits, _p(out), ctypes.byref(m))
    e = exp_in + rs
    if not -128 <= e <= 127:
        raise OverflowError("DFP exponent %d outside int8" % e)
    return out, e, rs, m.value


def dfp_from_float(f):
    """float32 tensor -> (int16 mantissas, shared exponent)."""
    f = _c(f, np.float32)
    out = np.empty(f.shape, np.int16)
    e = lib().ora_dfp_from_float(_p(f), f.size, _p(out))
    return out, e


def dfp_to_float(m, e: int):
    m = _c(m, np.int16)
    out = np.empty(m.shape, np.float32)
    lib().ora_dfp_to_float(_p(m), m.size, e, _p(out))
    return out


def p64_to_float(P, e: int):
    P = _c(P, np.int64)
    out = np.empty(P.shape, np.float32)
    lib().ora_p64_to_float(_p(P), P.size, e, _p(out))
    return out


def dfp_linear_fwd_f32_chained(x, ex: int, W, ew: int, chain: int, input_shift: bool = True):
    """Linear forward with FP32 output by the partial-accumulation scheme of
    [DFP] section 4 (ora_dfp_linear_fwd_f32_chained): inputs shifted by one bit,
    INT32 chains of `chain` terms, each converted to FP32, scaled by
    2^(E_inp + E_wt) and accumulated in FP32 in chain order."""
    x, W = _c(x, np.int16), _c(W, np.int16)
    B, IC = x.shape
    OC = W.shape[0]
    assert W.shape == (OC, IC)
    y = np.empty((B, OC), np.float32)
    lib().ora_dfp_linear_fwd_f32_chained(_p(x), int(ex), _p(W), int(ew), B, IC, OC, int(chain), int(input_shift),
                                         _p(y))
    return y


def bdfp_from_float(f, block: int):
    """float32 [rows][cols] -> (int16 mantissas, int32 exponents [rows][ceil(cols / block)])
    (Blocked-DFP: ora_bdfp_from_float)."""
    f = _c(f, np.float32)
    rows, cols = f.shape
    nb = (cols + block - 1) // block
    out = np.empty(f.shape, np.int16)
    ex = np.empty((rows, nb), np.int32)
    lib().ora_bdfp_from_float(_p(f), rows, cols, block, _p(out), _p(ex))
    if ex.size and (ex.min() < -128 or ex.max() > 127):
        raise OverflowError("a block exponent leaves int8")
    return out, ex


def bdfp_to_float(m, ex, block: int):
    m, ex = _c(m, np.int16), _c(ex, np.int32)
    out = np.empty(m.shape, np.float32)
    lib().ora_bdfp_to_float(_p(m), _p(ex), m.shape[0], m.shape[1], block, _p(out))
    return out


def bdfp_linear_fwd_f32(x, ex, W, ew, block: int):
    x, W = _c(x, np.int16), _c(W, np.int16)
    ex, ew = _c(ex, np.int32), _c(ew, np.int32)
    B, IC = x.shape
    OC = W.shape[0]
    nb = (IC + block - 1) // block
    assert W.shape == (OC, IC) and ex.shape == (B, nb) and ew.shape == (OC, nb)
    y = np.empty((B, OC), np.float32)
    lib().ora_bdfp_linear_fwd_f32(_p(x), _p(ex), _p(W), _p(ew), B, IC, OC, block, _p(y))
    return y


def dfp_update(W, Gm, k: int, bits: int = 16):
    """W <- sat_bits(W - rhu(Gm, k)) (left shift for k < 0) -> (W, nonzero count)"""
    if not 2 <= bits <= 16:
        raise ValueError("bits must be 2 .. 16")
    Wn = np.array(W, dtype=np.int16, copy=True, order="C")
    Gm = _c(Gm, np.int16)
    nz = lib().ora_dfp_update(_p(Wn), _p(Gm), Gm.size, k, bits)
    return Wn, nz


def dfp_set_bits(W, bits_old: int, bits_new: int):
    """Change a weight tensor's precision (ora_dfp_set_bits) -> (W, exponent change)."""
    if not (2 <= bits_old <= 16 and 2 <= bits_new <= 16):
        raise ValueError("bits must be 2 .. 16")
    Wn = np.array(W, dtype=np.int16, copy=True, order="C")
    if bits_new > bits_old and np.abs(Wn.astype(np.int64)).max(initial=0) > (1 << (bits_old - 1)) - 1:
        raise ValueError("weights exceed the old precision")
    de = lib().ora_dfp_set_bits(_p(Wn), Wn.size, bits_old, bits_new)
    return Wn, de


def abs_sum16(x) -> int:
    x = _c(x, np.int16)
    return int(lib().ora_abs_sum16(_p(x), x.size))


# ------------------------------------------------- adaptive precision (APT)
#
# "Adaptive Precision Training for Resource Constrained Devices", section III.
# Equation 4 (its formula is missing from the page text; reading from the
# prose): Gavg_i = (1/N_i) sum_j |g_ij| / eps_i, the mean gradient magnitude in
# units of the layer's weight resolution, with no learning rate in it. Here
# the weight gradient of the integer step is the batch SUM G * 2^E_G; the
# gradient of minibatch SGD that the page's g_ij denotes is its batch mean, so
# g = G * 2^E_G / B; eps = 2^E_W. Hence
# Gavg = sum|G| * 2^(E_G - E_W) / (N * B), evaluated in float64 as written below.

def apt_gavg(gabs: int, n: int, batch: int, exp_g: int, exp_w: int) -> float:
    return math.ldexp(float(gabs), exp_g - exp_w) / float(n * batch)


def apt_policy(bits, gavg, t_min: float, t_max: float, k_min: int, k_max: int):
    """Algorithm 1: raise a layer's precision by one bit when Gavg < T_min,
    lower it by one when Gavg > T_max, within [k_min, k_max]."""
    out = []
    for k, g in zip(bits, gavg):
        if g < t_min and k < k_max:
            k += 1
        elif g > t_max and k > k_min:
            k -= 1
        out.append(k)
    return out


def apt_run(workload, steps: int, callback=None, route="loops"):
    """Algorithm 2 on a DFP workload with an `apt` setting (seeded_inputs):
    the weights start at apt.k_init bits; inside each epoch of apt.epoch
    steps, Gavg is evaluated after every step whose index within the epoch is
    a multiple of apt.eval_every; between epochs Algorithm 1 adjusts each
    layer's precision from the mean of that epoch's evaluations.
    callback(t, record, state) after every step; state = dict(bits, exp_w,
    gavg (the means of the last finished epoch, or None)).
    Returns (weights, exp_w list, bits list)."""
    import seeded_inputs as si
    w, a = workload, workload.apt
    weights = [np.array(x) for x in si.make_weights(w)]
    L = len(weights)
    bits = [16] * L
    exp_w = [w.exp_w] * L
    for l in range(L):
        weights[l], de = dfp_set_bits(weights[l], 16, a.k_init)
        exp_w[l] += de
        bits[l] = a.k_init
    evals = [[] for _ in range(L)]
    last = None
    for t in range(steps):
        x, _ = si.make_batch(w, t)
        rec = dfp16_step(weights, exp_w, x, w.exp_x, eta=w.eta, route=route, wbits=bits)
        weights = [rec["w%d" % l] for l in range(L)]
        te = t % a.epoch
        if te % a.eval_every == 0:
            for l in range(L):
                evals[l].append(apt_gavg(rec["gabs%d" % l], weights[l].size, w.batch, rec["eg%d" % l], exp_w[l]))
        if te == a.epoch - 1:
            last = [sum(v) / len(v) for v in evals]
            new_bits = apt_policy(bits, last, a.t_min, a.t_max, a.k_min, a.k_max)
            for l in range(L):
                if new_bits[l] != bits[l]:
                    weights[l], de = dfp_set_bits(weights[l], bits[l], new_bits[l])
                    exp_w[l] += de
            bits = new_bits
            evals = [[] for _ in range(L)]
        if callback is not None:
            callback(t, rec, dict(bits=list(bits), exp_w=list(exp_w), gavg=last))
    return weights, exp_w, bits


# ------------------------------------------------------------- training steps

def _linear_ops(route):
    if route == "loops":
        return linear_fwd, linear_dgrad, linear_wgrad
    if route == "f64":
        return linear_fwd_f64, linear_dgrad_f64, linear_wgrad_f64
    raise ValueError(route)


def mlp_step(weights, x, labels, target_bits=TARGET_BITS, mu_weight=MU_WEIGHT,
             target_mag=TARGET_MAG, route="loops", trainable_from=0, static_q=None):
    """One NITI step of a sequential int8 MLP: Linear+ReLU layers and a final
    Linear producing int8 logits. `weights` is a list of int8 [OC, IC]; the
    updated weights are returned in the record (inputs are not modified).

    Record names (layer l counted from 0): y{l} int32 forward contraction,
    ymax{l}/ys{l} its max and shift, a{l} int8 output; e{l} int8 delta at the
    output of layer l (e{L-1} is the top error); d{l} int32 delta-propagation
    contraction of layer l (l >= 1) with dmax{l}/ds{l}; g{l} int32 weight
    gradient with gmax{l}/gs{l}/ws{l}; w{l} updated weights; nz{l} nonzero
    weight steps. route: "loops" (C loops) or "f64" (exact float64 BLAS).

    Partial-model training ("Integer On-Device Training: Overview", section 5,
    trainable_layers_from_last): layers before `trainable_from` are frozen and
    run forward only; backward stops at layer trainable_from (no delta is
    propagated into the frozen part). A uint8 `x` is the UINT8 input the
    library receives from a frozen prefix ending in ReLU (values 0..255).

    static_q: None, or per layer None / dict(offset, mult, k) for the TI
    library's static forward requantisation (requant_static) with trained
    INT32 offsets: record names off{l} (updated offsets), og{l} offset
    gradient, ogmax{l}/ogs{l}/ows{l}/onz{l}."""
    fwd, dgrad, wgrad = _linear_ops(route)
    L = len(weights)
    r = {}
    u8_input = np.asarray(x).dtype == np.uint8
    act = [np.ascontiguousarray(x, np.uint8 if u8_input else np.int8)]
    for l in range(L):
        if l == 0 and u8_input:
            y = linear_fwd_u8(act[-1], weights[l]) if route == "loops" else linear_fwd_f64(act[-1], weights[l])
        else:
            y = fwd(act[-1], weights[l])
        sq = static_q[l] if static_q else None
        if sq is not None:
            a = requant_static(y, sq["offset"], sq["mult"], sq["k"], relu=(l < L - 1))
            r["y%d" % l], r["ymax%d" % l], r["a%d" % l] = y, absmax32(y), a
        else:
            a, s, m = requant(y, relu=(l < L - 1), target_bits=target_bits)
            r["y%d" % l], r["ymax%d" % l], r["ys%d" % l], r["a%d" % l] = y, m, s, a
        act.append(a)
    e = top_error(act[-1], labels, target_mag)
    r["e%d" % (L - 1)] = e
    for l in range(L - 1, trainable_from - 1, -1):
        if l > trainable_from:
            d = dgrad(e, weights[l])
            e_prev, s, m = requant_mask(d, act[l], target_bits)
            r["d%d" % l], r["dmax%d" % l], r["ds%d" % l], r["e%d" % (l - 1)] = d, m, s, e_prev
        if l == 0 and u8_input:
            g = linear_wgrad_u8(e, act[0]) if route == "loops" else linear_wgrad_f64(e, act[0])
        else:
            g = wgrad(e, act[l])
        wn, s, ws, m, nz = niti_update(weights[l], g, target_bits, mu_weight)
        r["g%d" % l], r["gmax%d" % l], r["gs%d" % l], r["ws%d" % l] = g, m, s, ws
        r["w%d" % l], r["nz%d" % l] = wn, nz
        sq = static_q[l] if static_q else None
        if sq is not None:
            og = offset_grad(e)
            on, s, ws, m, nz = offset_update(sq["offset"], og, target_bits, mu_weight)
            r["og%d" % l], r["ogmax%d" % l], r["ogs%d" % l], r["ows%d" % l] = og, m, s, ws
            r["off%d" % l], r["onz%d" % l] = on, nz
        if l > trainable_from:
            e = e_prev
    for l in range(trainable_from):
        r["w%d" % l] = np.array(weights[l], copy=True)      # frozen
        if static_q and static_q[l] is not None:
            r["off%d" % l] = np.array(static_q[l]["offset"], dtype=np.int32, copy=True)
    return r


def cnn_step(weights, x, labels, convs, target_bits=TARGET_BITS, mu_weight=MU_WEIGHT,
             target_mag=TARGET_MAG):
    """One NITI step of the integer CNN: 3x3 Conv+ReLU layers (pad 1, strides
    from `convs`), integer-sum global pooling requantised without ReLU, and a
    final Linear to logits. weights = conv [OC,3,3,IC] ..., then fc [C, F].

    Extra record names: p int32 pooled sum with pmax/ps, pa int8 pooled
    activation; the fc layer is layer n = len(convs): y{n}, a{n} (logits),
    e{n} top error, d{n} its delta-propagation contraction and pe (pooled delta,
    no ReLU gate), then e{n-1} = pooling backward gated by a{n-1} > 0."""
    n = len(convs)
    r = {}
    act = [np.ascontiguousarray(x, np.int8)]
    for l, (_ic, _oc, stride) in enumerate(convs):
        y = conv2d_fwd(act[-1], weights[l], stride)
        a, s, m = requant(y, relu=True, target_bits=target_bits)
        r["y%d" % l], r["ymax%d" % l], r["ys%d" % l], r["a%d" % l] = y, m, s, a
        act.append(a)
    p = gap_fwd(act[-1])
    pa, s, m = requant(p, relu=False, target_bits=target_bits)
    r["p"], r["pmax"], r["ps"], r["pa"] = p, m, s, pa
    y = linear_fwd(pa, weights[n])
    logits, s, m = requant(y, relu=False, target_bits=target_bits)
    r["y%d" % n], r["ymax%d" % n], r["ys%d" % n], r["a%d" % n] = y, m, s, logits
    e = top_error(logits, labels, target_mag)
    r["e%d" % n] = e
    # fc layer
    d = linear_dgrad(e, weights[n])
    pe, s, m = requant_mask(d, None, target_bits)
    r["d%d" % n], r["dmax%d" % n], r["ds%d" % n], r["pe"] = d, m, s, pe
    g = linear_wgrad(e, pa)
    wn, s, ws, m, nz = niti_update(weights[n], g, target_bits, mu_weight)
    r["g%d" % n], r["gmax%d" % n], r["gs%d" % n], r["ws%d" % n] = g, m, s, ws
    r["w%d" % n], r["nz%d" % n] = wn, nz
    e = gap_bwd(pe, act[n])
    r["e%d" % (n - 1)] = e
    for l in range(n - 1, -1, -1):
        stride = convs[l][2]
        if l > 0:
            H, Wd = act[l].shape[1:3]
            d = conv2d_dgrad(e, weights[l], (H, Wd), stride)
            e_prev, s, m = requant_mask(d, act[l], target_bits)
            r["d%d" % l], r["dmax%d" % l], r["ds%d" % l], r["e%d" % (l - 1)] = d, m, s, e_prev
        g = conv2d_wgrad(e, act[l], 3, stride)
        wn, s, ws, m, nz = niti_update(weights[l], g, target_bits, mu_weight)
        r["g%d" % l], r["gmax%d" % l], r["gs%d" % l], r["ws%d" % l] = g, m, s, ws
        r["w%d" % l], r["nz%d" % l] = wn, nz
        if l > 0:
            e = e_prev
    return r


def dfp16_step(weights, exp_w, x, exp_x, eta=DFP_ETA, target_bits=DFP_BITS, route="loops", wbits=None):
    """One integer training step of a stack of DFP-16 Linear layers (no ReLU).
    weights: list of int16 mantissa tensors [OC, IC] with exponent exp_w (one
    int for all layers, or a list per layer; held fixed by the step); x: int16
    mantissas [B, IC0] with exponent exp_x. wbits: per-layer weight precision
    in bits (default 16), the saturation range of the update.

    Every contraction is exact in int64 and is down-converted to DFP-16 with a
    new exponent. The top error is the output itself (an MSE error against a
    zero target). The update is integer SGD with rate 2^-eta (ora_dfp_update).

    Record names: p{l} int64 forward contraction, pmax{l}, rs{l}, y{l} int16,
    ey{l} exponent; e{l}/ee{l} delta at the output of layer l; pd{l} int64
    delta-propagation contraction (l >= 1) with pdmax{l}, rsd{l}; pg{l} int64
    weight gradient with pgmax{l}, rsg{l}, g{l} int16, eg{l}; k{l} the update
    shift; w{l} updated weights; nz{l}; gabs{l} = sum |g{l}|. route: "loops"
    or "f64"."""
    if route == "loops":
        dfwd, ddgrad, dwgrad = dfp_linear_fwd, dfp_linear_dgrad, dfp_linear_wgrad
    elif route == "f64":
        dfwd, ddgrad, dwgrad = dfp_linear_fwd_f64, dfp_linear_dgrad_f64, dfp_linear_wgrad_f64
    else:
        raise ValueError(route)
    L = len(weights)
    ew = list(exp_w) if isinstance(exp_w, (list, tuple)) else [exp_w] * L
    wb = list(wbits) if wbits is not None else [16] * L
    r = {}
    act = [np.ascontiguousarray(x, np.int16)]
    ex = [exp_x]
    for l in range(L):
        p = dfwd(act[-1], weights[l])
        y, e_y, rs, m = dfp_down(p, ex[-1] + ew[l], target_bits)
        r["p%d" % l], r["pmax%d" % l], r["rs%d" % l], r["y%d" % l], r["ey%d" % l] = p, m, rs, y, e_y
        act.append(y)
        ex.append(e_y)
    e, ee = act[-1], ex[-1]
    r["e%d" % (L - 1)], r["ee%d" % (L - 1)] = e, ee
    for l in range(L - 1, -1, -1):
        if l > 0:
            pd = ddgrad(e, weights[l])
            e_prev, ee_prev, rs, m = dfp_down(pd, ee + ew[l], target_bits)
            r["pd%d" % l], r["pdmax%d" % l], r["rsd%d" % l] = pd, m, rs
            r["e%d" % (l - 1)], r["ee%d" % (l - 1)] = e_prev, ee_prev
        pg = dwgrad(e, act[l])
        g, eg, rs, m = dfp_down(pg, ee + ex[l], target_bits)
        k = ew[l] + eta - eg
        wn, nz = dfp_update(weights[l], g, k, wb[l])
        r["gabs%d" % l] = abs_sum16(g)
        r["pg%d" % l], r["pgmax%d" % l], r["rsg%d" % l], r["g%d" % l], r["eg%d" % l] = pg, m, rs, g, eg
        r["k%d" % l], r["w%d" % l], r["nz%d" % l] = k, wn, nz
        if l > 0:
            e, ee = e_prev, ee_prev
    return r


def run_steps(workload, steps: int, start_weights=None, callback=None, route="loops"):
    """Run `steps` training steps of a seeded workload (seeded_inputs.Workload),
    feeding each step's updated weights (and offsets) to the next.
    callback(t, record) is called after every step. Returns the final weights."""
    import seeded_inputs as si
    w = workload
    weights = [np.array(a) for a in (start_weights or si.make_weights(w))]
    static_q = si.make_static_requant(w)
    for t in range(steps):
        x, labels = si.make_batch(w, t)
        if w.kind == "mlp":
            rec = mlp_step(weights, x, labels, route=route, trainable_from=w.trainable_from, static_q=static_q)
            if static_q:
                static_q = [None if q is None else dict(q, offset=rec["off%d" % l]) for l, q in enumerate(static_q)]
        elif w.kind == "cnn":
            rec = cnn_step(weights, x, labels, w.convs)
        elif w.kind == "dfp16":
            rec = dfp16_step(weights, w.exp_w, x, w.exp_x, eta=w.eta, route=route)
        else:
            raise ValueError(w.kind)
        weights = [rec["w%d" % l] for l in range(len(weights))]
        if callback is not None:
            callback(t, rec)
    return weights
