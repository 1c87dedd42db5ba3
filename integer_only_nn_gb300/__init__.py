"""Python binding of libito.so, the integer-only (NITI / DFP16) training library
for one GB300 GPU.

Argument marshalling only: every function here hands torch tensors' device
pointers and the current CUDA stream to the C ABI declared in include/ito.h,
under the same names. All arithmetic runs in the library's CUDA kernels. If the
shared library has not been built, importing this package raises ImportError;
there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libito.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libito.so is not built: run `python -m integer_only_nn_gb300.build` "
                      "(or __graft_entry__.build()) on a machine with nvcc")

_lib = ctypes.CDLL(LIB_PATH)

ITO_OK, ITO_ERR_ARG, ITO_ERR_SHAPE, ITO_ERR_CUDA, ITO_ERR_TIMEOUT, ITO_ERR_EXPONENT, ITO_ERR_UNSUPPORTED = range(7)
ITO_LAYER_LINEAR, ITO_LAYER_LINEAR_RELU, ITO_LAYER_CONV3X3_RELU, ITO_LAYER_GAP = range(4)

_P = ctypes.c_void_p
_I = ctypes.c_int
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t


class NitiParams(ctypes.Structure):
    _fields_ = [("target_bits", ctypes.c_int32), ("mu_weight", ctypes.c_int32)]


class ModelOptions(ctypes.Structure):
    _fields_ = [("input_uint8", ctypes.c_int32), ("trainable_from", ctypes.c_int32),
                ("packed_masks", ctypes.c_int32), ("pingpong_grads", ctypes.c_int32),
                ("speculate_min_elems", ctypes.c_int32)]


class AptParams(ctypes.Structure):
    _fields_ = [("k_init", ctypes.c_int32), ("k_min", ctypes.c_int32), ("k_max", ctypes.c_int32),
                ("eval_every", ctypes.c_int32), ("t_min", ctypes.c_double), ("t_max", ctypes.c_double)]


class LayerDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("in_features", ctypes.c_int32), ("out_features", ctypes.c_int32),
                ("in_h", ctypes.c_int32), ("in_w", ctypes.c_int32), ("stride", ctypes.c_int32)]


_SIGS = {
    "ito_version": (_I, []),
    "ito_get_error": (_I, []),
    "ito_last_error_string": (ctypes.c_char_p, []),
    "ito_selftest_wait_timeout": (_I, [_P]),
    "ito_linear_workspace_size": (_SZ, [_I, _I, _I]),
    "ito_linear_fwd": (_I, [_P, _P, _I, _I, _I, _I, NitiParams, _P, _SZ, _P, _P, _P, _P, _P]),
    "ito_linear_fwd_noalloc": (_I, [_P, _P, _I, _I, _I, _I, NitiParams, _P, _P, _P, _P, _P]),
    "ito_linear_bwd_delta": (_I, [_P, _P, _P, _I, _I, _I, NitiParams, _P, _SZ, _P, _P, _P, _P, _P]),
    "ito_linear_wgrad": (_I, [_P, _P, _I, _I, _I, _P, _SZ, _P, _P, _P]),
    "ito_niti_update": (_I, [_P, _P, _I64, _P, NitiParams, _P, _P, _P, _P]),
    "ito_top_error": (_I, [_P, _P, _I, _I, _I32, _P, _P]),
    "ito_conv2d_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "ito_conv2d_fwd": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, NitiParams, _P, _SZ, _P, _P, _P, _P, _P]),
    "ito_conv2d_bwd_delta": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, NitiParams, _P, _SZ, _P, _P, _P, _P,
                                  _P]),
    "ito_conv2d_wgrad": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P, _P, _P]),
    "ito_gap_fwd": (_I, [_P, _I, _I, _I, NitiParams, _P, _P, _P, _P, _P]),
    "ito_gap_bwd": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "ito_model_create": (_I, [ctypes.POINTER(LayerDesc), _I, _I, NitiParams, _I32, ctypes.POINTER(_P)]),
    "ito_model_create_ex": (_I, [ctypes.POINTER(LayerDesc), _I, _I, NitiParams, _I32, ctypes.POINTER(ModelOptions),
                                 ctypes.POINTER(_P)]),
    "ito_model_destroy": (_I, [_P]),
    "ito_model_set_weights": (_I, [_P, _I, _P, _I, _P]),
    "ito_model_get_weights": (_I, [_P, _I, _P, _I, _P]),
    "ito_model_tensor": (_I, [_P, ctypes.c_char_p, ctypes.POINTER(_P), ctypes.POINTER(_I), ctypes.POINTER(_I64)]),
    "ito_model_stat_index": (_I, [_P, ctypes.c_char_p]),
    "ito_model_num_stats": (_I, [_P]),
    "ito_train_step": (_I, [_P, _P, _P, _P]),
    "ito_train_step_host": (_I, [_P, _P, _P, _P, _P]),
    "ito_train_step_host_async": (_I, [_P, _P, _P, _P, _P]),
    "ito_infer": (_I, [_P, _P, _P, _P]),
    "ito_model_save": (_I, [_P, ctypes.c_char_p]),
    "ito_model_load": (_I, [_P, ctypes.c_char_p]),
    "ito_dfp16_workspace_size": (_SZ, [_I, _I, _I]),
    "ito_dfp16_linear_fwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P, _P, _P, _P, _P, _P]),
    "ito_dfp16_linear_bwd_delta": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P, _P, _P, _P, _P, _P]),
    "ito_dfp16_linear_wgrad": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P, _P, _P, _P, _P, _P]),
    "ito_dfp16_update": (_I, [_P, _P, _P, _I64, _I32, _I32, _P, _P, _P]),
    "ito_dfp16_from_float": (_I, [_P, _I64, _P, _P, _P, _P]),
    "ito_dfp16_to_float": (_I, [_P, _P, _I64, _P, _P]),
    "ito_dfp16_linear_fwd_f32": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P, _P, _P, _P]),
    "ito_dfp16_linear_fwd_f32_chained": (_I, [_P, _P, _P, _P, _I, _I, _I, _I32, _I32, _P, _SZ, _P, _P]),
    "ito_dfp16_model_create": (_I, [_P, _I, _I, _I32, _I32, ctypes.POINTER(_P)]),
    "ito_dfp16_model_destroy": (_I, [_P]),
    "ito_dfp16_model_set_weights": (_I, [_P, _I, _P, _I, _P]),
    "ito_dfp16_model_tensor": (_I, [_P, ctypes.c_char_p, ctypes.POINTER(_P), ctypes.POINTER(_I),
                                    ctypes.POINTER(_I64)]),
    "ito_dfp16_model_num_stats": (_I, [_P]),
    "ito_dfp16_model_stat_index": (_I, [_P, ctypes.c_char_p]),
    "ito_dfp16_model_read_stats": (_I, [_P, _P, _I]),
    "ito_dfp16_train_step": (_I, [_P, _P, _I32, _P]),
    "ito_dfp16_train_step_host_async": (_I, [_P, _P, _I32, _P, _P]),
    "ito_dfp16_model_profile": (_I, [_P, _I]),
    "ito_dfp16_model_profile_read": (_I, [_P, _P, _P, _P]),
    "ito_dfp16_model_kernels_per_step": (_I, [_P]),
    "ito_model_use_graphs": (_I, [_P, _I]),
    "ito_model_set_overlap": (_I, [_P, _I]),
    "ito_model_set_speculation": (_I, [_P, _I]),
    "ito_model_get_speculation": (_I, [_P, _P]),
    "ito_model_get_overlap": (_I, [_P, _P]),
    "ito_model_set_static_requant": (_I, [_P, _I, _P, _P, _P, _I, _P]),
    "ito_model_profile": (_I, [_P, _I]),
    "ito_model_profile_read": (_I, [_P, _P, _P, _P]),
    "ito_model_kernels_per_step": (_I, [_P]),
    "ito_dfp16_update_bits": (_I, [_P, _P, _P, _I64, _I32, _I32, _I32, _P, _P, _P]),
    "ito_dfp_set_bits": (_I, [_P, _I64, _I32, _I32, _P]),
    "ito_bdfp16_from_float": (_I, [_P, _I64, _I64, _I32, _P, _P, _P]),
    "ito_bdfp16_to_float": (_I, [_P, _P, _I64, _I64, _I32, _P, _P]),
    "ito_bdfp16_linear_fwd_f32": (_I, [_P, _P, _P, _P, _I, _I, _I, _I32, _P, _SZ, _P, _P]),
    "ito_dfp16_model_get_precision": (_I, [_P, _I, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "ito_dfp16_model_set_precision": (_I, [_P, _I, _I32, _P]),
    "ito_dfp16_model_apt_enable": (_I, [_P, ctypes.POINTER(AptParams), _P]),
    "ito_dfp16_model_apt_epoch_end": (_I, [_P, _P, _P, _P]),
}

for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


class ItoError(RuntimeError):
    def __init__(self, code, text):
        super().__init__("ito status %d: %s" % (code, text))
        self.code = code


def _check(code):
    if code != ITO_OK:
        raise ItoError(code, _lib.ito_last_error_string().decode(errors="replace"))
    return code


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def params(target_bits=7, mu_weight=2) -> NitiParams:
    return NitiParams(target_bits, mu_weight)


def ito_version() -> int:
    return _lib.ito_version()


def ito_get_error() -> int:
    return _lib.ito_get_error()


def ito_selftest_wait_timeout(stream=None):
    """A kernel whose bounded wait runs out (about 2 s); ito_get_error() then reports ITO_ERR_TIMEOUT."""
    _check(_lib.ito_selftest_wait_timeout(_stream(stream)))


# ----------------------------------------------------------- single layer

def _workspace(B, IC, OC, device):
    torch = _torch()
    n = _lib.ito_linear_workspace_size(B, IC, OC)
    return torch.empty(n + 256, dtype=torch.uint8, device=device), n


def _aligned256(buf):
    off = (-buf.data_ptr()) % 256
    return ctypes.c_void_p(buf.data_ptr() + off)


def ito_linear_fwd(x, W, relu, p=None, stream=None):
    """-> (y32 int32 [B][OC], d_max uint32 as int32 [1], d_shift int32 [1], y int8 [B][OC])"""
    torch = _torch()
    B, IC = x.shape
    OC = W.shape[0]
    dev = x.device
    y32 = torch.empty((B, OC), dtype=torch.int32, device=dev)
    y = torch.empty((B, OC), dtype=torch.int8, device=dev)
    mx = torch.zeros(1, dtype=torch.int32, device=dev)
    sh = torch.zeros(1, dtype=torch.int32, device=dev)
    ws, n = _workspace(B, IC, OC, dev)
    _check(_lib.ito_linear_fwd(_ptr(x), _ptr(W), B, IC, OC, int(relu), p or params(), _aligned256(ws), n,
                               _ptr(y32), _ptr(mx), _ptr(sh), _ptr(y), _stream(stream)))
    return y32, mx, sh, y


def ito_linear_fwd_noalloc(x, W, relu, p=None, stream=None, out=None):
    """ito_linear_fwd using the library's built-in scratch instead of a
    workspace (the library allocates nothing). `out` may hold preallocated
    (y32, d_max, d_shift, y) tensors; -> the same four tensors."""
    torch = _torch()
    B, IC = x.shape
    OC = W.shape[0]
    dev = x.device
    if out is None:
        out = (torch.empty((B, OC), dtype=torch.int32, device=dev), torch.zeros(1, dtype=torch.int32, device=dev),
               torch.zeros(1, dtype=torch.int32, device=dev), torch.empty((B, OC), dtype=torch.int8, device=dev))
    y32, mx, sh, y = out
    _check(_lib.ito_linear_fwd_noalloc(_ptr(x), _ptr(W), B, IC, OC, int(relu), p or params(), _ptr(y32), _ptr(mx),
                                       _ptr(sh), _ptr(y), _stream(stream)))
    return y32, mx, sh, y


def ito_linear_bwd_delta(delta, W, a_prev, p=None, stream=None):
    """-> (d32 int32 [B][IC], d_max, d_shift, delta_prev int8 [B][IC])"""
    torch = _torch()
    B, OC = delta.shape
    IC = W.shape[1]
    dev = delta.device
    d32 = torch.empty((B, IC), dtype=torch.int32, device=dev)
    dp = torch.empty((B, IC), dtype=torch.int8, device=dev)
    mx = torch.zeros(1, dtype=torch.int32, device=dev)
    sh = torch.zeros(1, dtype=torch.int32, device=dev)
    ws, n = _workspace(B, IC, OC, dev)
    _check(_lib.ito_linear_bwd_delta(_ptr(delta), _ptr(W), _ptr(a_prev), B, IC, OC, p or params(),
                                     _aligned256(ws), n, _ptr(d32), _ptr(mx), _ptr(sh), _ptr(dp), _stream(stream)))
    return d32, mx, sh, dp


def ito_linear_wgrad(delta, a_prev, stream=None):
    """-> (G int32 [OC][IC], d_max)"""
    torch = _torch()
    B, OC = delta.shape
    IC = a_prev.shape[1]
    dev = delta.device
    G = torch.empty((OC, IC), dtype=torch.int32, device=dev)
    mx = torch.zeros(1, dtype=torch.int32, device=dev)
    ws, n = _workspace(B, IC, OC, dev)
    _check(_lib.ito_linear_wgrad(_ptr(delta), _ptr(a_prev), B, IC, OC, _aligned256(ws), n, _ptr(G), _ptr(mx),
                                 _stream(stream)))
    return G, mx


def ito_niti_update(W, G, d_max, p=None, stream=None):
    """In place on W; -> (d_shift, d_wshift, d_nonzero) device int32 [1] each."""
    torch = _torch()
    dev = W.device
    sh = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.zeros(1, dtype=torch.int32, device=dev)
    nz = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(_lib.ito_niti_update(_ptr(W), _ptr(G), W.numel(), _ptr(d_max), p or params(), _ptr(sh), _ptr(ws),
                                _ptr(nz), _stream(stream)))
    return sh, ws, nz


def ito_top_error(logits, labels, target_mag=64, stream=None):
    torch = _torch()
    B, C = logits.shape
    d = torch.empty((B, C), dtype=torch.int8, device=logits.device)
    _check(_lib.ito_top_error(_ptr(logits), _ptr(labels), B, C, target_mag, _ptr(d), _stream(stream)))
    return d


def _conv_ws(B, H, W, IC, OC, stride, device):
    torch = _torch()
    n = _lib.ito_conv2d_workspace_size(B, H, W, IC, OC, stride)
    if n == 0:
        raise ItoError(ITO_ERR_SHAPE, "invalid conv sizes")
    return torch.empty(n + 256, dtype=torch.uint8, device=device), n


def _conv_out(n, stride):
    return (n - 1) // stride + 1


def ito_conv2d_fwd(x, Wt, stride, relu, p=None, stream=None):
    """x int8 [B][H][W][IC], Wt int8 [OC][3][3][IC] -> (y32 int32 [B][OH][OW][OC],
    d_max, d_shift, y int8 [B][OH][OW][OC])"""
    torch = _torch()
    B, H, W, IC = x.shape
    OC = Wt.shape[0]
    OH, OW = _conv_out(H, stride), _conv_out(W, stride)
    dev = x.device
    y32 = torch.empty((B, OH, OW, OC), dtype=torch.int32, device=dev)
    y = torch.empty((B, OH, OW, OC), dtype=torch.int8, device=dev)
    mx = torch.zeros(1, dtype=torch.int32, device=dev)
    sh = torch.zeros(1, dtype=torch.int32, device=dev)
    ws, n = _conv_ws(B, H, W, IC, OC, stride, dev)
    _check(_lib.ito_conv2d_fwd(_ptr(x), _ptr(Wt), B, H, W, IC, OC, stride, int(relu), p or params(),
                               _aligned256(ws), n, _ptr(y32), _ptr(mx), _ptr(sh), _ptr(y), _stream(stream)))
    return y32, mx, sh, y


def ito_conv2d_bwd_delta(delta, Wt, a_prev, in_hw, stride, p=None, stream=None):
    """delta int8 [B][OH][OW][OC], a_prev int8 [B][H][W][IC] or None ->
    (d32 int32 [B][H][W][IC], d_max, d_shift, delta_prev int8 [B][H][W][IC])"""
    torch = _torch()
    B, OC = delta.shape[0], delta.shape[3]
    IC = Wt.shape[3]
    H, W = in_hw
    dev = delta.device
    d32 = torch.empty((B, H, W, IC), dtype=torch.int32, device=dev)
    dp = torch.empty((B, H, W, IC), dtype=torch.int8, device=dev)
    mx = torch.zeros(1, dtype=torch.int32, device=dev)
    sh = torch.zeros(1, dtype=torch.int32, device=dev)
    ws, n = _conv_ws(B, H, W, IC, OC, stride, dev)
    _check(_lib.ito_conv2d_bwd_delta(_ptr(delta), _ptr(Wt), _ptr(a_prev), B, H, W, IC, OC, stride, p or params(),
                                     _aligned256(ws), n, _ptr(d32), _ptr(mx), _ptr(sh), _ptr(dp), _stream(stream)))
    return d32, mx, sh, dp


def ito_conv2d_wgrad(delta, x, stride, stream=None):
    """-> (G int32 [OC][3][3][IC], d_max)"""
    torch = _torch()
    B, H, W, IC = x.shape
    OC = delta.shape[3]
    dev = x.device
    G = torch.empty((OC, 3, 3, IC), dtype=torch.int32, device=dev)
    mx = torch.zeros(1, dtype=torch.int32, device=dev)
    ws, n = _conv_ws(B, H, W, IC, OC, stride, dev)
    _check(_lib.ito_conv2d_wgrad(_ptr(delta), _ptr(x), B, H, W, IC, OC, stride, _aligned256(ws), n, _ptr(G),
                                 _ptr(mx), _stream(stream)))
    return G, mx


def ito_gap_fwd(a, p=None, stream=None):
    """a int8 [B][H][W][C] -> (P32 int32 [B][C], d_max, d_shift, pa int8 [B][C])"""
    torch = _torch()
    B, H, W, C = a.shape
    dev = a.device
    P = torch.empty((B, C), dtype=torch.int32, device=dev)
    pa = torch.empty((B, C), dtype=torch.int8, device=dev)
    mx = torch.zeros(1, dtype=torch.int32, device=dev)
    sh = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(_lib.ito_gap_fwd(_ptr(a), B, H * W, C, p or params(), _ptr(P), _ptr(mx), _ptr(sh), _ptr(pa),
                            _stream(stream)))
    return P, mx, sh, pa


def ito_gap_bwd(dP, a, stream=None):
    """dP int8 [B][C], a int8 [B][H][W][C] -> delta int8 [B][H][W][C]"""
    torch = _torch()
    B, H, W, C = a.shape
    d = torch.empty(a.shape, dtype=torch.int8, device=a.device)
    _check(_lib.ito_gap_bwd(_ptr(dP), _ptr(a), B, H * W, C, _ptr(d), _stream(stream)))
    return d


# ------------------------------------------------------------------ model

_DTYPES = {1: "int8", 2: "int16", 4: "int32", 8: "int64"}


def layers_for(workload):
    """ito layer descriptors of a seeded_inputs.Workload (mlp or cnn)."""
    out = []
    if workload.kind == "mlp":
        d = workload.dims
        for i in range(len(d) - 1):
            kind = ITO_LAYER_LINEAR if i == len(d) - 2 else ITO_LAYER_LINEAR_RELU
            out.append(LayerDesc(kind, d[i], d[i + 1], 0, 0, 0))
    elif workload.kind == "cnn":
        H, W, C = workload.image
        for (ic, oc, s) in workload.convs:
            out.append(LayerDesc(ITO_LAYER_CONV3X3_RELU, ic, oc, H, W, s))
            H, W = (H + 2 - 3) // s + 1, (W + 2 - 3) // s + 1
        out.append(LayerDesc(ITO_LAYER_GAP, workload.convs[-1][1], workload.convs[-1][1], H, W, 0))
        out.append(LayerDesc(ITO_LAYER_LINEAR, workload.fc[0], workload.fc[1], 0, 0, 0))
    else:
        raise ValueError(workload.kind)
    return out


class Model:
    """An ito_model: a sequential int8 layer stack that trains with NITI."""

    def __init__(self, layers, batch, target_bits=7, mu_weight=2, target_mag=64, input_uint8=False,
                 trainable_from=0, packed_masks=False, pingpong_grads=False, speculate_min_elems=0):
        arr = (LayerDesc * len(layers))(*layers)
        h = ctypes.c_void_p()
        opt = ModelOptions(int(input_uint8), int(trainable_from), int(packed_masks), int(pingpong_grads),
                           int(speculate_min_elems))
        _check(_lib.ito_model_create_ex(arr, len(layers), batch, NitiParams(target_bits, mu_weight), target_mag,
                                        ctypes.byref(opt), ctypes.byref(h)))
        self._h = h
        self.batch = batch
        self.n_weight_layers = sum(1 for l in layers if l.kind != ITO_LAYER_GAP)

    def close(self):
        if getattr(self, "_h", None):
            _lib.ito_model_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_weights(self, layer, W, stream=None):
        """W: torch int8 tensor on the GPU, or a numpy int8 array (host)."""
        if hasattr(W, "data_ptr"):
            _check(_lib.ito_model_set_weights(self._h, layer, _ptr(W.contiguous()), 0, _stream(stream)))
        else:
            import numpy as np
            a = np.ascontiguousarray(W, dtype=np.int8)
            _check(_lib.ito_model_set_weights(self._h, layer, a.ctypes.data_as(ctypes.c_void_p), 1,
                                              _stream(stream)))

    def set_static_requant(self, layer, offset, mult, shift, stream=None):
        """numpy int32 [OC] arrays (host)."""
        import numpy as np
        arrs = [np.ascontiguousarray(a, dtype=np.int32) for a in (offset, mult, shift)]
        _check(_lib.ito_model_set_static_requant(self._h, layer, *[a.ctypes.data_as(ctypes.c_void_p) for a in arrs],
                                                 1, _stream(stream)))

    def tensor(self, name):
        """A torch view (on the GPU) of a named model tensor."""
        torch = _torch()
        ptr, eb, n = ctypes.c_void_p(), ctypes.c_int(), ctypes.c_int64()
        _check(_lib.ito_model_tensor(self._h, name.encode(), ctypes.byref(ptr), ctypes.byref(eb), ctypes.byref(n)))
        dt = getattr(torch, _DTYPES[eb.value])
        return _from_ptr(ptr.value, n.value, dt, eb.value)

    def stat_index(self, name) -> int:
        return _lib.ito_model_stat_index(self._h, name.encode())

    def num_stats(self) -> int:
        return _lib.ito_model_num_stats(self._h)

    def stats(self) -> dict:
        """All named scalars of the last step, read back to the host."""
        v = self.tensor("stats").cpu().tolist()
        out = {}
        for key in ("ymax", "ys", "dmax", "ds", "gmax", "gs", "ws", "nz", "ogmax", "ogs", "ows", "onz"):
            l = 0
            while True:
                i = self.stat_index("%s%d" % (key, l))
                if i < 0:
                    break
                val = v[i]
                out["%s%d" % (key, l)] = val & 0xFFFFFFFF if key in ("ymax", "dmax", "gmax", "nz", "ogmax", "onz") else val
                l += 1
        for key in ("pmax", "ps"):
            i = self.stat_index(key)
            out[key] = v[i] & 0xFFFFFFFF if key == "pmax" else v[i]
        return out

    def train_step(self, x, labels, stream=None):
        _check(_lib.ito_train_step(self._h, _ptr(x), _ptr(labels), _stream(stream)))

    def train_step_host(self, x_host, labels_host, stats_host=None, stream=None):
        """Host (pinned) torch tensors in, stats out; synchronises."""
        _check(_lib.ito_train_step_host(self._h, _ptr(x_host), _ptr(labels_host), _ptr(stats_host),
                                        _stream(stream)))

    def train_step_host_async(self, x_host, labels_host, stats_host=None, stream=None):
        """Host (pinned) torch tensors in, no wait: the next call's input copy overlaps this
        step; synchronise the stream before reading stats_host or reusing the buffers."""
        _check(_lib.ito_train_step_host_async(self._h, _ptr(x_host), _ptr(labels_host), _ptr(stats_host),
                                              _stream(stream)))

    def infer(self, x, logits, stream=None):
        _check(_lib.ito_infer(self._h, _ptr(x), _ptr(logits), _stream(stream)))

    def set_overlap(self, mode):
        """0: one stream; 1: backward bandwidth passes beside the contractions; 2: updates only"""
        _check(_lib.ito_model_set_overlap(self._h, int(mode)))

    def set_speculation(self, enable=True):
        """speculative requantisation in the contraction epilogues (exact; see include/ito.h)"""
        _check(_lib.ito_model_set_speculation(self._h, int(bool(enable))))

    def overlap(self) -> int:
        mode = ctypes.c_int()
        _check(_lib.ito_model_get_overlap(self._h, ctypes.byref(mode)))
        return mode.value

    def speculation(self) -> bool:
        on = ctypes.c_int()
        _check(_lib.ito_model_get_speculation(self._h, ctypes.byref(on)))
        return on.value == 1

    def use_graphs(self, enable=True):
        _check(_lib.ito_model_use_graphs(self._h, int(enable)))

    def profile(self, enable=True):
        _check(_lib.ito_model_profile(self._h, int(enable)))

    def profile_read(self):
        """{class: (ms, work, launches)} summed since the last read."""
        ms = (ctypes.c_double * 4)()
        work = (ctypes.c_double * 4)()
        n = (ctypes.c_int64 * 4)()
        _check(_lib.ito_model_profile_read(self._h, ms, work, n))
        return {name: (ms[i], work[i], n[i]) for i, name in enumerate(("gemm", "requant", "update", "other"))}

    def kernels_per_step(self) -> int:
        return _lib.ito_model_kernels_per_step(self._h)

    def save(self, path):
        _check(_lib.ito_model_save(self._h, path.encode()))

    def load(self, path):
        _check(_lib.ito_model_load(self._h, path.encode()))


# ------------------------------------------------------------------ DFP16

def _i32dev(v):
    torch = _torch()
    return torch.tensor([int(v)], dtype=torch.int32, device="cuda")


def _dfp_ws(B, IC, OC):
    torch = _torch()
    n = _lib.ito_dfp16_workspace_size(B, IC, OC)
    return torch.empty(n + 256, dtype=torch.uint8, device="cuda"), n


def _dfp_call(fn, a, ea, b, eb, B, IC, OC, p_shape, out_shape, stream):
    torch = _torch()
    p64 = torch.empty(p_shape, dtype=torch.int64, device="cuda")
    out = torch.empty(out_shape, dtype=torch.int16, device="cuda")
    mx = torch.zeros(1, dtype=torch.int64, device="cuda")
    e_out = torch.zeros(1, dtype=torch.int32, device="cuda")
    rs = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws, n = _dfp_ws(B, IC, OC)
    _check(fn(_ptr(a), _ptr(ea), _ptr(b), _ptr(eb), B, IC, OC, _aligned256(ws), n, _ptr(p64), _ptr(mx), _ptr(out),
              _ptr(e_out), _ptr(rs), _stream(stream)))
    return p64, mx, out, e_out, rs


def ito_dfp16_linear_fwd(x, exp_x, W, exp_w, stream=None):
    """exp_x / exp_w: device int32 [1] tensors -> (p64, max, y, exp_y, rs)"""
    B, IC = x.shape
    OC = W.shape[0]
    return _dfp_call(_lib.ito_dfp16_linear_fwd, x, exp_x, W, exp_w, B, IC, OC, (B, OC), (B, OC), stream)


def ito_dfp16_linear_bwd_delta(delta, exp_delta, W, exp_w, stream=None):
    B, OC = delta.shape
    IC = W.shape[1]
    return _dfp_call(_lib.ito_dfp16_linear_bwd_delta, delta, exp_delta, W, exp_w, B, IC, OC, (B, IC), (B, IC),
                     stream)


def ito_dfp16_linear_wgrad(delta, exp_delta, x, exp_x, stream=None):
    B, OC = delta.shape
    IC = x.shape[1]
    return _dfp_call(_lib.ito_dfp16_linear_wgrad, delta, exp_delta, x, exp_x, B, IC, OC, (OC, IC), (OC, IC), stream)


def ito_dfp16_update(W, g, exp_g, exp_w, eta, stream=None):
    """In place on W -> (k, nonzero) device int32 [1] each."""
    torch = _torch()
    k = torch.zeros(1, dtype=torch.int32, device="cuda")
    nz = torch.zeros(1, dtype=torch.int32, device="cuda")
    _check(_lib.ito_dfp16_update(_ptr(W), _ptr(g), _ptr(exp_g), W.numel(), exp_w, eta, _ptr(k), _ptr(nz),
                                 _stream(stream)))
    return k, nz


def ito_dfp16_update_bits(W, g, exp_g, exp_w, eta, bits, stream=None):
    """ito_dfp16_update saturating to +-(2^(bits-1) - 1); in place on W -> (k, nonzero)."""
    torch = _torch()
    k = torch.zeros(1, dtype=torch.int32, device="cuda")
    nz = torch.zeros(1, dtype=torch.int32, device="cuda")
    _check(_lib.ito_dfp16_update_bits(_ptr(W), _ptr(g), _ptr(exp_g), W.numel(), exp_w, eta, bits, _ptr(k),
                                      _ptr(nz), _stream(stream)))
    return k, nz


def ito_dfp_set_bits(W, bits_old, bits_new, stream=None):
    """Precision change of an int16 mantissa tensor, in place (the exponent changes by bits_old - bits_new)."""
    _check(_lib.ito_dfp_set_bits(_ptr(W), W.numel(), bits_old, bits_new, _stream(stream)))
    return W


def ito_bdfp16_from_float(f, block, stream=None):
    """float32 [rows][cols] -> (int16 mantissas, int8 exponents [rows][ceil(cols / block)])"""
    torch = _torch()
    rows, cols = f.shape
    nb = (cols + block - 1) // block
    m = torch.empty((rows, cols), dtype=torch.int16, device=f.device)
    e = torch.empty((rows, nb), dtype=torch.int8, device=f.device)
    _check(_lib.ito_bdfp16_from_float(_ptr(f), rows, cols, block, _ptr(m), _ptr(e), _stream(stream)))
    return m, e


def ito_bdfp16_to_float(m, e, block, stream=None):
    torch = _torch()
    rows, cols = m.shape
    f = torch.empty((rows, cols), dtype=torch.float32, device=m.device)
    _check(_lib.ito_bdfp16_to_float(_ptr(m), _ptr(e), rows, cols, block, _ptr(f), _stream(stream)))
    return f


def ito_bdfp16_linear_fwd_f32(x, ex, W, ew, block, stream=None):
    """Blocked-DFP x [B][IC], W [OC][IC] (int8 exponents per block of IC) -> float32 [B][OC]"""
    torch = _torch()
    B, IC = x.shape
    OC = W.shape[0]
    y = torch.empty((B, OC), dtype=torch.float32, device=x.device)
    ws, n = _dfp_ws(B, IC, OC)
    _check(_lib.ito_bdfp16_linear_fwd_f32(_ptr(x), _ptr(ex), _ptr(W), _ptr(ew), B, IC, OC, block, _aligned256(ws), n,
                                          _ptr(y), _stream(stream)))
    return y


def ito_dfp16_from_float(f, stream=None):
    """float32 device tensor -> (int16 mantissas, device int32 [1] exponent)."""
    torch = _torch()
    mant = torch.empty(f.shape, dtype=torch.int16, device="cuda")
    e = torch.zeros(1, dtype=torch.int32, device="cuda")
    bits = torch.zeros(1, dtype=torch.int32, device="cuda")
    _check(_lib.ito_dfp16_from_float(_ptr(f), f.numel(), _ptr(bits), _ptr(mant), _ptr(e), _stream(stream)))
    return mant, e


def ito_dfp16_to_float(mant, exp, stream=None):
    torch = _torch()
    f = torch.empty(mant.shape, dtype=torch.float32, device="cuda")
    _check(_lib.ito_dfp16_to_float(_ptr(mant), _ptr(exp), mant.numel(), _ptr(f), _stream(stream)))
    return f


def ito_dfp16_linear_fwd_f32(x, exp_x, W, exp_w, stream=None):
    """-> (p64 int64 [B][OC], y float32 [B][OC])"""
    torch = _torch()
    B, IC = x.shape
    OC = W.shape[0]
    p64 = torch.empty((B, OC), dtype=torch.int64, device="cuda")
    y = torch.empty((B, OC), dtype=torch.float32, device="cuda")
    mx = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws, n = _dfp_ws(B, IC, OC)
    _check(_lib.ito_dfp16_linear_fwd_f32(_ptr(x), _ptr(exp_x), _ptr(W), _ptr(exp_w), B, IC, OC, _aligned256(ws), n,
                                         _ptr(p64), _ptr(mx), _ptr(y), _stream(stream)))
    return p64, y


def ito_dfp16_linear_fwd_f32_chained(x, exp_x, W, exp_w, chain, input_shift=1, stream=None):
    """-> y float32 [B][OC] (FP32 partial accumulation over INT32 chains of `chain` terms)"""
    torch = _torch()
    B, IC = x.shape
    OC = W.shape[0]
    y = torch.empty((B, OC), dtype=torch.float32, device="cuda")
    ws, n = _dfp_ws(B, IC, OC)
    _check(_lib.ito_dfp16_linear_fwd_f32_chained(_ptr(x), _ptr(exp_x), _ptr(W), _ptr(exp_w), B, IC, OC, int(chain),
                                                 int(input_shift), _aligned256(ws), n, _ptr(y), _stream(stream)))
    return y


class Dfp16Model:
    """An ito_dfp16_model: DFP16 Linear layers trained with integer SGD."""

    def __init__(self, dims, batch, exp_w, eta):
        arr = (ctypes.c_int32 * len(dims))(*dims)
        h = ctypes.c_void_p()
        _check(_lib.ito_dfp16_model_create(arr, len(dims) - 1, batch, exp_w, eta, ctypes.byref(h)))
        self._h = h
        self.batch = batch
        self.n_layers = len(dims) - 1

    def close(self):
        if getattr(self, "_h", None):
            _lib.ito_dfp16_model_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_weights(self, layer, W, stream=None):
        import numpy as np
        a = np.ascontiguousarray(W, dtype=np.int16)
        _check(_lib.ito_dfp16_model_set_weights(self._h, layer, a.ctypes.data_as(ctypes.c_void_p), 1,
                                                _stream(stream)))

    def tensor(self, name):
        ptr, eb, n = ctypes.c_void_p(), ctypes.c_int(), ctypes.c_int64()
        _check(_lib.ito_dfp16_model_tensor(self._h, name.encode(), ctypes.byref(ptr), ctypes.byref(eb),
                                           ctypes.byref(n)))
        return _from_ptr(ptr.value, n.value, None, eb.value)

    def stats(self) -> dict:
        n = _lib.ito_dfp16_model_num_stats(self._h)
        buf = (ctypes.c_int64 * n)()
        _check(_lib.ito_dfp16_model_read_stats(self._h, buf, n))
        out = {}
        for l in range(self.n_layers):
            for key in ("ey", "ee", "rs", "rsd", "rsg", "eg", "k", "nz", "pmax", "pdmax", "pgmax", "gabs"):
                i = _lib.ito_dfp16_model_stat_index(self._h, ("%s%d" % (key, l)).encode())
                out["%s%d" % (key, l)] = buf[i]
        return out

    def train_step(self, x, exp_x, stream=None):
        _check(_lib.ito_dfp16_train_step(self._h, _ptr(x), int(exp_x), _stream(stream)))

    def train_step_host_async(self, x_host, exp_x, stats_host=None, stream=None):
        """Host (pinned) int16 mantissas in, no wait: the next call's input copy overlaps this
        step; stats_host (int64, num_stats()) holds the step's statistics once the stream
        has passed it."""
        _check(_lib.ito_dfp16_train_step_host_async(self._h, _ptr(x_host), int(exp_x), _ptr(stats_host),
                                                    _stream(stream)))

    def num_stats(self) -> int:
        return _lib.ito_dfp16_model_num_stats(self._h)

    def profile(self, enable=True):
        _check(_lib.ito_dfp16_model_profile(self._h, int(enable)))

    def profile_read(self):
        """{class: (ms, work, launches)} summed since the last read."""
        ms = (ctypes.c_double * 4)()
        work = (ctypes.c_double * 4)()
        n = (ctypes.c_int64 * 4)()
        _check(_lib.ito_dfp16_model_profile_read(self._h, ms, work, n))
        return {name: (ms[i], work[i], n[i]) for i, name in enumerate(("gemm", "down", "update", "other"))}

    def kernels_per_step(self) -> int:
        return _lib.ito_dfp16_model_kernels_per_step(self._h)

    def precision(self, layer):
        """-> (bits, exp_w) of a layer's weights"""
        b, e = ctypes.c_int32(), ctypes.c_int32()
        _check(_lib.ito_dfp16_model_get_precision(self._h, layer, ctypes.byref(b), ctypes.byref(e)))
        return b.value, e.value

    def set_precision(self, layer, bits, stream=None):
        _check(_lib.ito_dfp16_model_set_precision(self._h, layer, bits, _stream(stream)))

    def apt_enable(self, k_init, k_min, k_max, t_min, t_max, eval_every=1, stream=None):
        p = AptParams(k_init, k_min, k_max, eval_every, float(t_min), float(t_max))
        _check(_lib.ito_dfp16_model_apt_enable(self._h, ctypes.byref(p), _stream(stream)))

    def apt_epoch_end(self, stream=None):
        """Algorithm 1 at the end of an epoch -> (mean Gavg per layer, new bits per layer)"""
        g = (ctypes.c_double * self.n_layers)()
        b = (ctypes.c_int32 * self.n_layers)()
        _check(_lib.ito_dfp16_model_apt_epoch_end(self._h, g, b, _stream(stream)))
        return list(g), list(b)


class _CudaArray:
    """Minimal __cuda_array_interface__ holder to view library-owned memory."""

    def __init__(self, ptr, n, typestr):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False), "version": 3}


def _from_ptr(ptr, n, dtype, eb):
    torch = _torch()
    typestr = {1: "|i1", 2: "<i2", 4: "<i4", 8: "<i8"}[eb]
    return torch.as_tensor(_CudaArray(ptr, n, typestr), device="cuda")
