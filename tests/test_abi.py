"""The C ABI: the library loads on a machine without a GPU, exports every
entry point include/ito.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib_path():
    # the build script is loaded by path: importing the package would bind the library first
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "ito_build", os.path.join(ROOT, "integer_only_nn_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


def declared_entry_points():
    text = open(os.path.join(ROOT, "include", "ito.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ito_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for n in ("ito_linear_fwd", "ito_linear_bwd_delta", "ito_linear_wgrad", "ito_niti_update",
              "ito_top_error", "ito_train_step", "ito_model_create"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(_lib_path())
    missing = [n for n in declared_entry_points() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    _lib_path()
    import integer_only_nn_gb300 as ito
    assert set(declared_entry_points()) <= set(ito.EXPORTED)


def test_host_side_argument_errors():
    _lib_path()
    import integer_only_nn_gb300 as ito
    L = ito._lib
    p = ito.params()
    assert L.ito_version() == 1
    assert L.ito_linear_workspace_size(0, 4, 4) == 0
    assert L.ito_linear_workspace_size(8, 4, 4) > 0
    # NULL tensors are rejected before anything is enqueued
    assert L.ito_linear_fwd(None, None, 4, 4, 4, 1, p, None, 0, None, None, None, None, None) == ito.ITO_ERR_ARG
    dummy = ctypes.c_void_p(256)
    assert L.ito_linear_fwd(dummy, dummy, 0, 4, 4, 1, p, dummy, 1 << 20, dummy, dummy, None, dummy,
                            None) == ito.ITO_ERR_SHAPE
    # misaligned workspace
    assert L.ito_linear_fwd(dummy, dummy, 4, 4, 4, 1, p, ctypes.c_void_p(257), 1 << 20, dummy, dummy, None,
                            dummy, None) == ito.ITO_ERR_ARG
    assert L.ito_niti_update(dummy, dummy, 0, dummy, p, None, None, None, None) == ito.ITO_ERR_SHAPE
    assert L.ito_top_error(None, dummy, 1, 1, 64, dummy, None) == ito.ITO_ERR_ARG
    h = ctypes.c_void_p()
    arr = (ito.LayerDesc * 1)(ito.LayerDesc(ito.ITO_LAYER_LINEAR, 4, 4, 0, 0, 0))
    assert L.ito_model_create(arr, 1, 8, ito.NitiParams(0, 2), 64, ctypes.byref(h)) == ito.ITO_ERR_ARG
    assert L.ito_model_create(arr, 0, 8, p, 64, ctypes.byref(h)) == ito.ITO_ERR_ARG
    assert L.ito_model_create(arr, 1, 0, p, 64, ctypes.byref(h)) == ito.ITO_ERR_SHAPE
    assert L.ito_model_stat_index(None, b"ys0") == -1
    assert L.ito_model_destroy(None) == ito.ITO_OK
    assert b"" != L.ito_last_error_string()


def test_host_side_argument_errors_new_entry_points():
    """Conv/pooling, DFP precision and Blocked-DFP calls reject bad arguments on
    the host, before anything is enqueued (no GPU needed)."""
    _lib_path()
    import integer_only_nn_gb300 as ito
    L = ito._lib
    p = ito.params()
    dummy = ctypes.c_void_p(256)
    # contraction longer than 2^20
    assert L.ito_linear_fwd(dummy, dummy, 4, (1 << 20) + 1, 4, 1, p, dummy, 1 << 30, dummy, dummy, None, dummy,
                            None) == ito.ITO_ERR_SHAPE
    # conv: workspace size 0 for invalid shapes, stride outside 1..4, NULL tensors
    assert L.ito_conv2d_workspace_size(1, 8, 8, 3, 16, 0) == 0
    assert L.ito_conv2d_workspace_size(1, 8, 8, 3, 16, 5) == 0
    assert L.ito_conv2d_workspace_size(1, 8, 8, 3, 16, 2) > 0
    assert L.ito_conv2d_fwd(None, dummy, 1, 8, 8, 3, 16, 1, 1, p, dummy, 1 << 20, dummy, dummy, None, dummy,
                            None) == ito.ITO_ERR_ARG
    assert L.ito_conv2d_fwd(dummy, dummy, 1, 8, 8, 3, 16, 9, 1, p, dummy, 1 << 20, dummy, dummy, None, dummy,
                            None) == ito.ITO_ERR_SHAPE
    assert L.ito_conv2d_wgrad(dummy, dummy, 0, 8, 8, 3, 16, 1, dummy, 1 << 20, dummy, dummy,
                              None) == ito.ITO_ERR_SHAPE
    assert L.ito_gap_fwd(dummy, 0, 4, 4, p, dummy, dummy, None, dummy, None) == ito.ITO_ERR_SHAPE
    assert L.ito_gap_bwd(None, dummy, 1, 4, 4, dummy, None) == ito.ITO_ERR_ARG
    # DFP precision: bits outside 2..16
    assert L.ito_dfp_set_bits(dummy, 16, 1, 8, None) == ito.ITO_ERR_ARG
    assert L.ito_dfp_set_bits(dummy, 16, 8, 17, None) == ito.ITO_ERR_ARG
    assert L.ito_dfp16_update_bits(dummy, dummy, dummy, 16, -10, 8, 17, None, None, None) == ito.ITO_ERR_ARG
    assert L.ito_dfp16_model_set_precision(None, 0, 8, None) == ito.ITO_ERR_ARG
    assert L.ito_dfp16_model_apt_epoch_end(None, None, None, None) == ito.ITO_ERR_ARG
    # Blocked-DFP
    assert L.ito_bdfp16_from_float(dummy, 4, 4, 0, dummy, dummy, None) == ito.ITO_ERR_SHAPE
    assert L.ito_bdfp16_to_float(None, dummy, 4, 4, 2, dummy, None) == ito.ITO_ERR_ARG
    big = ctypes.c_size_t(1 << 30)
    for chain, shift in ((100, 1), (32, 1), (1024, 0), (64, 2)):
        assert L.ito_dfp16_linear_fwd_f32_chained(dummy, dummy, dummy, dummy, 4, 64, 4, chain, shift, dummy, big,
                                                  dummy, None) == ito.ITO_ERR_ARG
    assert L.ito_dfp16_linear_fwd_f32_chained(dummy, None, dummy, dummy, 4, 64, 4, 64, 1, dummy, big, dummy,
                                              None) == ito.ITO_ERR_ARG
    assert L.ito_dfp16_linear_fwd_f32_chained(dummy, dummy, dummy, dummy, 4, 64, 4, 64, 1, None, 0, dummy,
                                              None) == ito.ITO_ERR_ARG
    assert L.ito_bdfp16_linear_fwd_f32(dummy, dummy, dummy, dummy, 4, 4, 4, 64, None, 0, dummy,
                                       None) == ito.ITO_ERR_ARG


def test_host_side_argument_errors_model_controls():
    """The model's stream, speculation and pipelining controls and the DFP16
    model's profiling reject NULL arguments on the host (no GPU needed)."""
    _lib_path()
    import integer_only_nn_gb300 as ito
    L = ito._lib
    dummy = ctypes.c_void_p(256)
    flag = ctypes.c_int(-7)
    assert L.ito_model_get_speculation(None, ctypes.byref(flag)) == ito.ITO_ERR_ARG
    assert L.ito_model_get_overlap(None, ctypes.byref(flag)) == ito.ITO_ERR_ARG
    assert flag.value == -7                       # nothing written on error
    assert L.ito_model_set_speculation(None, 1) == ito.ITO_ERR_ARG
    assert L.ito_model_set_overlap(None, 0) == ito.ITO_ERR_ARG
    assert L.ito_train_step_host_async(None, dummy, dummy, None, None) == ito.ITO_ERR_ARG
    assert L.ito_train_step_host(None, dummy, dummy, None, None) == ito.ITO_ERR_ARG
    assert L.ito_dfp16_model_profile(None, 1) == ito.ITO_ERR_ARG
    ms = (ctypes.c_double * 4)()
    n = (ctypes.c_int64 * 4)()
    assert L.ito_dfp16_model_profile_read(None, ms, ms, n) == ito.ITO_ERR_ARG
    assert L.ito_dfp16_model_kernels_per_step(None) == 0
    assert L.ito_model_kernels_per_step(None) == 0


def test_model_options_struct_matches_header():
    """The binding's ModelOptions has the header's fields in order (int32 each)."""
    import re
    text = open(os.path.join(ROOT, "include", "ito.h")).read()
    body = re.search(r"typedef struct ito_model_options \{(.*?)\} ito_model_options;", text, re.S).group(1)
    fields = re.findall(r"int32_t\s+(\w+);", body)
    _lib_path()
    import integer_only_nn_gb300 as ito
    assert [f for f, _ in ito.ModelOptions._fields_] == fields
    assert ctypes.sizeof(ito.ModelOptions) == 4 * len(fields)


def test_host_side_argument_errors_dfp16_pipelined_step():
    """The pipelined DFP16 host step rejects a NULL model or input on the host."""
    _lib_path()
    import integer_only_nn_gb300 as ito
    L = ito._lib
    dummy = ctypes.c_void_p(256)
    assert L.ito_dfp16_train_step_host_async(None, dummy, -12, None, None) == ito.ITO_ERR_ARG
    assert L.ito_dfp16_model_num_stats(None) == 0


def test_header_compiles_as_c_and_cpp(tmp_path):
    """include/ito.h is a C header (plain types, no C++ in the declarations): it compiles as
    C99 with warnings on and as C++17."""
    import shutil
    import subprocess
    if not shutil.which("gcc") or not shutil.which("g++"):
        pytest.skip("no host C compiler")
    inc = os.path.join(ROOT, "include")
    src = tmp_path / "use.c"
    src.write_text('#include "ito.h"\nint main(void) { return ito_get_error() == 0 ? 0 : 1; }\n')
    for cmd in (["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", inc, "-c", str(src), "-o",
                 str(tmp_path / "c.o")],
                ["g++", "-std=c++17", "-Wall", "-Werror", "-x", "c++", "-I", inc, "-c", str(src), "-o",
                 str(tmp_path / "cpp.o")]):
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
