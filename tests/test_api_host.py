"""Host-only checks of the C ABI (no GPU, no kernel launch).

The library must load, export every function include/mxq.h declares, and
reject bad arguments with the documented status codes before it touches
the GPU (argument validation is host code that runs before any launch).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from nvfp4_quantizers_gb300 import build as B
    B.build()
    import nvfp4_quantizers_gb300 as q
    lib = q.lib()
    lib.mxq_set_fault_inject(0)
    yield lib
    lib.mxq_set_fault_inject(0)


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "mxq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_0-9]+)\s*\(", src)) -
                  {"if", "sizeof", "defined"})


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert "mxfp8_quantize_rowcol" in names and len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    import nvfp4_quantizers_gb300 as q
    for s in range(9):
        assert q.status_string(s).startswith("MXQ")
    assert L.mxq_version() >= 100


def test_scale_bytes(L):
    import nvfp4_quantizers_gb300 as q
    assert q.scale_bytes(256, 8, "swizzled") == 2048
    assert q.scale_bytes(300, 5, "swizzled") == 384 * 8
    assert q.scale_bytes(300, 5, "linear") == 1500
    assert L.mxq_scale_bytes(1, 1, 7) == -1


FAKE = 0x10000          # aligned fake device addresses: never dereferenced


def test_mxfp8_argument_errors(L):
    f = L.mxfp8_quantize_rowcol
    import nvfp4_quantizers_gb300 as q
    assert f(FAKE, 64, 64, 64, FAKE, FAKE, FAKE, FAKE, 9, None) == q.MXQ_ERR_LAYOUT
    assert f(FAKE, 64, 64, 64, None, None, None, None, 1, None) == q.MXQ_ERR_NULL
    assert f(FAKE, 64, 64, 64, FAKE, None, None, None, 1, None) == q.MXQ_ERR_NULL
    assert f(None, 64, 64, 64, FAKE, FAKE, None, None, 1, None) == q.MXQ_ERR_NULL
    assert f(FAKE, 64, 48, 48, FAKE, FAKE, None, None, 1, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, 48, 64, 64, FAKE, FAKE, FAKE, FAKE, 1, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, -1, 64, 64, FAKE, FAKE, None, None, 1, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, 64, 64, 32, FAKE, FAKE, None, None, 1, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE + 2, 64, 64, 64, FAKE, FAKE, None, None, 1, None) == q.MXQ_ERR_ALIGN
    assert f(FAKE, 64, 64, 68, FAKE, FAKE, None, None, 1, None) == q.MXQ_ERR_ALIGN
    assert f(FAKE, 64, 64, 64, FAKE + 8, FAKE, None, None, 1, None) == q.MXQ_ERR_ALIGN
    # empty input: nothing to do, nothing launched
    assert f(FAKE, 0, 64, 64, FAKE, FAKE, FAKE, FAKE, 1, None) == q.MXQ_OK
    assert f(None, 64, 0, 0, FAKE, FAKE, None, None, 0, None) == q.MXQ_OK


def test_nvfp4_argument_errors(L):
    import nvfp4_quantizers_gb300 as q
    f = L.nvfp4_quantize_per_token
    assert f(FAKE, 4, 40, 40, FAKE, FAKE, FAKE, 1, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, 4, 32, 32, None, FAKE, FAKE, 1, None) == q.MXQ_ERR_NULL
    assert f(FAKE, 4, 32, 36, FAKE, FAKE, FAKE, 1, None) == q.MXQ_ERR_ALIGN
    assert f(FAKE, 4, 32, 32, FAKE, FAKE, FAKE + 4, 1, None) == q.MXQ_ERR_ALIGN
    assert f(FAKE, 4, 32, 32, FAKE, FAKE, FAKE, 3, None) == q.MXQ_ERR_LAYOUT
    assert f(None, 0, 32, 32, None, None, None, 1, None) == q.MXQ_OK

    g = L.nvfp4_quantize_weight_shared
    ptrs = (ctypes.c_void_p * 2)(FAKE, FAKE)
    rows = (ctypes.c_int64 * 2)(64, 64)
    P = ctypes.cast(ptrs, ctypes.c_void_p)
    R = ctypes.cast(rows, ctypes.c_void_p)
    assert g(1, 5, P, R, 64, FAKE, FAKE, FAKE, None, 1, FAKE, 256, None) == q.MXQ_ERR_ARG
    assert g(1, 2, P, R, 64, FAKE, FAKE, FAKE, None, 1, None, 0, None) == q.MXQ_ERR_WORKSPACE
    assert g(1, 2, P, R, 64, FAKE, FAKE, FAKE, None, 1, FAKE, 0, None) == q.MXQ_ERR_WORKSPACE
    assert g(1, 2, P, R, 40, FAKE, FAKE, FAKE, None, 1, FAKE, 256, None) == q.MXQ_ERR_SHAPE
    assert g(1, 2, None, R, 64, FAKE, FAKE, FAKE, None, 1, FAKE, 256, None) == q.MXQ_ERR_NULL
    # 256-byte header + an amax word and a progress counter per group
    assert L.nvfp4_quantize_weight_shared_workspace_size(128) == 1280
    assert L.nvfp4_quantize_weight_shared_workspace_size(0) == 0


def test_dequant_argument_errors(L):
    import nvfp4_quantizers_gb300 as q
    assert L.dequantize_mxfp8(FAKE, FAKE, 4, 48, 1, FAKE, None) == q.MXQ_ERR_SHAPE
    assert L.dequantize_mxfp8(None, FAKE, 4, 64, 1, FAKE, None) == q.MXQ_ERR_NULL
    assert L.dequantize_mxfp8(FAKE, FAKE, 4, 64, 1, FAKE + 2, None) == q.MXQ_ERR_ALIGN
    assert L.dequantize_nvfp4(FAKE, FAKE, FAKE, 5, 1, 4, 64, 1, FAKE, None) == q.MXQ_ERR_LAYOUT
    assert L.dequantize_nvfp4(FAKE, FAKE, FAKE, 0, 1, 4, 24, 1, FAKE, None) == q.MXQ_ERR_SHAPE
    assert L.dequantize_nvfp4(FAKE, FAKE, None, 0, 1, 4, 64, 1, FAKE, None) == q.MXQ_ERR_NULL
    assert L.dequantize_nvfp4(FAKE, FAKE, FAKE, 0, 0, 4, 64, 1, FAKE, None) == q.MXQ_OK


def test_moe_entry_point_argument_errors(L):
    import nvfp4_quantizers_gb300 as q
    g = L.nvfp4_quantize_per_token_gather
    assert g(FAKE, 10, 64, 64, None, 4, FAKE, FAKE, FAKE, 1, None) == q.MXQ_ERR_NULL
    assert g(FAKE, 10, 40, 40, FAKE, 4, FAKE, FAKE, FAKE, 1, None) == q.MXQ_ERR_SHAPE
    assert g(FAKE, 10, 64, 64, FAKE + 2, 4, FAKE, FAKE, FAKE, 1, None) == q.MXQ_ERR_ALIGN
    assert g(FAKE, 10, 64, 64, FAKE, 4, FAKE, FAKE, FAKE, 7, None) == q.MXQ_ERR_LAYOUT
    assert g(FAKE, 10, 64, 64, FAKE, 0, None, None, None, 1, None) == q.MXQ_OK
    f = L.mxq_moe_gate_up_swiglu_nvfp4
    offs = (ctypes.c_int64 * 3)(0, 128, 256)
    O = ctypes.cast(offs, ctypes.c_void_p)
    assert f(FAKE, FAKE, FAKE, O, 2, FAKE, FAKE, FAKE, 192, 256, FAKE, 192, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, O, 2, FAKE, FAKE, FAKE, 128, 128, FAKE, 128, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, O, 2, FAKE, FAKE, FAKE, 128, 256, None, 128, None) == q.MXQ_ERR_NULL
    assert f(FAKE, FAKE, FAKE, O, 2, FAKE, FAKE, FAKE, 128, 256, FAKE, 132, None) == q.MXQ_ERR_ALIGN
    bad = (ctypes.c_int64 * 3)(0, 100, 256)
    assert f(FAKE, FAKE, FAKE, ctypes.cast(bad, ctypes.c_void_p), 2, FAKE, FAKE,
             FAKE, 128, 256, FAKE, 128, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, FAKE, FAKE, O, 0, FAKE, FAKE, FAKE, 128, 256, FAKE, 128, None) == q.MXQ_OK


def test_rht_sr_argument_errors(L):
    import nvfp4_quantizers_gb300 as q
    f = L.nvfp4_quantize_per_token_rht_sr
    assert f(FAKE, 8, 64, 64, 1, 4, FAKE, FAKE, FAKE, 1, None) == q.MXQ_ERR_ARG
    assert f(FAKE, 8, 64, 64, 1, -1, FAKE, FAKE, FAKE, 1, None) == q.MXQ_ERR_ARG
    assert f(FAKE, 8, 40, 40, 1, 3, FAKE, FAKE, FAKE, 1, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, 8, 64, 32, 1, 3, FAKE, FAKE, FAKE, 1, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, 8, 64, 64, 1, 3, FAKE, None, FAKE, 1, None) == q.MXQ_ERR_NULL
    assert f(FAKE, 8, 64, 68, 1, 3, FAKE, FAKE, FAKE, 1, None) == q.MXQ_ERR_ALIGN
    assert f(FAKE, 8, 64, 64, 1, 3, FAKE, FAKE, FAKE, 5, None) == q.MXQ_ERR_LAYOUT
    assert f(FAKE, 0, 64, 64, 1, 3, None, None, None, 1, None) == q.MXQ_OK


def test_fp8_block_argument_errors(L):
    import nvfp4_quantizers_gb300 as q
    f = L.fp8_block_quantize
    assert f(FAKE, 64, 256, 256, 2, FAKE, FAKE, None) == q.MXQ_ERR_ARG
    assert f(FAKE, 64, 200, 200, 1, FAKE, FAKE, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, 100, 256, 256, 128, FAKE, FAKE, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, 64, 256, 128, 1, FAKE, FAKE, None) == q.MXQ_ERR_SHAPE
    assert f(None, 64, 256, 256, 1, FAKE, FAKE, None) == q.MXQ_ERR_NULL
    assert f(FAKE + 2, 64, 256, 256, 1, FAKE, FAKE, None) == q.MXQ_ERR_ALIGN
    assert f(FAKE, 64, 256, 260, 1, FAKE, FAKE, None) == q.MXQ_ERR_ALIGN
    assert f(FAKE, 0, 256, 256, 1, None, None, None) == q.MXQ_OK
    d = L.fp8_block_dequantize
    assert d(FAKE, FAKE, 64, 256, 3, FAKE, None) == q.MXQ_ERR_ARG
    assert d(FAKE, FAKE, 64, 192, 1, FAKE, None) == q.MXQ_ERR_SHAPE
    assert d(FAKE, FAKE, 64, 256, 128, FAKE, None) == q.MXQ_ERR_SHAPE
    assert d(FAKE, None, 64, 256, 1, FAKE, None) == q.MXQ_ERR_NULL
    assert d(FAKE, FAKE, 64, 256, 1, FAKE + 8, None) == q.MXQ_ERR_ALIGN
    t = L.fp8_block_requantize_transpose
    assert t(FAKE, FAKE, 64, 256, FAKE, FAKE, None) == q.MXQ_ERR_SHAPE
    assert t(FAKE, FAKE, 128, 200, FAKE, FAKE, None) == q.MXQ_ERR_SHAPE
    assert t(FAKE, FAKE, 128, 256, None, FAKE, None) == q.MXQ_ERR_NULL
    assert t(FAKE, FAKE, 128, 256, FAKE, FAKE + 4, None) == q.MXQ_ERR_ALIGN
    assert t(FAKE, FAKE, 0, 256, None, None, None) == q.MXQ_OK


def test_bf16_mxfp8_gemm_argument_errors(L):
    import nvfp4_quantizers_gb300 as q
    f = L.mxq_gemm_bf16_mxfp8
    assert f(FAKE, 128, FAKE, FAKE, 100, 128, 128, FAKE, 128, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, 128, FAKE, FAKE, 128, 128, 96, FAKE, 128, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, 64, FAKE, FAKE, 128, 128, 128, FAKE, 128, None) == q.MXQ_ERR_SHAPE
    assert f(FAKE, 128, None, FAKE, 128, 128, 128, FAKE, 128, None) == q.MXQ_ERR_NULL
    assert f(FAKE, 132, FAKE, FAKE, 128, 128, 128, FAKE, 128, None) == q.MXQ_ERR_ALIGN
    assert f(FAKE + 8, 128, FAKE, FAKE, 128, 128, 128, FAKE, 128, None) == q.MXQ_ERR_ALIGN
    assert f(FAKE, 128, FAKE, FAKE, 0, 128, 128, FAKE, 128, None) == q.MXQ_OK


def test_fault_injection_returns_errors_without_launching(L):
    import nvfp4_quantizers_gb300 as q
    try:
        L.mxq_set_fault_inject(2)
        assert L.mxfp8_quantize_rowcol(FAKE, 64, 64, 64, FAKE, FAKE, None,
                                       None, 1, None) == q.MXQ_ERR_ARG
        assert L.dequantize_mxfp8(FAKE, FAKE, 4, 64, 1, FAKE, None) == q.MXQ_ERR_ARG
        L.mxq_set_fault_inject(1)
        # valid arguments, but the launch is reported failed and not issued
        assert L.mxfp8_quantize_rowcol(FAKE, 64, 64, 64, FAKE, FAKE, None,
                                       None, 1, None) == q.MXQ_ERR_CUDA
        assert L.nvfp4_quantize_per_token(FAKE, 4, 32, 32, FAKE, FAKE, FAKE,
                                          1, None) == q.MXQ_ERR_CUDA
        assert L.dequantize_nvfp4(FAKE, FAKE, FAKE, 0, 1, 4, 64, 1, FAKE,
                                  None) == q.MXQ_ERR_CUDA
    finally:
        L.mxq_set_fault_inject(0)


def test_noalloc_entry_point_honours_fault_injection(L):
    import nvfp4_quantizers_gb300 as q
    f = L.nvfp4_quantize_weight_shared_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_void_p]
    ptrs = (ctypes.c_void_p * 2)(FAKE, FAKE)
    rows = (ctypes.c_int64 * 2)(16, 16)
    args = (1, 2, ctypes.cast(ptrs, ctypes.c_void_p),
            ctypes.cast(rows, ctypes.c_void_p), 64, FAKE, FAKE, FAKE, None, 1,
            None)
    try:
        L.mxq_set_fault_inject(2)
        assert f(*args) == q.MXQ_ERR_ARG
        L.mxq_set_fault_inject(1)
        # valid arguments: reported as a failed launch, nothing issued
        assert f(*args) == q.MXQ_ERR_CUDA
    finally:
        L.mxq_set_fault_inject(0)
    # argument errors come before any device call
    assert f(4097, 2, ctypes.cast(ptrs, ctypes.c_void_p),
             ctypes.cast(rows, ctypes.c_void_p), 64, FAKE, FAKE, FAKE, None,
             1, None) == q.MXQ_ERR_SHAPE
    assert f(1, 2, ctypes.cast(ptrs, ctypes.c_void_p),
             ctypes.cast(rows, ctypes.c_void_p), 64, FAKE + 8, FAKE, FAKE,
             None, 1, None) == q.MXQ_ERR_ALIGN


def test_python_binding_raises_on_error(L):
    import nvfp4_quantizers_gb300 as q
    with pytest.raises(q.MxqError) as ei:
        q._lib._check(q.MXQ_ERR_SHAPE, "op")
    assert ei.value.status == q.MXQ_ERR_SHAPE
    with pytest.raises(ValueError):
        q.scale_bytes(4, 4, "bogus")


def test_product_does_not_import_oracle():
    """The product package shares no code with the oracle."""
    pkg = os.path.join(ROOT, "nvfp4_quantizers_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text
                assert "mxq_oracle" not in text and "liboracle" not in text
