"""nvfp4_quantizers_gb300 -- GB300 (sm_103a) MXFP8 / NVFP4 quantizer library.

The compute lives in ``libmxq.so`` (CUDA kernels behind the C ABI declared
in ``include/mxq.h``); this package is its thin Python binding.  Importing
the package does not load the library; the first call does, and raises if
it has not been built (``nvfp4_quantizers_gb300.build.build()``).
"""
from ._lib import (  # noqa: F401
    MXQ_ERR_ALIGN, MXQ_ERR_ARG, MXQ_ERR_CUDA, MXQ_ERR_LAYOUT, MXQ_ERR_NULL,
    MXQ_ERR_SHAPE, MXQ_ERR_TIMEOUT, MXQ_ERR_WORKSPACE, MXQ_OK, SCALE_LINEAR,
    SCALE_SWIZZLED, S_PER_BATCH, S_PER_ROW, Fp8BlockQuantized,
    Mxfp8Quantized, MxqError, Nvfp4Quantized, dequantize_mxfp8,
    dequantize_nvfp4, fp8_block_dequantize, fp8_block_quantize,
    fp8_block_requantize_transpose, gemm_bf16_mxfp8, gemm_mxfp8,
    gemm_nvfp4_grouped, gemm_nvfp4_grouped_gather, get_last_error, lib,
    moe_gate_up_swiglu, moe_gate_up_swiglu_gather,
    mxfp8_quantize_rowcol, nvfp4_quantize_per_token,
    NVFP4_RHT, NVFP4_SR, nvfp4_quantize_per_token_gather,
    nvfp4_quantize_per_token_rht_sr, nvfp4_quantize_weight_shared,
    scale_bytes, selftest_wait_timeout, set_fault_inject, status_string)

__version__ = "0.1.0"
