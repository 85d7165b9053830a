"""CPU oracle for the MXFP8 / NVFP4 quantizer contract.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.
The product (``nvfp4_quantizers_gb300``) never imports it, and this package
never imports the product: the two share no code.

The arithmetic lives in ``mxq_oracle.c`` (plain scalar C, tables built by
enumerating bit patterns, rounding by brute-force nearest search).  This
module only compiles it, loads it with ctypes and marshals numpy arrays.
The GEMM oracle is a float64 numpy matmul over exactly dequantized operands.

Every bf16 tensor is passed as a numpy ``uint16`` array of bit patterns.
Sources are cited per function as (page title, section).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_C = ctypes
_p = ctypes.c_void_p
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, -O2, strict
    IEEE binary32/binary64: no fast math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.oracle_decode_bf16.restype = ctypes.c_double
            L.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
            L.oracle_decode_e4m3.restype = ctypes.c_double
            L.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
            L.oracle_decode_e2m1.restype = ctypes.c_double
            L.oracle_decode_e2m1.argtypes = [ctypes.c_uint8]
            L.oracle_decode_e8m0.restype = ctypes.c_double
            L.oracle_decode_e8m0.argtypes = [ctypes.c_uint8]
            L.oracle_rne_e4m3.restype = ctypes.c_uint8
            L.oracle_rne_e4m3.argtypes = [ctypes.c_double]
            L.oracle_rne_e2m1.restype = ctypes.c_uint8
            L.oracle_rne_e2m1.argtypes = [ctypes.c_double]
            L.oracle_rne_bf16.restype = ctypes.c_uint16
            L.oracle_rne_bf16.argtypes = [ctypes.c_float]
            L.oracle_mxfp8_scale_exponent.restype = ctypes.c_int
            L.oracle_mxfp8_scale_exponent.argtypes = [ctypes.c_double]
            for name in ("oracle_mxfp8_quantize_rowwise",
                         "oracle_mxfp8_quantize_colwise"):
                f = getattr(L, name)
                f.restype = ctypes.c_int
                f.argtypes = [_p, _i64, _i64, _i64, _p, _p]
            L.oracle_mxfp8_dequantize.restype = ctypes.c_int
            L.oracle_mxfp8_dequantize.argtypes = [_p, _p, _i64, _i64, _p]
            L.oracle_bf16_amax.restype = ctypes.c_float
            L.oracle_bf16_amax.argtypes = [_p, _i64, _i64, _i64]
            L.oracle_nvfp4_tensor_scale.restype = ctypes.c_float
            L.oracle_nvfp4_tensor_scale.argtypes = [ctypes.c_float]
            L.oracle_nvfp4_encode_rows.restype = ctypes.c_int
            L.oracle_nvfp4_encode_rows.argtypes = [_p, _i64, _i64, _i64, _p,
                                                   _i64, _p, _p]
            L.oracle_nvfp4_quantize_per_token.restype = ctypes.c_int
            L.oracle_nvfp4_quantize_per_token.argtypes = [_p, _i64, _i64,
                                                          _i64, _p, _p, _p]
            L.oracle_nvfp4_dequantize.restype = ctypes.c_int
            L.oracle_nvfp4_dequantize.argtypes = [_p, _p, _p, _i64, _i64,
                                                  _i64, _p]
            L.oracle_swizzled_scale_bytes.restype = ctypes.c_int64
            L.oracle_swizzled_scale_bytes.argtypes = [_i64, _i64]
            L.oracle_scale_swizzle.restype = ctypes.c_int
            L.oracle_scale_swizzle.argtypes = [_p, _i64, _i64, _p]
            L.oracle_scale_unswizzle.restype = ctypes.c_int
            L.oracle_scale_unswizzle.argtypes = [_p, _i64, _i64, _p]
            L.oracle_fp8blk_scale.restype = ctypes.c_float
            L.oracle_fp8blk_scale.argtypes = [ctypes.c_float]
            L.oracle_fp8blk_quantize.restype = ctypes.c_int
            L.oracle_fp8blk_quantize.argtypes = [_p, _i64, _i64, _i64, _i64,
                                                 _i64, _p, _p]
            L.oracle_fp8blk_dequantize.restype = ctypes.c_int
            L.oracle_fp8blk_dequantize.argtypes = [_p, _p, _i64, _i64, _i64,
                                                   _i64, _p]
            L.oracle_philox4x64.restype = None
            L.oracle_philox4x64.argtypes = [_p, _p, _p]
            L.oracle_rht_signs.restype = ctypes.c_uint32
            L.oracle_rht_signs.argtypes = [ctypes.c_uint64]
            L.oracle_rht16.restype = None
            L.oracle_rht16.argtypes = [_p, ctypes.c_uint32, _p]
            L.oracle_nvfp4_rht_sr_rows.restype = ctypes.c_int
            L.oracle_nvfp4_rht_sr_rows.argtypes = [_p, _i64, _i64, _i64,
                                                   ctypes.c_uint64, ctypes.c_int,
                                                   _i64, _p, _p, _p]
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("bf16 tensors are passed as uint16 bit patterns")
    return x


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: bad shape")


# --------------------------------------------------------------------------
# Scalar codecs (formats section of "Miles: end-to-end MXFP8 and per-token
# NVFP4 RL"; bit layouts are the standard format definitions).
# --------------------------------------------------------------------------
def decode_bf16(b: int) -> float:
    return lib().oracle_decode_bf16(int(b))


def decode_e4m3(c: int) -> float:
    return lib().oracle_decode_e4m3(int(c))


def decode_e2m1(c: int) -> float:
    return lib().oracle_decode_e2m1(int(c))


def decode_e8m0(c: int) -> float:
    return lib().oracle_decode_e8m0(int(c))


def rne_e4m3(v: float) -> int:
    return lib().oracle_rne_e4m3(float(v))


def rne_e2m1(v: float) -> int:
    return lib().oracle_rne_e2m1(float(v))


def rne_bf16(f: float) -> int:
    """Round a binary32 value (given as a Python float that is exactly a
    binary32 value) to bf16 bits, nearest-even."""
    return lib().oracle_rne_bf16(float(f))


def mxfp8_scale_exponent(a: float) -> int:
    """k = smallest integer in [-127, 127] with 448 * 2^k >= a (formats
    section: the power-of-two scale is rounded up so the block max is not
    clipped)."""
    return lib().oracle_mxfp8_scale_exponent(float(a))


# --------------------------------------------------------------------------
# MXFP8 tensor ops (formats section; MXFP8 recipe section for the
# independent rowwise / columnwise copies).
# --------------------------------------------------------------------------
def mxfp8_quantize_rowwise(x: np.ndarray):
    """1x32 blocks along each row of x [R, C] (bf16 bits).
    Returns (codes u8 [R, C], scales u8 [R, C/32]) in logical layout."""
    x = _bf16(x)
    R, C = x.shape
    codes = np.empty((R, C), np.uint8)
    scales = np.empty((R, C // 32), np.uint8)
    _check(lib().oracle_mxfp8_quantize_rowwise(_ptr(x), R, C, C, _ptr(codes),
                                               _ptr(scales)), "rowwise")
    return codes, scales


def mxfp8_quantize_colwise(x: np.ndarray):
    """32x1 blocks down each column of x [M, K], quantized from x itself.
    Returns (codes_t u8 [K, M], scales_t u8 [K, M/32]): the copy is stored
    transposed so each 32x1 block is 32 contiguous bytes."""
    x = _bf16(x)
    M, K = x.shape
    codes = np.empty((K, M), np.uint8)
    scales = np.empty((K, M // 32), np.uint8)
    _check(lib().oracle_mxfp8_quantize_colwise(_ptr(x), M, K, K, _ptr(codes),
                                               _ptr(scales)), "colwise")
    return codes, scales


def mxfp8_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """bf16 bits of E4M3(code) * 2^(e-127), blocks of 32 along rows
    (backward-mode section: the exact forward operands, dequantized)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    R, C = codes.shape
    y = np.empty((R, C), np.uint16)
    _check(lib().oracle_mxfp8_dequantize(_ptr(codes), _ptr(scales), R, C,
                                         _ptr(y)), "mxfp8 dequant")
    return y


# --------------------------------------------------------------------------
# NVFP4 tensor ops (formats section: E2M1 + E4M3 per 16 + FP32 scope scale;
# NVFP4 recipe section: per-token FP32 activation scale, gate/up share one
# FP32 weight scale).
# --------------------------------------------------------------------------
def bf16_amax(x: np.ndarray) -> float:
    x = _bf16(x)
    x2 = x.reshape(-1, x.shape[-1]) if x.ndim > 1 else x.reshape(1, -1)
    return float(lib().oracle_bf16_amax(_ptr(x2), x2.shape[0], x2.shape[1],
                                        x2.shape[1]))


def nvfp4_tensor_scale(amax: float) -> float:
    """S = amax / (6 * 448) in binary32 (a decode scale)."""
    return float(lib().oracle_nvfp4_tensor_scale(float(amax)))


def nvfp4_encode_rows(x: np.ndarray, S: np.ndarray):
    """Encode rows of x [R, C] with FP32 scales S (shape [R] or [1]).
    Returns (codes u8 [R, C/2] packed low-nibble-first, scales u8 [R, C/16])."""
    x = _bf16(x)
    R, C = x.shape
    S = np.ascontiguousarray(S, np.float32).reshape(-1)
    stride = 1 if S.size == R else 0
    if S.size not in (1, R):
        raise ValueError("S must have one entry per row or one in total")
    codes = np.empty((R, C // 2), np.uint8)
    scales = np.empty((R, C // 16), np.uint8)
    _check(lib().oracle_nvfp4_encode_rows(_ptr(x), R, C, C, _ptr(S), stride,
                                          _ptr(codes), _ptr(scales)),
           "nvfp4 encode")
    return codes, scales


def nvfp4_quantize_per_token(x: np.ndarray):
    """Per-token NVFP4: S_t = amax_t / 2688 (FP32), then E4M3 block scales
    and packed E2M1 codes.  Returns (codes [T, H/2], scales [T, H/16],
    S f32 [T])."""
    x = _bf16(x)
    T, H = x.shape
    codes = np.empty((T, H // 2), np.uint8)
    scales = np.empty((T, H // 16), np.uint8)
    S = np.empty((T,), np.float32)
    _check(lib().oracle_nvfp4_quantize_per_token(_ptr(x), T, H, H,
                                                 _ptr(codes), _ptr(scales),
                                                 _ptr(S)), "per-token")
    return codes, scales, S


def nvfp4_quantize_group(parts, S_in: float | None = None):
    """Quantize the parts of one weight group (e.g. gate and up of one
    expert) under ONE shared FP32 scale S = max_parts amax / 2688, or under
    ``S_in`` when given (live weight update reusing a stored scale).
    Output rows are the parts' rows concatenated.
    Returns (codes [sum_rows, K/2], scales [sum_rows, K/16], S)."""
    parts = [_bf16(p) for p in parts]
    K = parts[0].shape[1]
    if S_in is None:
        amax = max(bf16_amax(p) for p in parts)
        S = nvfp4_tensor_scale(amax)
    else:
        S = float(np.float32(S_in))
    x = np.concatenate(parts, axis=0)
    codes, scales = nvfp4_encode_rows(x, np.array([S], np.float32))
    assert x.shape[1] == K
    return codes, scales, np.float32(S)


def nvfp4_dequantize(codes: np.ndarray, scales: np.ndarray,
                     S: np.ndarray) -> np.ndarray:
    """bf16 bits of (E2M1(c) * E4M3(sb)) * S; S has one entry per row or
    one in total."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    R, half = codes.shape
    C = half * 2
    S = np.ascontiguousarray(S, np.float32).reshape(-1)
    stride = 1 if S.size == R else 0
    y = np.empty((R, C), np.uint16)
    _check(lib().oracle_nvfp4_dequantize(_ptr(codes), _ptr(scales), _ptr(S),
                                         stride, R, C, _ptr(y)),
           "nvfp4 dequant")
    return y


# --------------------------------------------------------------------------
# Swizzled scale layout (not on the pages; the 128x4-tile layout read by
# block-scaled tensor-core MMA).
# --------------------------------------------------------------------------
def swizzled_scale_bytes(R: int, C: int) -> int:
    return int(lib().oracle_swizzled_scale_bytes(R, C))


def scale_swizzle(logical: np.ndarray) -> np.ndarray:
    logical = np.ascontiguousarray(logical, np.uint8)
    R, C = logical.shape
    out = np.empty((swizzled_scale_bytes(R, C),), np.uint8)
    lib().oracle_scale_swizzle(_ptr(logical), R, C, _ptr(out))
    return out


def scale_unswizzle(swz: np.ndarray, R: int, C: int) -> np.ndarray:
    swz = np.ascontiguousarray(swz, np.uint8).reshape(-1)
    if swz.size < swizzled_scale_bytes(R, C):
        raise ValueError("swizzled buffer too small")
    out = np.empty((R, C), np.uint8)
    lib().oracle_scale_unswizzle(_ptr(swz), R, C, _ptr(out))
    return out


# --------------------------------------------------------------------------
# Decoded value tables (exact, float64) built from the scalar decoders.
# --------------------------------------------------------------------------
_E4M3_F64 = None
_E2M1_F64 = None


def e4m3_table() -> np.ndarray:
    global _E4M3_F64
    if _E4M3_F64 is None:
        _E4M3_F64 = np.array([decode_e4m3(c) for c in range(256)], np.float64)
    return _E4M3_F64


def e2m1_table() -> np.ndarray:
    global _E2M1_F64
    if _E2M1_F64 is None:
        _E2M1_F64 = np.array([decode_e2m1(c) for c in range(16)], np.float64)
    return _E2M1_F64


# --------------------------------------------------------------------------
# GEMM oracle (experiments section: FP4 / MXFP8 tensor-core GEMMs with the
# per-token FP32 scale applied in the epilogue).  float64 accumulation over
# operands dequantized exactly (code x block scale is exact in float64).
# --------------------------------------------------------------------------
def mxfp8_operand_f64(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Exact float64 values of an MXFP8 operand, blocks of 32 along rows."""
    R, C = codes.shape
    v = e4m3_table()[codes]
    s = np.ldexp(1.0, scales.astype(np.int64) - 127)
    return v * np.repeat(s, 32, axis=1)[:, :C]


def nvfp4_operand_f64(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Exact float64 values E2M1(c) * E4M3(sb) (without the FP32 scale)."""
    R, half = codes.shape
    lo = codes & 0xF
    hi = codes >> 4
    q = np.empty((R, half * 2), np.uint8)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    v = e2m1_table()[q]
    sb = e4m3_table()[scales]
    return v * np.repeat(sb, 16, axis=1)


def gemm_mxfp8(a_codes, a_scales, bt_codes, bt_scales) -> np.ndarray:
    """C[m, n] = sum_k A[m, k] * B[k, n] over dequantized operands, with A
    given rowwise [M, K] and B given as its columnwise copy B^T [N, K]."""
    A = mxfp8_operand_f64(a_codes, a_scales)
    Bt = mxfp8_operand_f64(bt_codes, bt_scales)
    return A @ Bt.T


def gemm_nvfp4_grouped(a_codes, a_scales, a_S, offsets, w_codes, w_scales,
                       w_S) -> np.ndarray:
    """Grouped expert GEMM: rows offsets[e]:offsets[e+1] of A use expert e's
    weight W_e [N, K]; C[r, :] = S_tok[r] * S_w[e] * sum_k a * w, with the
    two FP32 scales applied after the float64 accumulation."""
    M = a_codes.shape[0]
    N = w_codes.shape[1]
    C = np.zeros((M, N), np.float64)
    A = nvfp4_operand_f64(a_codes, a_scales)
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 <= r0:
            continue
        W = nvfp4_operand_f64(w_codes[e], w_scales[e])
        acc = A[r0:r1] @ W.T
        C[r0:r1] = acc * (a_S[r0:r1, None].astype(np.float64)
                          * float(w_S[e]))
    return C


# --------------------------------------------------------------------------
# MoE expert forward up to the activation ("Miles: end-to-end MXFP8 and
# per-token NVFP4 RL", NVFP4 recipe section: SwiGLU MoE layers fuse the gate
# and up projections into one GEMM under one FP32 weight scale).  SwiGLU is
# taken in its standard form h = silu(gate) * up, silu(z) = z * sigmoid(z),
# evaluated in float64 on the float64 GEMM result.
# --------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + exp(-z)), float64 (exp overflow -> 0)."""
    z = np.asarray(z, np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def gather_rows(x: np.ndarray, row_index: np.ndarray) -> np.ndarray:
    """Row t of the result is x[row_index[t]], or a zero row where the index
    is outside [0, len(x)) (the padding rows of an expert group)."""
    out = np.zeros((len(row_index),) + x.shape[1:], x.dtype)
    ok = (row_index >= 0) & (row_index < x.shape[0])
    out[ok] = x[row_index[ok]]
    return out


def moe_gate_up_swiglu(a_codes, a_scales, a_S, offsets, w_codes, w_scales,
                       w_S) -> np.ndarray:
    """Grouped gate/up GEMM (expert e's weight = [gate_e ; up_e], 2F x K,
    one FP32 scale per expert) with both FP32 scales, then SwiGLU:
    h[r, j] = silu(C[r, j]) * C[r, F + j]."""
    F = w_codes.shape[1] // 2
    C = gemm_nvfp4_grouped(a_codes, a_scales, a_S, offsets, w_codes,
                           w_scales, w_S)
    return silu(C[:, :F]) * C[:, F:]


# --------------------------------------------------------------------------
# FP8 E4M3 with FP32 block scales: the DeepSeek-V3-style recipe named in the
# introduction of "Miles: end-to-end MXFP8 and per-token NVFP4 RL" (weights
# in 128x128 blocks, activations in 1x128 tiles, scales computed online) and
# its backward conversion (MXFP8 recipe section: dequantize, then requantize
# in the backward orientation).  Arithmetic in mxq_oracle.c.
# --------------------------------------------------------------------------
def fp8_block_scale(amax: float) -> float:
    """S = amax / 448 in binary32 (a decode scale)."""
    return float(lib().oracle_fp8blk_scale(float(amax)))


def fp8_block_quantize(x: np.ndarray, block_rows: int = 1,
                       block_cols: int = 128):
    """E4M3 codes u8 [R, C] and FP32 scales [R/block_rows, C/block_cols] of
    x [R, C] (bf16 bits): 1x128 tiles (block_rows = 1) or 128x128 blocks."""
    x = _bf16(x)
    R, C = x.shape
    codes = np.empty((R, C), np.uint8)
    scales = np.empty((R // block_rows, C // block_cols), np.float32)
    _check(lib().oracle_fp8blk_quantize(_ptr(x), R, C, C, block_rows,
                                        block_cols, _ptr(codes), _ptr(scales)),
           "fp8 block quantize")
    return codes, scales


def fp8_block_dequantize(codes: np.ndarray, scales: np.ndarray,
                         block_rows: int = 1, block_cols: int = 128) -> np.ndarray:
    """bf16 bits of E4M3(code) * S, S the code's block scale."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    R, C = codes.shape
    y = np.empty((R, C), np.uint16)
    _check(lib().oracle_fp8blk_dequantize(_ptr(codes), _ptr(scales), R, C,
                                          block_rows, block_cols, _ptr(y)),
           "fp8 block dequantize")
    return y


def fp8_block_requantize_transpose(codes: np.ndarray, scales: np.ndarray):
    """The backward-orientation conversion of 1x128-tile FP8 activations
    X [M, K]: dequantize to bf16, then quantize the transpose X^T [K, M]
    in 1x128 tiles (128x1 blocks of X).  Returns (codes_t [K, M], scales_t
    [K, M/128])."""
    y = fp8_block_dequantize(codes, scales, 1, 128)
    return fp8_block_quantize(np.ascontiguousarray(y.T), 1, 128)


# --------------------------------------------------------------------------
# NVFP4 with the original pretraining recipe's stabilizers (NVFP4 recipe
# section of "Miles: end-to-end MXFP8 and per-token NVFP4 RL": stochastic
# rounding for unbiased quantized gradients, Random Hadamard Transforms to
# disperse block outliers).  Readings and arithmetic in mxq_oracle.c.
# --------------------------------------------------------------------------
RHT = 1
SR = 2


def philox4x64(counter, key) -> np.ndarray:
    """Philox4x64-10 (Salmon et al., SC 2011) of a 4-word counter and a
    2-word key."""
    c = np.ascontiguousarray(counter, np.uint64)
    k = np.ascontiguousarray(key, np.uint64)
    out = np.empty(4, np.uint64)
    lib().oracle_philox4x64(_ptr(c), _ptr(k), _ptr(out))
    return out


def rht_signs(seed: int) -> int:
    """The 16 RHT sign bits of a seed (bit i set: s_i = -1)."""
    return int(lib().oracle_rht_signs(ctypes.c_uint64(seed)))


def rht16(x: np.ndarray, signs: int) -> np.ndarray:
    """(1/4) H16 (s * x) for one block of 16 binary32 values."""
    x = np.ascontiguousarray(x, np.float32)
    y = np.empty(16, np.float32)
    lib().oracle_rht16(_ptr(x), signs, _ptr(y))
    return y


def nvfp4_quantize_rht_sr(x: np.ndarray, seed: int, flags: int,
                          row0: int = 0):
    """Per-token NVFP4 of x [R, C] (bf16 bits) with the optional RHT
    (flags & RHT) and stochastic rounding (flags & SR); x holds rows
    row0 .. row0 + R - 1 of the tensor.  Returns (codes u8 [R, C/2], block
    scales u8 [R, C/16] logical, S f32 [R])."""
    x = _bf16(x)
    R, C = x.shape
    codes = np.empty((R, C // 2), np.uint8)
    scales = np.empty((R, C // 16), np.uint8)
    S = np.empty(R, np.float32)
    _check(lib().oracle_nvfp4_rht_sr_rows(_ptr(x), R, C, C, ctypes.c_uint64(seed),
                                          flags, row0, _ptr(codes),
                                          _ptr(scales), _ptr(S)),
           "nvfp4 rht/sr")
    return codes, scales, S


def gemm_bf16_mxfp8(a: np.ndarray, bt_codes: np.ndarray,
                    bt_scales: np.ndarray) -> np.ndarray:
    """The dequantized-backward GEMM (backward-mode section of "Miles:
    end-to-end MXFP8 and per-token NVFP4 RL": BF16 GEMMs on BF16
    dequantizations of the exact forward operands): float64
    A [M, K] (bf16 bits) @ dequant(B^T [N, K])^T, the dequantization
    exact (E4M3 x 2^k lands on the bf16 grid)."""
    a64 = W_bits_to_f64(a)
    b64 = W_bits_to_f64(mxfp8_dequantize(bt_codes, bt_scales))
    return a64 @ b64.T


def W_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    u = np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)
