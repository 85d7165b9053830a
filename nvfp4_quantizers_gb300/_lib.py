"""ctypes binding of libmxq (include/mxq.h).

Argument marshalling only: every step of every operation runs in the CUDA
kernels of libmxq.so.  There is no fallback: if the library has not been
built, or a call fails, a RuntimeError is raised.  PyTorch supplies device
memory (outputs are allocated with ``torch.empty`` on the input's device)
and the stream (``torch.cuda.current_stream()``).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import NamedTuple, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmxq.so")

MXQ_OK = 0
MXQ_ERR_NULL = 1
MXQ_ERR_SHAPE = 2
MXQ_ERR_ALIGN = 3
MXQ_ERR_LAYOUT = 4
MXQ_ERR_WORKSPACE = 5
MXQ_ERR_CUDA = 6
MXQ_ERR_TIMEOUT = 7
MXQ_ERR_ARG = 8

SCALE_LINEAR = 0
SCALE_SWIZZLED = 1
S_PER_ROW = 0
S_PER_BATCH = 1

_LAYOUTS = {"linear": SCALE_LINEAR, "swizzled": SCALE_SWIZZLED,
            SCALE_LINEAR: SCALE_LINEAR, SCALE_SWIZZLED: SCALE_SWIZZLED}

_lib = None
_lock = threading.Lock()
_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int


class MxqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libmxq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libmxq.so not found at {LIB_PATH}; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        L.mxq_status_string.restype = ctypes.c_char_p
        L.mxq_status_string.argtypes = [_int]
        L.mxq_version.restype = _int
        L.mxq_version.argtypes = []
        L.mxq_scale_bytes.restype = _i64
        L.mxq_scale_bytes.argtypes = [_i64, _i64, _int]
        L.mxq_get_last_error.restype = _int
        L.mxq_get_last_error.argtypes = []
        L.mxq_selftest_wait_timeout.restype = _int
        L.mxq_selftest_wait_timeout.argtypes = [_p]
        L.mxq_set_fault_inject.restype = None
        L.mxq_set_fault_inject.argtypes = [_int]
        L.mxfp8_quantize_rowcol.restype = _int
        L.mxfp8_quantize_rowcol.argtypes = [_p, _i64, _i64, _i64, _p, _p, _p,
                                            _p, _int, _p]
        L.nvfp4_quantize_per_token.restype = _int
        L.nvfp4_quantize_per_token.argtypes = [_p, _i64, _i64, _i64, _p, _p,
                                               _p, _int, _p]
        L.nvfp4_quantize_per_token_gather.restype = _int
        L.nvfp4_quantize_per_token_gather.argtypes = [
            _p, _i64, _i64, _i64, _p, _i64, _p, _p, _p, _int, _p]
        L.nvfp4_quantize_weight_shared_workspace_size.restype = ctypes.c_size_t
        L.nvfp4_quantize_weight_shared_workspace_size.argtypes = [_i64]
        L.nvfp4_quantize_weight_shared.restype = _int
        L.nvfp4_quantize_weight_shared.argtypes = [
            _i64, _int, _p, _p, _i64, _p, _p, _p, _p, _int, _p,
            ctypes.c_size_t, _p]
        L.dequantize_mxfp8.restype = _int
        L.dequantize_mxfp8.argtypes = [_p, _p, _i64, _i64, _int, _p, _p]
        L.mxq_gemm_mxfp8.restype = _int
        L.mxq_gemm_mxfp8.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p,
                                     _i64, _p]
        L.mxq_gemm_nvfp4_grouped.restype = _int
        L.mxq_gemm_nvfp4_grouped.argtypes = [_p, _p, _p, _p, _i64, _p, _p, _p,
                                             _i64, _i64, _p, _i64, _p]
        L.mxq_moe_gate_up_swiglu_nvfp4.restype = _int
        L.mxq_moe_gate_up_swiglu_nvfp4.argtypes = [
            _p, _p, _p, _p, _i64, _p, _p, _p, _i64, _i64, _p, _i64, _p]
        L.mxq_gemm_nvfp4_grouped_gather.restype = _int
        L.mxq_gemm_nvfp4_grouped_gather.argtypes = [
            _p, _p, _p, _i64, _p, _p, _i64, _p, _p, _p, _i64, _i64, _p, _i64, _p]
        L.mxq_moe_gate_up_swiglu_nvfp4_gather.restype = _int
        L.mxq_moe_gate_up_swiglu_nvfp4_gather.argtypes = [
            _p, _p, _p, _i64, _p, _p, _i64, _p, _p, _p, _i64, _i64, _p, _i64, _p]
        L.dequantize_nvfp4.restype = _int
        L.dequantize_nvfp4.argtypes = [_p, _p, _p, _int, _i64, _i64, _i64,
                                       _int, _p, _p]
        L.mxq_gemm_bf16_mxfp8.restype = _int
        L.mxq_gemm_bf16_mxfp8.argtypes = [_p, _i64, _p, _p, _i64, _i64, _i64,
                                          _p, _i64, _p]
        L.nvfp4_quantize_per_token_rht_sr.restype = _int
        L.nvfp4_quantize_per_token_rht_sr.argtypes = [
            _p, _i64, _i64, _i64, ctypes.c_uint64, _int, _p, _p, _p, _int, _p]
        L.fp8_block_quantize.restype = _int
        L.fp8_block_quantize.argtypes = [_p, _i64, _i64, _i64, _int, _p, _p,
                                         _p]
        L.fp8_block_dequantize.restype = _int
        L.fp8_block_dequantize.argtypes = [_p, _p, _i64, _i64, _int, _p, _p]
        L.fp8_block_requantize_transpose.restype = _int
        L.fp8_block_requantize_transpose.argtypes = [_p, _p, _i64, _i64, _p,
                                                     _p, _p]
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().mxq_status_string(int(status)).decode()


def scale_bytes(rows: int, cols: int, scale_layout="swizzled") -> int:
    n = lib().mxq_scale_bytes(int(rows), int(cols), _layout(scale_layout))
    if n < 0:
        raise ValueError("bad scale layout or size")
    return int(n)


def get_last_error() -> int:
    """Synchronizes the device; returns the status of bounded device waits
    (MXQ_ERR_TIMEOUT) or of the CUDA runtime (MXQ_ERR_CUDA)."""
    return int(lib().mxq_get_last_error())


def selftest_wait_timeout(device=None) -> None:
    """Launch the failure-detection self-test kernel (a bounded device wait
    that runs out after 20 ms); the next get_last_error() reports
    MXQ_ERR_TIMEOUT (C: mxq_selftest_wait_timeout)."""
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if device is None else torch.device(device)
    _check(lib().mxq_selftest_wait_timeout(_stream(dev)),
           "mxq_selftest_wait_timeout")


def set_fault_inject(mode: int) -> None:
    lib().mxq_set_fault_inject(int(mode))


def _layout(scale_layout) -> int:
    try:
        return _LAYOUTS[scale_layout]
    except KeyError:
        raise ValueError(f"unknown scale layout {scale_layout!r}") from None


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(status: int, what: str):
    if status != MXQ_OK:
        raise MxqError(status, what)


def _bf16_2d(x: torch.Tensor, name: str) -> torch.Tensor:
    if x.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with unit column stride")
    return x


class Mxfp8Quantized(NamedTuple):
    row_codes: torch.Tensor | None      # u8 [M, K]
    row_scales: torch.Tensor | None     # E8M0 bytes, logical [M, K/32]
    col_codes_t: torch.Tensor | None    # u8 [K, M] (columnwise copy, transposed)
    col_scales_t: torch.Tensor | None   # E8M0 bytes, logical [K, M/32]
    scale_layout: int


class Nvfp4Quantized(NamedTuple):
    codes: torch.Tensor                 # u8 [..., R, H/2]
    block_scales: torch.Tensor          # E4M3 bytes
    scales: torch.Tensor                # f32 per token [T] or per group [G]
    scale_layout: int


def mxfp8_quantize_rowcol(x: torch.Tensor, rowwise: bool = True,
                          colwise: bool = True,
                          scale_layout="swizzled") -> Mxfp8Quantized:
    """MXFP8 rowwise (1x32) and/or columnwise (32x1) quantization of a bf16
    [M, K] tensor in one pass (C: mxfp8_quantize_rowcol)."""
    x = _bf16_2d(x, "x")
    lay = _layout(scale_layout)
    M, K = x.shape
    dev = x.device
    rc = rs = cc = cs = None
    if rowwise:
        rc = torch.empty((M, K), dtype=torch.uint8, device=dev)
        rs = torch.empty((scale_bytes(M, K // 32, lay),), dtype=torch.uint8,
                         device=dev)
    if colwise:
        cc = torch.empty((K, M), dtype=torch.uint8, device=dev)
        cs = torch.empty((scale_bytes(K, M // 32, lay),), dtype=torch.uint8,
                         device=dev)
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    _check(lib().mxfp8_quantize_rowcol(
        x.data_ptr(), M, K, x.stride(0), ptr(rc), ptr(rs), ptr(cc), ptr(cs),
        lay, _stream(dev)), "mxfp8_quantize_rowcol")
    return Mxfp8Quantized(rc, rs, cc, cs, lay)


def nvfp4_quantize_per_token(x: torch.Tensor,
                             scale_layout="swizzled") -> Nvfp4Quantized:
    """NVFP4 quantization with one FP32 scale per token (row) of a bf16
    [T, H] tensor (C: nvfp4_quantize_per_token)."""
    x = _bf16_2d(x, "x")
    lay = _layout(scale_layout)
    T, H = x.shape
    dev = x.device
    codes = torch.empty((T, H // 2), dtype=torch.uint8, device=dev)
    bs = torch.empty((scale_bytes(T, H // 16, lay),), dtype=torch.uint8,
                     device=dev)
    S = torch.empty((T,), dtype=torch.float32, device=dev)
    _check(lib().nvfp4_quantize_per_token(
        x.data_ptr(), T, H, x.stride(0), codes.data_ptr(), bs.data_ptr(),
        S.data_ptr(), lay, _stream(dev)), "nvfp4_quantize_per_token")
    return Nvfp4Quantized(codes, bs, S, lay)


def nvfp4_quantize_per_token_gather(x: torch.Tensor, row_index: torch.Tensor,
                                    scale_layout="swizzled") -> Nvfp4Quantized:
    """Per-token NVFP4 quantization of gathered rows: output row t is row
    row_index[t] of the bf16 [T_src, H] tensor x, or a zero row where the
    index is outside [0, T_src) (C: nvfp4_quantize_per_token_gather)."""
    x = _bf16_2d(x, "x")
    if (row_index.dtype != torch.int32 or row_index.dim() != 1
            or row_index.device != x.device or not row_index.is_contiguous()):
        raise ValueError("row_index must be a contiguous int32 vector on "
                         "x's device")
    lay = _layout(scale_layout)
    T_src, H = x.shape
    T = row_index.numel()
    dev = x.device
    codes = torch.empty((T, H // 2), dtype=torch.uint8, device=dev)
    bs = torch.empty((scale_bytes(T, H // 16, lay),), dtype=torch.uint8,
                     device=dev)
    S = torch.empty((T,), dtype=torch.float32, device=dev)
    _check(lib().nvfp4_quantize_per_token_gather(
        x.data_ptr(), T_src, H, x.stride(0), row_index.data_ptr(), T,
        codes.data_ptr(), bs.data_ptr(), S.data_ptr(), lay, _stream(dev)),
        "nvfp4_quantize_per_token_gather")
    return Nvfp4Quantized(codes, bs, S, lay)


NVFP4_RHT = 1
NVFP4_SR = 2


def nvfp4_quantize_per_token_rht_sr(x: torch.Tensor, seed: int, flags: int,
                                    scale_layout="swizzled") -> Nvfp4Quantized:
    """Per-token NVFP4 with the pretraining recipe's stabilizers: a 16-value
    Random Hadamard Transform (flags & NVFP4_RHT) and stochastic rounding
    (flags & NVFP4_SR), random bits from Philox4x64-10 keyed by seed
    (C: nvfp4_quantize_per_token_rht_sr)."""
    x = _bf16_2d(x, "x")
    lay = _layout(scale_layout)
    T, H = x.shape
    dev = x.device
    codes = torch.empty((T, H // 2), dtype=torch.uint8, device=dev)
    bs = torch.empty((scale_bytes(T, H // 16, lay),), dtype=torch.uint8,
                     device=dev)
    S = torch.empty((T,), dtype=torch.float32, device=dev)
    _check(lib().nvfp4_quantize_per_token_rht_sr(
        x.data_ptr(), T, H, x.stride(0), ctypes.c_uint64(seed), flags,
        codes.data_ptr(), bs.data_ptr(), S.data_ptr(), lay, _stream(dev)),
        "nvfp4_quantize_per_token_rht_sr")
    return Nvfp4Quantized(codes, bs, S, lay)


def nvfp4_quantize_weight_shared(groups: Sequence[Sequence[torch.Tensor]],
                                 group_scales_in: torch.Tensor | None = None,
                                 scale_layout="swizzled",
                                 workspace: torch.Tensor | None = None
                                 ) -> Nvfp4Quantized:
    """NVFP4 weight quantization where all parts of a group share one FP32
    scale (gate/up pair: two parts per group)
    (C: nvfp4_quantize_weight_shared).

    groups[g][p] is a contiguous bf16 [rows_p, K] CUDA tensor; every group
    has the same part shapes.  Returns codes [G, R, K/2], block scales
    [G, scale_bytes(R, K/16)] and S [G]."""
    lay = _layout(scale_layout)
    G = len(groups)
    if G == 0:
        raise ValueError("no groups")
    P = len(groups[0])
    shapes = [tuple(t.shape) for t in groups[0]]
    K = shapes[0][1]
    for grp in groups:
        if [tuple(t.shape) for t in grp] != shapes:
            raise ValueError("every group must have the same part shapes")
        for t in grp:
            _bf16_2d(t, "part")
            if not t.is_contiguous():
                raise ValueError("parts must be contiguous")
    dev = groups[0][0].device
    R = sum(s[0] for s in shapes)
    ptrs = (ctypes.c_void_p * (G * P))(*[t.data_ptr() for grp in groups
                                         for t in grp])
    rows = (ctypes.c_int64 * P)(*[s[0] for s in shapes])
    codes = torch.empty((G, R, K // 2), dtype=torch.uint8, device=dev)
    sb = scale_bytes(R, K // 16, lay)
    bs = torch.empty((G, sb), dtype=torch.uint8, device=dev)
    S = torch.empty((G,), dtype=torch.float32, device=dev)
    ws_bytes = int(lib().nvfp4_quantize_weight_shared_workspace_size(G))
    if group_scales_in is None:
        if workspace is None:
            workspace = torch.empty((max(ws_bytes, 16),), dtype=torch.uint8,
                                    device=dev)
        ws_ptr, ws_len = workspace.data_ptr(), workspace.numel()
        sin = None
    else:
        if group_scales_in.dtype != torch.float32 or group_scales_in.numel() != G:
            raise ValueError("group_scales_in must be float32 [G]")
        sin = group_scales_in.contiguous()
        ws_ptr, ws_len = None, 0
    _check(lib().nvfp4_quantize_weight_shared(
        G, P, ctypes.cast(ptrs, ctypes.c_void_p), ctypes.cast(rows, ctypes.c_void_p),
        K, codes.data_ptr(), bs.data_ptr(), S.data_ptr(),
        None if sin is None else sin.data_ptr(), lay, ws_ptr, ws_len,
        _stream(dev)), "nvfp4_quantize_weight_shared")
    return Nvfp4Quantized(codes, bs, S, lay)


def dequantize_mxfp8(codes: torch.Tensor, scales: torch.Tensor,
                     scale_layout="swizzled") -> torch.Tensor:
    """bf16 [rows, cols] from MXFP8 codes [rows, cols] and their E8M0 scales
    (C: dequantize_mxfp8)."""
    lay = _layout(scale_layout)
    if codes.dtype != torch.uint8 or codes.dim() != 2 or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous uint8 [rows, cols] tensor")
    rows, cols = codes.shape
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device=codes.device)
    _check(lib().dequantize_mxfp8(codes.data_ptr(), scales.data_ptr(), rows,
                                  cols, lay, y.data_ptr(),
                                  _stream(codes.device)), "dequantize_mxfp8")
    return y


def dequantize_nvfp4(codes: torch.Tensor, block_scales: torch.Tensor,
                     S: torch.Tensor, scale_layout="swizzled") -> torch.Tensor:
    """bf16 from NVFP4 codes.  codes [rows, cols/2] with S per row [rows]
    (activations), or codes [batch, rows, cols/2] with S per batch entry
    [batch] (weight groups) (C: dequantize_nvfp4)."""
    lay = _layout(scale_layout)
    if codes.dtype != torch.uint8 or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous uint8 tensor")
    if codes.dim() == 2:
        batch, (rows, half) = 1, codes.shape
        mode = S_PER_ROW
        shape = (rows, half * 2)
    elif codes.dim() == 3:
        batch, rows, half = codes.shape
        mode = S_PER_BATCH
        shape = (batch, rows, half * 2)
    else:
        raise ValueError("codes must be 2-D or 3-D")
    if S.dtype != torch.float32:
        raise TypeError("S must be float32")
    y = torch.empty(shape, dtype=torch.bfloat16, device=codes.device)
    _check(lib().dequantize_nvfp4(codes.data_ptr(), block_scales.data_ptr(),
                                  S.data_ptr(), mode, batch, rows, half * 2,
                                  lay, y.data_ptr(), _stream(codes.device)),
           "dequantize_nvfp4")
    return y


def gemm_mxfp8(a_codes: torch.Tensor, a_scales: torch.Tensor,
               bt_codes: torch.Tensor, bt_scales: torch.Tensor) -> torch.Tensor:
    """fp32 C [M, N] = A @ B from the rowwise MXFP8 copy of A [M, K] and
    B^T [N, K] (the columnwise copy of B [K, N]); swizzled scales
    (C: mxq_gemm_mxfp8)."""
    M, K = a_codes.shape
    N = bt_codes.shape[0]
    if bt_codes.shape[1] != K:
        raise ValueError("A and B^T must share K")
    C = torch.empty((M, N), dtype=torch.float32, device=a_codes.device)
    _check(lib().mxq_gemm_mxfp8(a_codes.data_ptr(), a_scales.data_ptr(),
                                bt_codes.data_ptr(), bt_scales.data_ptr(), M, N,
                                K, C.data_ptr(), N, _stream(a_codes.device)),
           "mxq_gemm_mxfp8")
    return C


def gemm_bf16_mxfp8(a: torch.Tensor, bt_codes: torch.Tensor,
                    bt_scales: torch.Tensor) -> torch.Tensor:
    """fp32 C [M, N] = A (bf16 [M, K]) times the dequantization of an MXFP8
    operand given as B^T [N, K] (codes + swizzled E8M0 scales), its bf16
    values formed in shared memory only (C: mxq_gemm_bf16_mxfp8)."""
    _bf16_2d(a, "a")
    M, K = a.shape
    N = bt_codes.shape[0]
    if bt_codes.dtype != torch.uint8 or tuple(bt_codes.shape) != (N, K) or \
            not bt_codes.is_contiguous():
        raise ValueError("bt_codes must be a contiguous uint8 [N, K] tensor")
    C = torch.empty((M, N), dtype=torch.float32, device=a.device)
    _check(lib().mxq_gemm_bf16_mxfp8(a.data_ptr(), a.stride(0),
                                     bt_codes.data_ptr(), bt_scales.data_ptr(),
                                     M, N, K, C.data_ptr(), N,
                                     _stream(a.device)), "mxq_gemm_bf16_mxfp8")
    return C


def gemm_nvfp4_grouped(a_codes: torch.Tensor, a_scales: torch.Tensor,
                       a_token_scales: torch.Tensor, group_offsets,
                       w_codes: torch.Tensor, w_scales: torch.Tensor,
                       w_group_scales: torch.Tensor) -> torch.Tensor:
    """Expert-grouped NVFP4 GEMM with the per-token and per-group FP32
    scales applied in the epilogue (C: mxq_gemm_nvfp4_grouped).
    group_offsets: num_groups + 1 row offsets, multiples of 128."""
    offs = [int(v) for v in group_offsets]
    G = len(offs) - 1
    M_total, half = a_codes.shape
    K = half * 2
    N = w_codes.shape[1]
    off_arr = (ctypes.c_int64 * len(offs))(*offs)
    C = torch.empty((M_total, N), dtype=torch.float32, device=a_codes.device)
    _check(lib().mxq_gemm_nvfp4_grouped(
        a_codes.data_ptr(), a_scales.data_ptr(), a_token_scales.data_ptr(),
        ctypes.cast(off_arr, ctypes.c_void_p), G, w_codes.data_ptr(),
        w_scales.data_ptr(), w_group_scales.data_ptr(), N, K, C.data_ptr(), N,
        _stream(a_codes.device)), "mxq_gemm_nvfp4_grouped")
    return C


def moe_gate_up_swiglu(a_codes: torch.Tensor, a_scales: torch.Tensor,
                       a_token_scales: torch.Tensor, group_offsets,
                       w_codes: torch.Tensor, w_scales: torch.Tensor,
                       w_group_scales: torch.Tensor) -> torch.Tensor:
    """Grouped NVFP4 gate/up GEMM with SwiGLU in the epilogue
    (C: mxq_moe_gate_up_swiglu_nvfp4).  w_codes [G, 2F, K/2] holds each
    expert's F gate rows then its F up rows; returns bf16 h [rows, F],
    h = silu(gate) * up with both FP32 scales applied first."""
    offs = [int(v) for v in group_offsets]
    G = len(offs) - 1
    M_total, half = a_codes.shape
    K = half * 2
    F = w_codes.shape[1] // 2
    off_arr = (ctypes.c_int64 * len(offs))(*offs)
    h = torch.empty((M_total, F), dtype=torch.bfloat16, device=a_codes.device)
    _check(lib().mxq_moe_gate_up_swiglu_nvfp4(
        a_codes.data_ptr(), a_scales.data_ptr(), a_token_scales.data_ptr(),
        ctypes.cast(off_arr, ctypes.c_void_p), G, w_codes.data_ptr(),
        w_scales.data_ptr(), w_group_scales.data_ptr(), F, K, h.data_ptr(), F,
        _stream(a_codes.device)), "mxq_moe_gate_up_swiglu_nvfp4")
    return h


def _gather_operand(x: Nvfp4Quantized, row_index: torch.Tensor):
    if x.scale_layout != SCALE_LINEAR:
        raise ValueError("the gathered GEMMs take the tokens' block scales in "
                         "the linear layout (nvfp4_quantize_per_token(x, "
                         "'linear'))")
    if (row_index.dtype != torch.int32 or row_index.dim() != 1
            or row_index.device != x.codes.device or not row_index.is_contiguous()):
        raise ValueError("row_index must be a contiguous int32 vector on the "
                         "tokens' device")
    T_src, half = x.codes.shape
    return T_src, half * 2


def gemm_nvfp4_grouped_gather(x: Nvfp4Quantized, row_index: torch.Tensor,
                              group_offsets, w_codes: torch.Tensor,
                              w_scales: torch.Tensor,
                              w_group_scales: torch.Tensor) -> torch.Tensor:
    """Expert-grouped NVFP4 GEMM whose routed rows are gathered from the
    per-token operand x (quantized once, linear scales) as the GEMM loads
    them: row r is token row_index[r], padding rows (index outside
    [0, T_src)) give +0 (C: mxq_gemm_nvfp4_grouped_gather)."""
    T_src, K = _gather_operand(x, row_index)
    offs = [int(v) for v in group_offsets]
    G = len(offs) - 1
    if row_index.numel() != offs[-1]:
        raise ValueError("row_index must hold one entry per routed row")
    N = w_codes.shape[1]
    off_arr = (ctypes.c_int64 * len(offs))(*offs)
    C = torch.empty((offs[-1], N), dtype=torch.float32, device=x.codes.device)
    _check(lib().mxq_gemm_nvfp4_grouped_gather(
        x.codes.data_ptr(), x.block_scales.data_ptr(), x.scales.data_ptr(),
        T_src, row_index.data_ptr(), ctypes.cast(off_arr, ctypes.c_void_p), G,
        w_codes.data_ptr(), w_scales.data_ptr(), w_group_scales.data_ptr(), N,
        K, C.data_ptr(), N, _stream(x.codes.device)),
        "mxq_gemm_nvfp4_grouped_gather")
    return C


def moe_gate_up_swiglu_gather(x: Nvfp4Quantized, row_index: torch.Tensor,
                              group_offsets, w_codes: torch.Tensor,
                              w_scales: torch.Tensor,
                              w_group_scales: torch.Tensor) -> torch.Tensor:
    """MoE gate/up GEMM with SwiGLU in the epilogue, the routed rows
    gathered from the per-token operand x as the GEMM loads them
    (C: mxq_moe_gate_up_swiglu_nvfp4_gather).  Returns bf16 h [rows, F]."""
    T_src, K = _gather_operand(x, row_index)
    offs = [int(v) for v in group_offsets]
    G = len(offs) - 1
    if row_index.numel() != offs[-1]:
        raise ValueError("row_index must hold one entry per routed row")
    F = w_codes.shape[1] // 2
    off_arr = (ctypes.c_int64 * len(offs))(*offs)
    h = torch.empty((offs[-1], F), dtype=torch.bfloat16, device=x.codes.device)
    _check(lib().mxq_moe_gate_up_swiglu_nvfp4_gather(
        x.codes.data_ptr(), x.block_scales.data_ptr(), x.scales.data_ptr(),
        T_src, row_index.data_ptr(), ctypes.cast(off_arr, ctypes.c_void_p), G,
        w_codes.data_ptr(), w_scales.data_ptr(), w_group_scales.data_ptr(), F,
        K, h.data_ptr(), F, _stream(x.codes.device)),
        "mxq_moe_gate_up_swiglu_nvfp4_gather")
    return h


# --------------------------------------------------------------------------
# FP8 E4M3 with one FP32 scale per block (1x128 activation tiles, 128x128
# weight blocks) and the backward-orientation conversion of 1x128 tiles.
# --------------------------------------------------------------------------
class Fp8BlockQuantized(NamedTuple):
    codes: torch.Tensor                 # u8 [rows, cols]
    scales: torch.Tensor                # f32 [rows / block_rows, cols / 128]
    block_rows: int


def fp8_block_quantize(x: torch.Tensor, block_rows: int = 1) -> Fp8BlockQuantized:
    """E4M3 codes with one FP32 scale per 1x128 tile (block_rows = 1) or per
    128x128 block (block_rows = 128) (C: fp8_block_quantize)."""
    _bf16_2d(x, "x")
    rows, cols = x.shape
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    scales = torch.empty((max(rows // block_rows, 0), cols // 128),
                         dtype=torch.float32, device=x.device)
    _check(lib().fp8_block_quantize(x.data_ptr(), rows, cols, x.stride(0),
                                    block_rows, codes.data_ptr(),
                                    scales.data_ptr(), _stream(x.device)),
           "fp8_block_quantize")
    return Fp8BlockQuantized(codes, scales, block_rows)


def fp8_block_dequantize(codes: torch.Tensor, scales: torch.Tensor,
                         block_rows: int = 1) -> torch.Tensor:
    """bf16 [rows, cols] = E4M3(code) * S (C: fp8_block_dequantize)."""
    if codes.dtype != torch.uint8 or codes.dim() != 2 or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous uint8 [rows, cols] tensor")
    if scales.dtype != torch.float32 or not scales.is_contiguous():
        raise ValueError("scales must be a contiguous float32 tensor")
    rows, cols = codes.shape
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device=codes.device)
    _check(lib().fp8_block_dequantize(codes.data_ptr(), scales.data_ptr(),
                                      rows, cols, block_rows, y.data_ptr(),
                                      _stream(codes.device)),
           "fp8_block_dequantize")
    return y


def fp8_block_requantize_transpose(codes: torch.Tensor, scales: torch.Tensor
                                   ) -> Fp8BlockQuantized:
    """1x128 tiles of X^T from the 1x128 tiles of X [rows, cols], through
    X's bf16 dequantization (C: fp8_block_requantize_transpose)."""
    if codes.dtype != torch.uint8 or codes.dim() != 2 or not codes.is_contiguous():
        raise ValueError("codes must be a contiguous uint8 [rows, cols] tensor")
    if scales.dtype != torch.float32 or not scales.is_contiguous():
        raise ValueError("scales must be a contiguous float32 tensor")
    rows, cols = codes.shape
    codes_t = torch.empty((cols, rows), dtype=torch.uint8, device=codes.device)
    scales_t = torch.empty((cols, rows // 128), dtype=torch.float32,
                           device=codes.device)
    _check(lib().fp8_block_requantize_transpose(
        codes.data_ptr(), scales.data_ptr(), rows, cols, codes_t.data_ptr(),
        scales_t.data_ptr(), _stream(codes.device)),
        "fp8_block_requantize_transpose")
    return Fp8BlockQuantized(codes_t, scales_t, 1)
