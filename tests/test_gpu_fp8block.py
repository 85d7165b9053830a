"""GPU parity of FP8 with FP32 block scales: 1x128 activation tiles, 128x128
weight blocks, their dequantization, and the backward-orientation
conversion of 1x128 tiles ("Miles: end-to-end MXFP8 and per-token NVFP4
RL", introduction: the DeepSeek-V3-style recipe; MXFP8 recipe section: its
dequantize-and-requantize step before the backward GEMM).

Codes and FP32 scales are compared bit for bit with the oracle, the bf16
dequantization bit for bit; the conversion against the oracle's
composition (dequantize to bf16, transpose, quantize in 1x128 tiles).
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import assert_bytes_equal, dev_bf16, host_bits, host_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from nvfp4_quantizers_gb300 import build
    build.build()
    import nvfp4_quantizers_gb300 as q
    q.lib()
    return q


def _scales_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint32)


def check_fp8blk(q, x_bits, block_rows, x_dev=None):
    x = dev_bf16(x_bits) if x_dev is None else x_dev
    r = q.fp8_block_quantize(x, block_rows)
    y = q.fp8_block_dequantize(r.codes, r.scales, block_rows)
    torch.cuda.synchronize()
    oc, osc = O.fp8_block_quantize(x_bits, block_rows)
    assert_bytes_equal(host_u8(r.codes), oc, f"codes [{block_rows}]")
    assert_bytes_equal(_scales_bits(r.scales), osc.view(np.uint32),
                       f"scales [{block_rows}]")
    assert_bytes_equal(host_bits(y), O.fp8_block_dequantize(oc, osc, block_rows),
                       f"dequant [{block_rows}]")
    return r


def _classes(R, C):
    rng = np.random.default_rng(41)
    tiny = W.to_bf16_bits((rng.uniform(-1, 1, (R, C)) * 1e-37).astype(np.float32))
    mixed = W.to_bf16_bits((rng.standard_t(3, (R, C)) * 10.0 ** rng.uniform(
        -20, 20, (R, 1))).astype(np.float32))
    return {"random": W.mxfp8_random(R, C, seed=2), "boundary": W.mxfp8_boundary(R, C),
            "zeros": W.mxfp8_zeros(R, C), "maxes": W.mxfp8_maxes(R, C),
            "tiny": tiny, "mixed": mixed}


@pytest.mark.parametrize("cls", ["random", "boundary", "zeros", "maxes", "tiny",
                                 "mixed"])
def test_tiles_and_blocks_classes(mxq, cls):
    x = _classes(256, 384)[cls]
    check_fp8blk(mxq, x, 1)
    check_fp8blk(mxq, x, 128)


@pytest.mark.parametrize("R", [1, 7, 77, 300])
def test_tiles_any_rows(mxq, R):
    x = W.mxfp8_random(R, 640, seed=R)
    check_fp8blk(mxq, x, 1)


def test_strided_and_16_byte_aligned_input(mxq):
    """Rows with a stride wider than the tensor, and a base 16 (not 32)
    bytes past a 32-byte boundary: the 16-byte load path."""
    base = W.mxfp8_random(256, 520, seed=5)
    t = dev_bf16(base)
    check_fp8blk(mxq, np.ascontiguousarray(base[:, :384]), 1, x_dev=t[:, :384])
    check_fp8blk(mxq, np.ascontiguousarray(base[:, 8:392]), 1, x_dev=t[:, 8:392])
    check_fp8blk(mxq, np.ascontiguousarray(base[:, 8:392]), 128, x_dev=t[:, 8:392])


def test_backward_conversion_small(mxq):
    x = W.mxfp8_random(384, 256, seed=6)
    r = mxq.fp8_block_quantize(dev_bf16(x), 1)
    t = mxq.fp8_block_requantize_transpose(r.codes, r.scales)
    torch.cuda.synchronize()
    oc, osc = O.fp8_block_quantize(x, 1)
    ct, st = O.fp8_block_requantize_transpose(oc, osc)
    assert_bytes_equal(host_u8(t.codes), ct, "converted codes")
    assert_bytes_equal(_scales_bits(t.scales), st.view(np.uint32), "converted scales")


@pytest.mark.parametrize("cls", ["boundary", "mixed", "zeros"])
def test_backward_conversion_classes(mxq, cls):
    x = _classes(256, 384)[cls]
    r = mxq.fp8_block_quantize(dev_bf16(x), 1)
    t = mxq.fp8_block_requantize_transpose(r.codes, r.scales)
    torch.cuda.synchronize()
    ct, st = O.fp8_block_requantize_transpose(host_u8(r.codes),
                                              r.scales.cpu().numpy())
    assert_bytes_equal(host_u8(t.codes), ct, f"converted codes [{cls}]")
    assert_bytes_equal(_scales_bits(t.scales), st.view(np.uint32),
                       f"converted scales [{cls}]")


def test_full_size_sampled(mxq):
    """X [8192 x 4096] N(0,1) with outliers: 1x128 tiles of 64 sampled rows,
    every FP32 scale against the closed form amax / 448, and the backward
    conversion of 64 sampled columns, each from its full column of X's
    codes.  The linear layer's weight [8192 x 2048] N(0, 0.02) in 128x128
    blocks is checked whole."""
    M, K = 8192, 4096
    x = W.mxfp8_random(M, K)
    xd = dev_bf16(x)
    r = mxq.fp8_block_quantize(xd, 1)
    t = mxq.fp8_block_requantize_transpose(r.codes, r.scales)
    torch.cuda.synchronize()
    codes = host_u8(r.codes)
    scales = r.scales.cpu().numpy()
    rows = np.union1d(np.random.default_rng(7).choice(M, 64, replace=False), [0, M - 1])
    oc, osc = O.fp8_block_quantize(x[rows], 1)
    assert_bytes_equal(codes[rows], oc, "sampled rows, codes")
    assert_bytes_equal(scales[rows].view(np.uint32), osc.view(np.uint32),
                       "sampled rows, scales")
    amax = np.abs(W.bits_to_f32(x)).reshape(M, K // 128, 128).max(axis=2)
    assert np.array_equal(scales, (amax / np.float32(448.0)).astype(np.float32))
    cols = np.union1d(np.random.default_rng(8).choice(K, 64, replace=False), [0, K - 1])
    ct_all = host_u8(t.codes)
    st_all = t.scales.cpu().numpy()
    for c in cols:
        tile = c // 128
        y = O.fp8_block_dequantize(np.ascontiguousarray(codes[:, tile * 128:(tile + 1) * 128]),
                                   np.ascontiguousarray(scales[:, tile:tile + 1]), 1)
        oc, osc = O.fp8_block_quantize(np.ascontiguousarray(y[:, c - tile * 128][None, :]), 1)
        assert_bytes_equal(ct_all[c][None, :], oc, f"converted column {c}")
        assert_bytes_equal(st_all[c][None, :].view(np.uint32), osc.view(np.uint32),
                           f"converted column {c} scales")
    w = W.linear_weight()
    check_fp8blk(mxq, w, 128)
