"""Buffers that are 16-byte aligned but not 32-byte aligned.

The C ABI asks for 16-byte alignment.  The kernels use 32-byte loads and
stores when every buffer allows them and 16-byte accesses otherwise; these
tests run each entry point on buffers offset by 16 bytes (and rows whose
stride is an odd multiple of 16 bytes) and require the same bytes as the
aligned call."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import assert_bytes_equal, dev_bf16, host_u8

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


def _off16(nbytes, dev="cuda"):
    """A uint8 view of nbytes starting 16 bytes past a 256-byte boundary."""
    buf = torch.zeros(nbytes + 256, dtype=torch.uint8, device=dev)
    base = buf.data_ptr()
    start = (-base) % 256 + 16
    v = buf[start:start + nbytes]
    assert v.data_ptr() % 32 == 16
    return v


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_rowcol_unaligned_outputs(mxq):
    M, K = 256, 384
    x = dev_bf16(W.mxfp8_random(M, K, seed=31))
    ref = mxq.mxfp8_quantize_rowcol(x)
    rc, cc = _off16(M * K), _off16(K * M)
    rs, cs = torch.empty_like(ref.row_scales), torch.empty_like(ref.col_scales_t)
    st = mxq.lib().mxfp8_quantize_rowcol(
        x.data_ptr(), M, K, K, rc.data_ptr(), rs.data_ptr(), cc.data_ptr(),
        cs.data_ptr(), mxq.SCALE_SWIZZLED, _stream())
    assert st == 0
    torch.cuda.synchronize()
    assert_bytes_equal(host_u8(rc).reshape(M, K), host_u8(ref.row_codes), "row codes")
    assert_bytes_equal(host_u8(cc).reshape(K, M), host_u8(ref.col_codes_t), "col codes")
    assert_bytes_equal(host_u8(rs), host_u8(ref.row_scales), "row scales")
    assert_bytes_equal(host_u8(cs), host_u8(ref.col_scales_t), "col scales")


def test_dequant_unaligned_outputs(mxq):
    M, K = 256, 512
    x = dev_bf16(W.mxfp8_random(M, K, seed=32))
    r = mxq.mxfp8_quantize_rowcol(x, colwise=False)
    ref = mxq.dequantize_mxfp8(r.row_codes, r.row_scales)
    y = _off16(M * K * 2)
    assert mxq.lib().dequantize_mxfp8(
        r.row_codes.data_ptr(), r.row_scales.data_ptr(), M, K,
        mxq.SCALE_SWIZZLED, y.data_ptr(), _stream()) == 0
    t = mxq.nvfp4_quantize_per_token(x)
    ref4 = mxq.dequantize_nvfp4(t.codes, t.block_scales, t.scales)
    y4 = _off16(M * K * 2)
    assert mxq.lib().dequantize_nvfp4(
        t.codes.data_ptr(), t.block_scales.data_ptr(), t.scales.data_ptr(),
        mxq.S_PER_ROW, 1, M, K, mxq.SCALE_SWIZZLED, y4.data_ptr(),
        _stream()) == 0
    torch.cuda.synchronize()
    assert_bytes_equal(host_u8(y), host_u8(ref.view(torch.uint8)).reshape(-1),
                       "mxfp8 dequant")
    assert_bytes_equal(host_u8(y4), host_u8(ref4.view(torch.uint8)).reshape(-1),
                       "nvfp4 dequant")


@pytest.mark.parametrize("H", [2048, 4096])
def test_per_token_unaligned_rows_and_scales(mxq, H):
    """x at a 16-byte offset with row stride H + 8 values (rows alternate
    between 32-byte and 16-byte alignment), scales at a 16-byte offset."""
    T = 256
    bits = W.to_bf16_bits(np.random.default_rng(33).standard_normal((T, H)))
    ref = mxq.nvfp4_quantize_per_token(dev_bf16(bits))
    ldx = H + 8
    xb = _off16(T * ldx * 2)
    xv = xb.view(torch.bfloat16).view(T, ldx)
    xv[:, :H] = dev_bf16(bits)
    codes = torch.empty_like(ref.codes)
    sc = _off16(ref.block_scales.numel())
    S = torch.empty_like(ref.scales)
    assert mxq.lib().nvfp4_quantize_per_token(
        xv.data_ptr(), T, H, ldx, codes.data_ptr(), sc.data_ptr(),
        S.data_ptr(), mxq.SCALE_SWIZZLED, _stream()) == 0
    idx = torch.arange(T, dtype=torch.int32, device="cuda").flip(0).contiguous()
    gref = mxq.nvfp4_quantize_per_token_gather(dev_bf16(bits), idx)
    gcodes = torch.empty_like(gref.codes)
    gsc = _off16(gref.block_scales.numel())
    gS = torch.empty_like(gref.scales)
    assert mxq.lib().nvfp4_quantize_per_token_gather(
        xv.data_ptr(), T, H, ldx, idx.data_ptr(), T, gcodes.data_ptr(),
        gsc.data_ptr(), gS.data_ptr(), mxq.SCALE_SWIZZLED, _stream()) == 0
    torch.cuda.synchronize()
    assert_bytes_equal(host_u8(codes), host_u8(ref.codes), "codes")
    assert_bytes_equal(host_u8(sc), host_u8(ref.block_scales), "scales")
    assert torch.equal(S, ref.scales)
    assert_bytes_equal(host_u8(gcodes), host_u8(gref.codes), "gather codes")
    assert_bytes_equal(host_u8(gsc), host_u8(gref.block_scales), "gather scales")
    assert torch.equal(gS, gref.scales)


def test_weights_unaligned_parts_and_scales(mxq):
    """Gate/up parts at 16-byte offsets, scale matrices at a 16-byte
    offset: same bytes as the aligned call."""
    G, F, Hd = 3, 256, 4096
    experts = [W.moe_expert(e, hidden=Hd, ffn=F, seed=9)[:2] for e in range(G)]
    ref = mxq.nvfp4_quantize_weight_shared(
        [[dev_bf16(g), dev_bf16(u)] for g, u in experts])
    keep, ptrs = [], []
    for g, u in experts:
        for part in (g, u):
            b = _off16(part.size * 2)
            b.view(torch.bfloat16).view(part.shape).copy_(dev_bf16(part))
            keep.append(b)
            ptrs.append(b.data_ptr())
    P = (ctypes.c_void_p * len(ptrs))(*ptrs)
    rows = (ctypes.c_int64 * 2)(F, F)
    codes = torch.empty_like(ref.codes)
    sc = _off16(ref.block_scales.numel())
    gS = torch.empty_like(ref.scales)
    L = mxq.lib()
    wsb = int(L.nvfp4_quantize_weight_shared_workspace_size(G))
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    assert L.nvfp4_quantize_weight_shared(
        G, 2, ctypes.cast(P, ctypes.c_void_p), ctypes.cast(rows, ctypes.c_void_p),
        Hd, codes.data_ptr(), sc.data_ptr(), gS.data_ptr(), None,
        mxq.SCALE_SWIZZLED, ws.data_ptr(), wsb, _stream()) == 0
    torch.cuda.synchronize()
    assert_bytes_equal(host_u8(codes), host_u8(ref.codes), "codes")
    assert_bytes_equal(host_u8(sc), host_u8(ref.block_scales).reshape(-1), "scales")
    assert torch.equal(gS, ref.scales)
