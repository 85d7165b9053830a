"""GPU parity of the dequantized-backward GEMM without a bf16 copy of the
quantized operand ("Miles: end-to-end MXFP8 and per-token NVFP4 RL",
backward-mode section: BF16 backward GEMMs consume BF16 dequantizations of
the exact forward operands).  The MXFP8 operand is made by the oracle
(codes and scales of B's columnwise copy), so the GEMM's inputs do not come
from the GPU quantizer; the product is compared with the float64 oracle by
relative Frobenius error (fp32 accumulation: about 1e-6; the bar is 1e-4,
inside the 1e-3 of the GEMM contract)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import dev_bf16

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


def rel_fro(c, ref):
    return np.linalg.norm(c - ref) / max(np.linalg.norm(ref), 1e-300)


def _case(q, M, K, N, seed, rows=None):
    rng = np.random.default_rng(seed)
    A = W.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    Bw = W.to_bf16_bits((0.02 * rng.standard_normal((K, N)) *
                         10.0 ** rng.uniform(-3, 3, (1, N))).astype(np.float32))
    bc, bs = O.mxfp8_quantize_colwise(Bw)          # B^T [N x K], logical scales
    C = q.gemm_bf16_mxfp8(dev_bf16(A), torch.from_numpy(bc).cuda(),
                          torch.from_numpy(O.scale_swizzle(bs)).cuda())
    torch.cuda.synchronize()
    assert q.get_last_error() == q.MXQ_OK
    got = C.cpu().numpy().astype(np.float64)
    sel = np.arange(M) if rows is None else rows
    ref = O.gemm_bf16_mxfp8(A[sel], bc, bs)
    err = rel_fro(got[sel], ref)
    assert err <= 1e-4, err
    return err


@pytest.mark.parametrize("M,K,N", [(128, 64, 128), (128, 128, 256),
                                   (384, 512, 512), (256, 1024, 384)])
def test_small(mxq, M, K, N):
    _case(mxq, M, K, N, seed=M + K + N)


def test_linear_dgrad_shape(mxq):
    """The linear layer (2048, 2048) -> 8192 of the memory section, data
    gradient: dX [2048 x 2048] = dY [2048 x 8192] x W, W's columnwise copy
    as B^T [2048 x 8192]; 64 sampled rows against the oracle."""
    rows = np.union1d(np.random.default_rng(3).choice(2048, 62, replace=False),
                      [0, 2047])
    _case(mxq, 2048, 8192, 2048, seed=9, rows=rows)


def test_in_smem_dequantization_exact(mxq):
    """A = I (bf16 ones on the diagonal): every C[m, n] is one product
    1 x Bq[m, n] plus zeros, so C must equal the oracle's bf16
    dequantization of B bit for bit -- a check of the operand the tensor
    core read, value by value.  Every E4M3 code but the NaN pair, scales
    from 2^-117 to 2^119 (bf16-normal products, no overflow), with rows
    pinned on both sides of the one-multiply limit (exponent byte 134/135)
    and at the ends of the range."""
    M = K = 256
    N = 384
    rng = np.random.default_rng(21)
    codes = rng.integers(0, 256, (N, K), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x00
    codes[4, :254] = np.setdiff1d(np.arange(256), [0x7F, 0xFF]).astype(np.uint8)
    scales = rng.integers(10, 247, (N, K // 32), dtype=np.uint8)
    scales[0], scales[1], scales[2], scales[3] = 134, 135, 10, 246
    # NaN sources: the E8M0 NaN byte on row 5, an E4M3 NaN code on row 6;
    # with A = I every row of C sums over them, so columns 5 and 6 of C are
    # NaN throughout
    scales[5, 2] = 0xFF
    codes[6, 77] = 0x7F
    A = np.where(np.eye(M, K, dtype=bool), 0x3F80, 0).astype(np.uint16)
    C = mxq.gemm_bf16_mxfp8(dev_bf16(A), torch.from_numpy(codes).cuda(),
                            torch.from_numpy(O.scale_swizzle(scales)).cuda())
    torch.cuda.synchronize()
    assert mxq.get_last_error() == mxq.MXQ_OK
    want = W.bits_to_f32(O.mxfp8_dequantize(codes, scales)).T
    assert np.isnan(want[64:96, 5]).all() and np.isnan(want[77, 6])
    got = C.cpu().numpy()
    assert np.isnan(got[:, 5:7]).all()
    got[:, 5:7] = want[:, 5:7] = 0
    bad = np.argwhere(got != want)
    assert bad.size == 0, (len(bad), bad[:5], got[tuple(bad[0])],
                           want[tuple(bad[0])])


def test_strided_a_and_wide_c(mxq):
    """A as a column slice of a wider matrix (lda = K + 64) and C written
    with ldc = N + 32 through the C ABI: the product lands in C's first N
    columns, the 32 padding columns keep their sentinel."""
    M, K, N = 256, 512, 256
    rng = np.random.default_rng(17)
    wide = W.to_bf16_bits(rng.standard_normal((M, K + 64)).astype(np.float32))
    A = np.ascontiguousarray(wide[:, :K])
    Bw = W.to_bf16_bits((0.05 * rng.standard_normal((K, N))).astype(np.float32))
    bc, bs = O.mxfp8_quantize_colwise(Bw)
    a_dev = dev_bf16(wide)[:, :K]
    assert a_dev.stride(0) == K + 64
    codes = torch.from_numpy(bc).cuda()
    scales = torch.from_numpy(O.scale_swizzle(bs)).cuda()
    ldc = N + 32
    C = torch.full((M, ldc), -7.0, dtype=torch.float32, device="cuda")
    st = mxq.lib().mxq_gemm_bf16_mxfp8(a_dev.data_ptr(), a_dev.stride(0),
                                        codes.data_ptr(), scales.data_ptr(),
                                        M, N, K, C.data_ptr(), ldc,
                                        torch.cuda.current_stream().cuda_stream)
    assert st == mxq.MXQ_OK
    torch.cuda.synchronize()
    assert mxq.get_last_error() == mxq.MXQ_OK
    got = C.cpu().numpy()
    assert np.all(got[:, N:] == -7.0)
    ref = O.gemm_bf16_mxfp8(A, bc, bs)
    assert rel_fro(got[:, :N].astype(np.float64), ref) <= 1e-4
    # the binding passes the slice's row stride as lda
    C2 = mxq.gemm_bf16_mxfp8(a_dev, codes, scales)
    torch.cuda.synchronize()
    assert np.array_equal(C2.cpu().numpy(), got[:, :N])
