"""GPU parity of the tcgen05 block-scaled GEMM consumers.

The reference is the oracle GEMM: float64 accumulation over operands
dequantized exactly from the same codes and scales (MXFP8: E4M3 x 2^k;
NVFP4: E2M1 x E4M3, with the per-token and per-group FP32 scales applied
after the sum).  The kernel accumulates in fp32, so the bar is a relative
Frobenius error of 1e-3, the benchmark spec's tolerance; an error in the scale
layout (the swizzled 128x4 tiles the tensor core reads) shows up as
factor-of-two errors far above it.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import dev_bf16, host_u8

pytestmark = pytest.mark.gpu

TOL = 1e-3


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
    return float(np.linalg.norm(c - ref) / max(np.linalg.norm(ref), 1e-300))


def _mxfp8_case(q, M, K, N, seed, scale_spread=0):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K))
    b = 0.02 * rng.standard_normal((K, N))
    if scale_spread:
        # distinct power-of-two magnitudes per 32-block make every scale
        # byte matter
        a *= np.exp2(rng.integers(-scale_spread, scale_spread, (M, K // 32))
                     ).repeat(32, axis=1)
        b *= np.exp2(rng.integers(-scale_spread, scale_spread, (K // 32, N))
                     ).repeat(32, axis=0)
    A = W.to_bf16_bits(a)
    B = W.to_bf16_bits(b)
    qa = q.mxfp8_quantize_rowcol(dev_bf16(A), rowwise=True, colwise=False)
    qb = q.mxfp8_quantize_rowcol(dev_bf16(B), rowwise=False, colwise=True)
    C = q.gemm_mxfp8(qa.row_codes, qa.row_scales, qb.col_codes_t,
                     qb.col_scales_t)
    torch.cuda.synchronize()
    ac, asc = host_u8(qa.row_codes), O.scale_unswizzle(host_u8(qa.row_scales), M, K // 32)
    bc, bsc = host_u8(qb.col_codes_t), O.scale_unswizzle(host_u8(qb.col_scales_t), N, K // 32)
    ref = O.gemm_mxfp8(ac, asc, bc, bsc)
    return C.cpu().numpy().astype(np.float64), ref


@pytest.mark.parametrize("M,K,N", [(128, 128, 128), (256, 512, 384)])
def test_gemm_mxfp8_small(mxq, M, K, N):
    C, ref = _mxfp8_case(mxq, M, K, N, seed=M + K + N)
    err = rel_fro(C, ref)
    assert err <= TOL, err


def test_gemm_mxfp8_scale_layout(mxq):
    """Per-block magnitudes spread over 2^-6 .. 2^6: a permuted or
    misread scale tile would be off by powers of two."""
    C, ref = _mxfp8_case(mxq, 256, 256, 256, seed=3, scale_spread=6)
    assert rel_fro(C, ref) <= TOL


def _nvfp4_grouped_case(q, rows_per_group, K, N, seed):
    rng = np.random.default_rng(seed)
    G = len(rows_per_group)
    offs = np.concatenate([[0], np.cumsum(rows_per_group)])
    a = rng.standard_normal((int(offs[-1]), K)) * np.exp2(
        rng.integers(-4, 4, (int(offs[-1]), 1)))
    A = W.to_bf16_bits(a)
    Wts = [W.to_bf16_bits(0.02 * rng.standard_normal((N, K))) for _ in range(G)]
    ta = q.nvfp4_quantize_per_token(dev_bf16(A))
    tw = q.nvfp4_quantize_weight_shared([[dev_bf16(w)] for w in Wts])
    C = q.gemm_nvfp4_grouped(ta.codes, ta.block_scales, ta.scales, offs,
                             tw.codes, tw.block_scales, tw.scales)
    torch.cuda.synchronize()
    Mt = int(offs[-1])
    a_sc = O.scale_unswizzle(host_u8(ta.block_scales), Mt, K // 16)
    w_sc = np.stack([O.scale_unswizzle(host_u8(tw.block_scales[g]), N, K // 16)
                     for g in range(G)])
    ref = O.gemm_nvfp4_grouped(host_u8(ta.codes), a_sc, ta.scales.cpu().numpy(),
                               offs, host_u8(tw.codes), w_sc,
                               tw.scales.cpu().numpy())
    return C.cpu().numpy().astype(np.float64), ref


@pytest.mark.parametrize("rows,K,N", [([128], 256, 128),
                                      ([128, 256, 0, 128], 512, 256)])
def test_gemm_nvfp4_grouped_small(mxq, rows, K, N):
    C, ref = _nvfp4_grouped_case(mxq, rows, K, N, seed=sum(rows) + K)
    err = rel_fro(C, ref)
    assert err <= TOL, err


def test_gemm_mxfp8_many_tiles_per_cta(mxq):
    """320 output tiles over at most 152 persistent CTAs: every CTA runs
    two or three tiles through its tensor-memory accumulator, and the
    3-stage K loop wraps the 4-deep operand ring across tiles.
    Every element of C is checked."""
    C, ref = _mxfp8_case(mxq, 2048, 384, 2560, seed=11)
    assert rel_fro(C, ref) <= TOL
    # no tile may be left unwritten or written twice with the wrong data:
    # a per-tile check catches an error hidden by the global norm
    for i in range(0, 2048, 128):
        for j in range(0, 2560, 128):
            assert rel_fro(C[i:i + 128, j:j + 128],
                           ref[i:i + 128, j:j + 128]) <= TOL, (i, j)


def test_gemm_mxfp8_strided_unaligned_c(mxq):
    """C with a row stride of N + 4 floats and its base 16 bytes past a
    32-byte boundary (the epilogue's 16-byte store path instead of whole
    32-byte sectors), N = 384 so the second column tile holds 128 valid
    columns: C is byte-identical to the contiguous call's, and every byte
    around it keeps its sentinel."""
    M, K, N = 256, 256, 384
    rng = np.random.default_rng(21)
    A = W.to_bf16_bits(rng.standard_normal((M, K)))
    B = W.to_bf16_bits(0.02 * rng.standard_normal((K, N)))
    qa = mxq.mxfp8_quantize_rowcol(dev_bf16(A), rowwise=True, colwise=False)
    qb = mxq.mxfp8_quantize_rowcol(dev_bf16(B), rowwise=False, colwise=True)
    ref = mxq.gemm_mxfp8(qa.row_codes, qa.row_scales, qb.col_codes_t,
                         qb.col_scales_t)
    ldc = N + 4
    buf = torch.full((M * ldc + 8,), -7.0, dtype=torch.float32, device="cuda")
    C = buf[4:4 + M * ldc]
    assert C.data_ptr() % 32 == 16
    st = mxq.lib().mxq_gemm_mxfp8(
        qa.row_codes.data_ptr(), qa.row_scales.data_ptr(),
        qb.col_codes_t.data_ptr(), qb.col_scales_t.data_ptr(), M, N, K,
        C.data_ptr(), ldc, torch.cuda.current_stream().cuda_stream)
    assert st == 0, mxq.status_string(st)
    torch.cuda.synchronize()
    got = C.view(M, ldc)
    assert torch.equal(got[:, :N].contiguous().view(torch.int32),
                       ref.view(torch.int32))
    assert bool((got[:, N:] == -7.0).all())
    assert bool((buf[:4] == -7.0).all()) and bool((buf[4 + M * ldc:] == -7.0).all())


def test_gemm_nvfp4_grouped_many_tiles_per_cta(mxq):
    """Ragged expert groups (one empty) giving 38 row tiles x 8 column
    tiles = 304 tiles, K = 512 (two stages per tile): several tiles per
    persistent CTA, tiles that straddle group boundaries in the schedule."""
    rows = [128 * 7, 0, 128 * 13, 256, 128 * 5, 128 * 11]
    C, ref = _nvfp4_grouped_case(mxq, rows, 512, 1024, seed=5)
    assert rel_fro(C, ref) <= TOL
    for i in range(0, C.shape[0], 128):
        assert rel_fro(C[i:i + 128], ref[i:i + 128]) <= TOL, i


def test_gemm_mxfp8_full_size_sampled(mxq):
    """A [2048 x 2048] N(0,1) times B [2048 x 8192] N(0, 0.02), B consumed
    through its columnwise copy; 256 sampled rows of C vs the oracle."""
    M, K, N = 2048, 2048, 8192
    A, B = W.gemm_mxfp8_inputs(M, K, N)
    qa = mxq.mxfp8_quantize_rowcol(dev_bf16(A), rowwise=True, colwise=False)
    qb = mxq.mxfp8_quantize_rowcol(dev_bf16(B), rowwise=False, colwise=True)
    C = mxq.gemm_mxfp8(qa.row_codes, qa.row_scales, qb.col_codes_t,
                       qb.col_scales_t)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(0).choice(M, 256, replace=False))
    ac = host_u8(qa.row_codes)[rows]
    asc = O.scale_unswizzle(host_u8(qa.row_scales), M, K // 32)[rows]
    bc = host_u8(qb.col_codes_t)
    bsc = O.scale_unswizzle(host_u8(qb.col_scales_t), N, K // 32)
    ref = O.gemm_mxfp8(ac, asc, bc, bsc)
    got = C.cpu().numpy()[rows].astype(np.float64)
    assert rel_fro(got, ref) <= TOL


def test_gemm_nvfp4_grouped_moe_sampled(mxq):
    """4096 tokens (hidden 2048), top-8 of 128 experts, gate/up weights
    [1536 x 2048] per expert: tokens gathered by expert into 128-row-padded
    groups, quantized per token, multiplied by each expert's NVFP4 weight
    with both FP32 scales in the epilogue.  Four experts are checked row by
    row against the oracle."""
    E, H, F = 128, 2048, 768
    tokens = W.gemm_tokens(4096, H)
    route = W.topk_routing(4096, E, 8)
    rows_by_e = [np.nonzero((route == e).any(axis=1))[0] for e in range(E)]
    sizes = [len(r) for r in rows_by_e]
    padded = [((s + 127) // 128) * 128 for s in sizes]
    offs = np.concatenate([[0], np.cumsum(padded)])
    gathered = np.zeros((int(offs[-1]), H), np.uint16)
    for e in range(E):
        gathered[offs[e]:offs[e] + sizes[e]] = tokens[rows_by_e[e]]
    ta = mxq.nvfp4_quantize_per_token(dev_bf16(gathered))
    experts = [W.moe_expert(e, hidden=H, ffn=F) for e in range(E)]
    tw = mxq.nvfp4_quantize_weight_shared(
        [[dev_bf16(g), dev_bf16(u)] for g, u, _ in experts])
    del experts
    C = mxq.gemm_nvfp4_grouped(ta.codes, ta.block_scales, ta.scales, offs,
                               tw.codes, tw.block_scales, tw.scales)
    torch.cuda.synchronize()
    Mt = int(offs[-1])
    a_codes = host_u8(ta.codes)
    a_sc = O.scale_unswizzle(host_u8(ta.block_scales), Mt, H // 16)
    a_S = ta.scales.cpu().numpy()
    Cn = C.cpu().numpy()
    for e in (0, 17, 64, 127):
        r0, r1 = int(offs[e]), int(offs[e]) + sizes[e]
        w_sc = O.scale_unswizzle(host_u8(tw.block_scales[e]), 2 * F, H // 16)
        ref = O.gemm_nvfp4_grouped(a_codes[r0:r1], a_sc[r0:r1], a_S[r0:r1],
                                   [0, r1 - r0], host_u8(tw.codes[e])[None],
                                   w_sc[None], tw.scales.cpu().numpy()[e:e + 1])
        assert rel_fro(Cn[r0:r1].astype(np.float64), ref) <= TOL, e
