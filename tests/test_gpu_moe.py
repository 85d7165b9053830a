"""GPU parity of the MoE expert forward up to the activation: routing
gather fused into the per-token NVFP4 quantizer, and the grouped gate/up
GEMM with SwiGLU in the epilogue ("Miles: end-to-end MXFP8 and per-token
NVFP4 RL", NVFP4 recipe section: SwiGLU MoE layers fuse gate and up into one
GEMM under one FP32 weight scale; experiments section: per-token scale in
the GEMM epilogue).

The gather quantizer is byte-exact against the oracle applied to the
gathered rows.  The SwiGLU GEMM writes bf16: the kernel accumulates in fp32
and evaluates silu with a fast exponential and divide (relative error below
2^-20), so each output is within
one bf16 ulp (2^-7 relative) of the float64 oracle rounded the same way,
except where the value is tiny against the row's scale (cancellation in the
fp32 sums): an absolute floor of 1e-3 of the output's RMS covers those.
The relative Frobenius error stays below 4e-3 (bf16 rounding alone is about
1.6e-3).
"""
import numpy as np
import pytest
import torch

import oracle as O
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


def _bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def _check_h(got: np.ndarray, ref: np.ndarray, what: str):
    floor = 1e-3 * np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    bad = err > 2.0 ** -7 * np.abs(ref) + floor
    assert not bad.any(), (what, int(bad.sum()), float(err[bad].max()))
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert fro <= 4e-3, (what, fro)


@pytest.mark.parametrize("layout", ["swizzled", "linear"])
def test_gather_quantize_bit_exact(mxq, layout):
    """Repeated, padding (-1) and out-of-range indices; H = 2048."""
    rng = np.random.default_rng(21)
    T_src, H = 300, 2048
    x = W.to_bf16_bits(rng.standard_t(4, (T_src, H)).astype(np.float32))
    idx = rng.integers(0, T_src, 517).astype(np.int32)
    idx[::7] = -1
    idx[5] = T_src + 3
    idx[6] = idx[8]
    out = mxq.nvfp4_quantize_per_token_gather(
        dev_bf16(x), torch.from_numpy(idx).cuda(), scale_layout=layout)
    torch.cuda.synchronize()
    g = O.gather_rows(x, idx)
    codes, sc, S = O.nvfp4_quantize_per_token(g)
    assert_bytes_equal(host_u8(out.codes), codes, "codes")
    got_sc = host_u8(out.block_scales)
    if layout == "swizzled":
        got_sc = O.scale_unswizzle(got_sc, len(idx), H // 16)
    else:
        got_sc = got_sc.reshape(len(idx), H // 16)
    assert_bytes_equal(got_sc, sc, "block scales")
    assert np.array_equal(out.scales.cpu().numpy().view(np.uint32),
                          S.view(np.uint32))
    assert np.all(S[idx < 0] == 0)


def _moe_case(q, rows_per_group, F, K, seed):
    rng = np.random.default_rng(seed)
    G = len(rows_per_group)
    T_src = 512
    x = W.to_bf16_bits(rng.standard_normal((T_src, K)).astype(np.float32))
    idx, offs = [], [0]
    for r in rows_per_group:
        n_real = max(0, r - rng.integers(0, 20)) if r else 0
        idx.append(np.concatenate([rng.integers(0, T_src, n_real),
                                   np.full(r - n_real, -1)]))
        offs.append(offs[-1] + r)
    idx = np.concatenate(idx).astype(np.int32)
    offs = np.array(offs, np.int64)
    Wg = [W.to_bf16_bits(0.05 * rng.standard_normal((F, K)).astype(np.float32))
          for _ in range(G)]
    Wu = [W.to_bf16_bits(0.05 * rng.standard_normal((F, K)).astype(np.float32))
          for _ in range(G)]
    ta = q.nvfp4_quantize_per_token_gather(dev_bf16(x),
                                           torch.from_numpy(idx).cuda())
    tw = q.nvfp4_quantize_weight_shared(
        [[dev_bf16(Wg[g]), dev_bf16(Wu[g])] for g in range(G)])
    h = q.moe_gate_up_swiglu(ta.codes, ta.block_scales, ta.scales, offs,
                             tw.codes, tw.block_scales, tw.scales)
    torch.cuda.synchronize()
    Mt = int(offs[-1])
    a_sc = O.scale_unswizzle(host_u8(ta.block_scales), Mt, K // 16)
    w_sc = np.stack([O.scale_unswizzle(host_u8(tw.block_scales[g]), 2 * F,
                                       K // 16) for g in range(G)])
    ref = O.moe_gate_up_swiglu(host_u8(ta.codes), a_sc,
                               ta.scales.cpu().numpy(), offs,
                               host_u8(tw.codes), w_sc,
                               tw.scales.cpu().numpy())
    return _bf16_to_f64(h), ref, offs


@pytest.mark.parametrize("rows,F,K", [([128], 128, 256),
                                      ([128, 256, 0, 128], 256, 512),
                                      ([384, 128, 256], 384, 1024)])
def test_moe_swiglu_small(mxq, rows, F, K):
    """Ragged groups (one empty), F with odd and even tile counts, several
    stages per tile."""
    got, ref, _ = _moe_case(mxq, rows, F, K, seed=sum(rows) + F + K)
    _check_h(got, ref, f"rows={rows} F={F} K={K}")


def test_moe_swiglu_strided_unaligned_h(mxq):
    """h with a row stride of F + 8 bf16 and its base 16 bytes past a
    32-byte boundary (the epilogue's 16-byte store path): h is
    byte-identical to the contiguous call's, and every byte around it keeps
    its sentinel."""
    rng = np.random.default_rng(31)
    F, K, rows = 256, 512, [128, 256]
    T_src = 256
    x = W.to_bf16_bits(rng.standard_normal((T_src, K)).astype(np.float32))
    idx = rng.integers(0, T_src, sum(rows)).astype(np.int32)
    offs = np.array([0, rows[0], rows[0] + rows[1]], np.int64)
    Wg = [W.to_bf16_bits(0.05 * rng.standard_normal((F, K)).astype(np.float32))
          for _ in rows]
    Wu = [W.to_bf16_bits(0.05 * rng.standard_normal((F, K)).astype(np.float32))
          for _ in rows]
    ta = mxq.nvfp4_quantize_per_token_gather(dev_bf16(x),
                                             torch.from_numpy(idx).cuda())
    tw = mxq.nvfp4_quantize_weight_shared(
        [[dev_bf16(Wg[g]), dev_bf16(Wu[g])] for g in range(len(rows))])
    ref = mxq.moe_gate_up_swiglu(ta.codes, ta.block_scales, ta.scales, offs,
                                 tw.codes, tw.block_scales, tw.scales)
    M = int(offs[-1])
    ldh = F + 8
    buf = torch.full((M * ldh + 16,), 12345, dtype=torch.int16, device="cuda")
    h = buf[8:8 + M * ldh]
    assert h.data_ptr() % 32 == 16
    import ctypes
    off_arr = (ctypes.c_int64 * len(offs))(*[int(v) for v in offs])
    st = mxq.lib().mxq_moe_gate_up_swiglu_nvfp4(
        ta.codes.data_ptr(), ta.block_scales.data_ptr(), ta.scales.data_ptr(),
        ctypes.cast(off_arr, ctypes.c_void_p), len(rows), tw.codes.data_ptr(),
        tw.block_scales.data_ptr(), tw.scales.data_ptr(), F, K, h.data_ptr(),
        ldh, torch.cuda.current_stream().cuda_stream)
    assert st == 0, mxq.status_string(st)
    torch.cuda.synchronize()
    got = h.view(M, ldh)
    assert torch.equal(got[:, :F].contiguous(), ref.view(torch.int16))
    assert bool((got[:, F:] == 12345).all())
    assert bool((buf[:8] == 12345).all()) and bool((buf[8 + M * ldh:] == 12345).all())


def test_moe_swiglu_many_tiles_per_cta(mxq):
    """40 row tiles x 6 column tiles over the persistent grid: every CTA runs
    several tiles through the single accumulator."""
    rows = [128 * 9, 128 * 3, 0, 128 * 17, 128 * 11]
    got, ref, offs = _moe_case(mxq, rows, 768, 512, seed=77)
    for i in range(0, got.shape[0], 128):
        _check_h(got[i:i + 128], ref[i:i + 128], f"rows {i}")


def test_moe_forward_full_size_sampled(mxq):
    """4096 tokens (hidden 2048) routed top-8 over 128 experts, gate/up
    [768 x 2048] each: gather-quantize, then gate/up GEMM + SwiGLU; five
    experts checked against the oracle."""
    E, H, F = 128, 2048, 768
    tokens = W.gemm_tokens(4096, H)
    route = W.topk_routing(4096, E, 8)
    idx, offs, sizes = W.expert_gather_index(route, E)
    ta = mxq.nvfp4_quantize_per_token_gather(dev_bf16(tokens),
                                             torch.from_numpy(idx).cuda())
    experts = [W.moe_expert(e, hidden=H, ffn=F) for e in range(E)]
    tw = mxq.nvfp4_quantize_weight_shared(
        [[dev_bf16(g), dev_bf16(u)] for g, u, _ in experts])
    del experts
    h = mxq.moe_gate_up_swiglu(ta.codes, ta.block_scales, ta.scales, offs,
                               tw.codes, tw.block_scales, tw.scales)
    torch.cuda.synchronize()
    Mt = int(offs[-1])
    a_codes = host_u8(ta.codes)
    a_sc = O.scale_unswizzle(host_u8(ta.block_scales), Mt, H // 16)
    a_S = ta.scales.cpu().numpy()
    hn = _bf16_to_f64(h)
    for e in (0, 5, 63, 100, 127):
        r0 = int(offs[e])
        r1 = r0 + int(sizes[e])
        w_sc = O.scale_unswizzle(host_u8(tw.block_scales[e]), 2 * F, H // 16)
        ref = O.moe_gate_up_swiglu(a_codes[r0:r1], a_sc[r0:r1], a_S[r0:r1],
                                   [0, r1 - r0], host_u8(tw.codes[e])[None],
                                   w_sc[None],
                                   tw.scales.cpu().numpy()[e:e + 1])
        _check_h(hn[r0:r1], ref, f"expert {e}")
        assert np.all(hn[r1:int(offs[e + 1])] == 0), "padding rows"


# --------------------------------------------------------------------------
# The routing gather inside the GEMM's operand load: the unique tokens are
# quantized once (per-token quantization does not depend on the batch) and
# each routed row is gathered by the GEMM.  The outputs must be the bytes of
# the path that writes the gathered operand first.
# --------------------------------------------------------------------------
def _gather_case(q, T_src, H, F, E, k, seed):
    tokens = W.gemm_tokens(T_src, H, seed=seed)
    route = W.topk_routing(T_src, E, k, seed=seed)
    idx, offs, _ = W.expert_gather_index(route, E)
    x = dev_bf16(tokens)
    idx_dev = torch.from_numpy(idx).cuda()
    experts = [W.moe_expert(e, hidden=H, ffn=F, seed=seed) for e in range(E)]
    tw = q.nvfp4_quantize_weight_shared(
        [[dev_bf16(g), dev_bf16(u)] for g, u, _ in experts])
    return x, idx_dev, offs, tw


@pytest.mark.parametrize("T_src,H,F,E,k", [(300, 512, 128, 5, 2),
                                           (1000, 1024, 384, 16, 4),
                                           (4096, 2048, 768, 128, 8)])
def test_gather_in_gemm_matches_materialized(mxq, T_src, H, F, E, k):
    q = mxq
    x, idx, offs, tw = _gather_case(q, T_src, H, F, E, k, seed=T_src + E)
    ref_a = q.nvfp4_quantize_per_token_gather(x, idx)
    ref_h = q.moe_gate_up_swiglu(ref_a.codes, ref_a.block_scales, ref_a.scales,
                                 offs, tw.codes, tw.block_scales, tw.scales)
    ref_c = q.gemm_nvfp4_grouped(ref_a.codes, ref_a.block_scales, ref_a.scales,
                                 offs, tw.codes, tw.block_scales, tw.scales)
    xq = q.nvfp4_quantize_per_token(x, "linear")
    h = q.moe_gate_up_swiglu_gather(xq, idx, offs, tw.codes, tw.block_scales,
                                    tw.scales)
    c = q.gemm_nvfp4_grouped_gather(xq, idx, offs, tw.codes, tw.block_scales,
                                    tw.scales)
    torch.cuda.synchronize()
    assert q.get_last_error() == q.MXQ_OK
    assert torch.equal(h.view(torch.int16), ref_h.view(torch.int16))
    assert torch.equal(c.view(torch.int32), ref_c.view(torch.int32))


def test_gather_in_gemm_index_edges(mxq):
    """Padding (-1), out-of-range and repeated indices, the last token."""
    q = mxq
    T_src, H, F = 200, 512, 256
    x = dev_bf16(W.gemm_tokens(T_src, H, seed=41))
    rows = [256, 128]
    idx = np.arange(384, dtype=np.int32) % T_src
    idx[5::9] = -1
    idx[7] = T_src
    idx[11] = T_src - 1
    idx[200:260] = 3
    offs = np.array([0, 256, 384])
    experts = [W.moe_expert(e, hidden=H, ffn=F, seed=41) for e in range(2)]
    tw = q.nvfp4_quantize_weight_shared(
        [[dev_bf16(g), dev_bf16(u)] for g, u, _ in experts])
    idx_dev = torch.from_numpy(idx).cuda()
    ref_a = q.nvfp4_quantize_per_token_gather(x, idx_dev)
    ref_h = q.moe_gate_up_swiglu(ref_a.codes, ref_a.block_scales, ref_a.scales,
                                 offs, tw.codes, tw.block_scales, tw.scales)
    xq = q.nvfp4_quantize_per_token(x, "linear")
    h = q.moe_gate_up_swiglu_gather(xq, idx_dev, offs, tw.codes,
                                    tw.block_scales, tw.scales)
    torch.cuda.synchronize()
    assert torch.equal(h.view(torch.int16), ref_h.view(torch.int16))
    pad = (idx < 0) | (idx >= T_src)
    assert torch.all(h[torch.from_numpy(pad).cuda()].view(torch.int16) == 0)
