"""Guard bands around every output buffer (the stand-in for a memory checker,
which this GPU pool does not offer).

Each output of each C-ABI entry point is placed inside a larger device
buffer whose 4 KiB bands before and after it hold 0xA5.  The calls run on
ragged and tail shapes -- partial 128-row scale tiles, K = 48 (a padding
scale column), single rows, a 32-row tail, N = 128 mod 256 for the GEMMs --
and the bands must be untouched afterwards, so a kernel that writes past
either end of any output is caught.  The bytes between the bands must equal
the outputs of the same call through the Python binding (fresh buffers).
Every test runs twice: with each output 32-byte aligned, and with each
output 16 bytes past a 32-byte boundary (the kernels' 16-byte store paths).
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu

BAND = 4096
CANARY = 0xA5
SHIFT = 0            # bytes past a 32-byte boundary for every output


@pytest.fixture(params=[0, 16], ids=["aligned32", "shift16"], autouse=True)
def _output_shift(request):
    global SHIFT
    SHIFT = request.param
    yield
    SHIFT = 0


@pytest.fixture(scope="module")
def mxq():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from nvfp4_quantizers_gb300 import build
    build.build()
    import nvfp4_quantizers_gb300 as q
    q.lib()
    return q


class Guarded:
    """An output of `nbytes` bytes inside a canary-filled buffer."""

    def __init__(self, nbytes):
        self.n = int(nbytes)
        self.lo = BAND + SHIFT
        self.buf = torch.full((self.lo + self.n + BAND,), CANARY,
                              dtype=torch.uint8, device="cuda")
        assert (self.buf.data_ptr() + self.lo) % 32 == SHIFT

    @property
    def ptr(self):
        return self.buf.data_ptr() + self.lo

    def body(self):
        return self.buf[self.lo:self.lo + self.n]

    def check(self, what):
        torch.cuda.synchronize()
        lo = self.buf[:self.lo].cpu().numpy()
        hi = self.buf[self.lo + self.n:].cpu().numpy()
        bad_lo = np.nonzero(lo != CANARY)[0]
        bad_hi = np.nonzero(hi != CANARY)[0]
        assert bad_lo.size == 0, f"{what}: {bad_lo.size} bytes written before the buffer (last at -{self.lo - bad_lo[-1]})"
        assert bad_hi.size == 0, f"{what}: {bad_hi.size} bytes written after the buffer (first at +{bad_hi[0]})"


def same(g: Guarded, t: torch.Tensor, what):
    """The guarded body equals tensor t's bytes."""
    tb = t.contiguous().view(torch.uint8).reshape(-1)
    assert tb.numel() == g.n, f"{what}: size {g.n} != {tb.numel()}"
    assert torch.equal(g.body(), tb), f"{what}: bytes differ from the binding's"


def stream():
    return torch.cuda.current_stream().cuda_stream


def ok(q, st, what):
    assert st == q.MXQ_OK, f"{what}: {q.status_string(st)}"


@pytest.mark.parametrize("lay", ["swizzled", "linear"])
@pytest.mark.parametrize("M,K", [(32, 32), (96, 160), (160, 96), (288, 2080)])
def test_guard_mxfp8_rowcol_and_dequant(mxq, lay, M, K):
    q = mxq
    L = q.lib()
    lc = q._lib._layout(lay)
    x = dev_bf16(W.mxfp8_random(M, K, seed=M + K))
    ref = q.mxfp8_quantize_rowcol(x, scale_layout=lay)
    rc, cc = Guarded(M * K), Guarded(M * K)
    rs, cs = Guarded(q.scale_bytes(M, K // 32, lay)), Guarded(q.scale_bytes(K, M // 32, lay))
    ok(q, L.mxfp8_quantize_rowcol(x.data_ptr(), M, K, K, rc.ptr, rs.ptr, cc.ptr,
                                  cs.ptr, lc, stream()), "rowcol")
    for g, t, nm in ((rc, ref.row_codes, "row codes"), (rs, ref.row_scales, "row scales"),
                     (cc, ref.col_codes_t, "col codes"), (cs, ref.col_scales_t, "col scales")):
        g.check(nm)
        same(g, t, nm)
    for nm, c, s, rows, cols in (("row", ref.row_codes, ref.row_scales, M, K),
                                 ("col", ref.col_codes_t, ref.col_scales_t, K, M)):
        y = Guarded(rows * cols * 2)
        ok(q, L.dequantize_mxfp8(c.data_ptr(), s.data_ptr(), rows, cols, lc, y.ptr,
                                 stream()), "dequant")
        y.check(f"{nm} dequant")
        same(y, q.dequantize_mxfp8(c, s, lay), f"{nm} dequant")


@pytest.mark.parametrize("lay", ["swizzled", "linear"])
@pytest.mark.parametrize("T,H", [(1, 48), (31, 48), (129, 2064), (160, 4096),
                                 (3, 20000)])
def test_guard_nvfp4_per_token_and_dequant(mxq, lay, T, H):
    q = mxq
    L = q.lib()
    lc = q._lib._layout(lay)
    x = dev_bf16(W.ragged_tokens([T], H=H, seed=T))
    ref = q.nvfp4_quantize_per_token(x, lay)
    c, s, S = Guarded(T * H // 2), Guarded(q.scale_bytes(T, H // 16, lay)), Guarded(4 * T)
    ok(q, L.nvfp4_quantize_per_token(x.data_ptr(), T, H, H, c.ptr, s.ptr, S.ptr, lc,
                                     stream()), "per-token")
    for g, t, nm in ((c, ref.codes, "codes"), (s, ref.block_scales, "scales"),
                     (S, ref.scales, "S")):
        g.check(nm)
        same(g, t, nm)
    y = Guarded(T * H * 2)
    ok(q, L.dequantize_nvfp4(ref.codes.data_ptr(), ref.block_scales.data_ptr(),
                             ref.scales.data_ptr(), q.S_PER_ROW, 1, T, H, lc, y.ptr,
                             stream()), "dequant")
    y.check("dequant")
    same(y, q.dequantize_nvfp4(ref.codes, ref.block_scales, ref.scales, lay), "dequant")
    # with the pretraining recipe's transform and stochastic rounding
    if H % 16 == 0 and H <= 8192:
        for fl in (q.NVFP4_RHT, q.NVFP4_RHT | q.NVFP4_SR):
            ref2 = q.nvfp4_quantize_per_token_rht_sr(x, 7, fl, lay)
            c2, s2, S2 = Guarded(T * H // 2), Guarded(q.scale_bytes(T, H // 16, lay)), Guarded(4 * T)
            ok(q, L.nvfp4_quantize_per_token_rht_sr(
                x.data_ptr(), T, H, H, ctypes.c_uint64(7), fl, c2.ptr, s2.ptr, S2.ptr,
                lc, stream()), "rht/sr")
            for g, t, nm in ((c2, ref2.codes, "rht codes"), (s2, ref2.block_scales, "rht scales"),
                             (S2, ref2.scales, "rht S")):
                g.check(nm)
                same(g, t, nm)


def test_guard_nvfp4_gather(mxq):
    q = mxq
    L = q.lib()
    x = dev_bf16(W.ragged_tokens([200], H=512, seed=4))
    idx = torch.tensor([5, -1, 199, 0, 7, 200, 3] * 19 + [1], dtype=torch.int32,
                       device="cuda")
    T = idx.numel()
    ref = q.nvfp4_quantize_per_token_gather(x, idx)
    c, s, S = Guarded(T * 256), Guarded(q.scale_bytes(T, 32)), Guarded(4 * T)
    ok(q, L.nvfp4_quantize_per_token_gather(x.data_ptr(), 200, 512, 512, idx.data_ptr(),
                                            T, c.ptr, s.ptr, S.ptr, 1, stream()), "gather")
    for g, t, nm in ((c, ref.codes, "codes"), (s, ref.block_scales, "scales"),
                     (S, ref.scales, "S")):
        g.check(nm)
        same(g, t, nm)


@pytest.mark.parametrize("lay", ["swizzled", "linear"])
@pytest.mark.parametrize("rows,K,G", [((100, 60), 48, 3), ((768, 768), 2048, 2),
                                      ((2048,), 768, 2), ((33,), 4096, 3),
                                      ((77, 30), 640, 3)])
def test_guard_nvfp4_weights_and_dequant(mxq, lay, rows, K, G):
    q = mxq
    L = q.lib()
    lc = q._lib._layout(lay)
    rng = np.random.default_rng(sum(rows) + K)
    groups = [[dev_bf16(W.to_bf16_bits(rng.standard_normal((r, K)) * (g + 1)))
               for r in rows] for g in range(G)]
    ref = q.nvfp4_quantize_weight_shared(groups, scale_layout=lay)
    R = sum(rows)
    P = len(rows)
    sb = q.scale_bytes(R, K // 16, lay)
    c, s, S = Guarded(G * R * K // 2), Guarded(G * sb), Guarded(4 * G)
    wsb = int(L.nvfp4_quantize_weight_shared_workspace_size(G))
    ws = Guarded(wsb)
    ptrs = (ctypes.c_void_p * (G * P))(*[t.data_ptr() for g in groups for t in g])
    rws = (ctypes.c_int64 * P)(*rows)
    ok(q, L.nvfp4_quantize_weight_shared(G, P, ctypes.cast(ptrs, ctypes.c_void_p),
                                         ctypes.cast(rws, ctypes.c_void_p), K, c.ptr,
                                         s.ptr, S.ptr, None, lc, ws.ptr, wsb, stream()),
       "weights")
    for g, t, nm in ((c, ref.codes, "codes"), (s, ref.block_scales, "scales"),
                     (S, ref.scales, "S")):
        g.check(nm)
        same(g, t, nm)
    ws.check("workspace")
    y = Guarded(G * R * K * 2)
    ok(q, L.dequantize_nvfp4(ref.codes.data_ptr(), ref.block_scales.data_ptr(),
                             ref.scales.data_ptr(), q.S_PER_BATCH, G, R, K, lc, y.ptr,
                             stream()), "dequant")
    y.check("dequant")
    same(y, q.dequantize_nvfp4(ref.codes, ref.block_scales, ref.scales, lay), "dequant")


@pytest.mark.parametrize("rows,cols,br", [(1, 128, 1), (129, 384, 1), (256, 1152, 128),
                                          (128, 128, 128)])
def test_guard_fp8_block(mxq, rows, cols, br):
    q = mxq
    L = q.lib()
    x = dev_bf16(W.mxfp8_random(rows, cols, seed=rows + cols))
    ref = q.fp8_block_quantize(x, br)
    c, s = Guarded(rows * cols), Guarded(4 * (rows // br) * (cols // 128))
    ok(q, L.fp8_block_quantize(x.data_ptr(), rows, cols, cols, br, c.ptr, s.ptr,
                               stream()), "fp8 block")
    c.check("codes")
    s.check("scales")
    same(c, ref.codes, "codes")
    same(s, ref.scales, "scales")
    y = Guarded(rows * cols * 2)
    ok(q, L.fp8_block_dequantize(ref.codes.data_ptr(), ref.scales.data_ptr(), rows, cols,
                                 br, y.ptr, stream()), "fp8 dequant")
    y.check("dequant")
    same(y, q.fp8_block_dequantize(ref.codes, ref.scales, br), "dequant")
    if br == 1 and rows % 128 == 0:
        t = q.fp8_block_requantize_transpose(ref.codes, ref.scales)
        ct, st = Guarded(rows * cols), Guarded(4 * cols * (rows // 128))
        ok(q, L.fp8_block_requantize_transpose(ref.codes.data_ptr(), ref.scales.data_ptr(),
                                               rows, cols, ct.ptr, st.ptr, stream()),
           "requant-t")
        ct.check("codes_t")
        st.check("scales_t")
        same(ct, t.codes, "codes_t")
        same(st, t.scales, "scales_t")


def test_guard_fp8_block_requant_tail(mxq):
    """Requantize-transpose with rows a multiple of 128 and odd column
    tiles."""
    q = mxq
    L = q.lib()
    rows, cols = 384, 640
    x = dev_bf16(W.mxfp8_random(rows, cols, seed=9))
    ref = q.fp8_block_quantize(x, 1)
    t = q.fp8_block_requantize_transpose(ref.codes, ref.scales)
    ct, st = Guarded(rows * cols), Guarded(4 * cols * (rows // 128))
    ok(q, L.fp8_block_requantize_transpose(ref.codes.data_ptr(), ref.scales.data_ptr(),
                                           rows, cols, ct.ptr, st.ptr, stream()),
       "requant-t")
    ct.check("codes_t")
    st.check("scales_t")
    same(ct, t.codes, "codes_t")
    same(st, t.scales, "scales_t")


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 256), (384, 640, 512)])
def test_guard_gemm_mxfp8(mxq, M, N, K):
    q = mxq
    L = q.lib()
    A, B = W.gemm_mxfp8_inputs(M, K, N, seed=M + N)
    qa = q.mxfp8_quantize_rowcol(dev_bf16(A), rowwise=True, colwise=False)
    qb = q.mxfp8_quantize_rowcol(dev_bf16(B), rowwise=False, colwise=True)
    ref = q.gemm_mxfp8(qa.row_codes, qa.row_scales, qb.col_codes_t, qb.col_scales_t)
    C = Guarded(M * N * 4)
    ok(q, L.mxq_gemm_mxfp8(qa.row_codes.data_ptr(), qa.row_scales.data_ptr(),
                           qb.col_codes_t.data_ptr(), qb.col_scales_t.data_ptr(), M, N, K,
                           C.ptr, N, stream()), "gemm")
    C.check("C")
    same(C, ref, "C")
    # the dequantized-backward GEMM on a bf16 A with the same B
    a16 = dev_bf16(W.gemm_tokens(M, K, seed=3))
    ref2 = q.gemm_bf16_mxfp8(a16, qb.col_codes_t, qb.col_scales_t)
    C2 = Guarded(M * N * 4)
    ok(q, L.mxq_gemm_bf16_mxfp8(a16.data_ptr(), K, qb.col_codes_t.data_ptr(),
                                qb.col_scales_t.data_ptr(), M, N, K, C2.ptr, N, stream()),
       "bf16 x mxfp8 gemm")
    C2.check("C")
    same(C2, ref2, "C")


def test_guard_grouped_nvfp4_and_swiglu(mxq):
    q = mxq
    L = q.lib()
    E, H, F = 3, 512, 128
    rows = [128, 256, 128]
    offs = np.concatenate([[0], np.cumsum(rows)])
    toks = dev_bf16(W.gemm_tokens(int(offs[-1]), H, seed=5))
    ta = q.nvfp4_quantize_per_token(toks)
    wts = [dev_bf16(np.concatenate(W.moe_expert(e, hidden=H, ffn=F, seed=5)[:2]))
           for e in range(E)]
    tw = q.nvfp4_quantize_weight_shared([[w] for w in wts])
    off_arr = (ctypes.c_int64 * (E + 1))(*[int(v) for v in offs])
    Mt = int(offs[-1])
    ref = q.gemm_nvfp4_grouped(ta.codes, ta.block_scales, ta.scales, offs, tw.codes,
                               tw.block_scales, tw.scales)
    C = Guarded(Mt * 2 * F * 4)
    ok(q, L.mxq_gemm_nvfp4_grouped(ta.codes.data_ptr(), ta.block_scales.data_ptr(),
                                   ta.scales.data_ptr(), ctypes.cast(off_arr, ctypes.c_void_p),
                                   E, tw.codes.data_ptr(), tw.block_scales.data_ptr(),
                                   tw.scales.data_ptr(), 2 * F, H, C.ptr, 2 * F, stream()),
       "grouped gemm")
    C.check("C")
    same(C, ref, "C")
    ref2 = q.moe_gate_up_swiglu(ta.codes, ta.block_scales, ta.scales, offs, tw.codes,
                                tw.block_scales, tw.scales)
    h = Guarded(Mt * F * 2)
    ok(q, L.mxq_moe_gate_up_swiglu_nvfp4(ta.codes.data_ptr(), ta.block_scales.data_ptr(),
                                         ta.scales.data_ptr(),
                                         ctypes.cast(off_arr, ctypes.c_void_p), E,
                                         tw.codes.data_ptr(), tw.block_scales.data_ptr(),
                                         tw.scales.data_ptr(), F, H, h.ptr, F, stream()),
       "swiglu")
    h.check("h")
    same(h, ref2, "h")


def test_guard_gather_in_gemm(mxq):
    """The routing gather inside the grouped GEMMs' operand load."""
    q = mxq
    L = q.lib()
    T_src, H, F, E = 300, 512, 128, 3
    x = dev_bf16(W.gemm_tokens(T_src, H, seed=6))
    xq = q.nvfp4_quantize_per_token(x, "linear")
    rows = [128, 256, 128]
    offs = np.concatenate([[0], np.cumsum(rows)])
    Mt = int(offs[-1])
    idx = (np.arange(Mt, dtype=np.int32) * 7) % T_src
    idx[::5] = -1
    idx_dev = torch.from_numpy(idx).cuda()
    wts = [dev_bf16(np.concatenate(W.moe_expert(e, hidden=H, ffn=F, seed=6)[:2]))
           for e in range(E)]
    tw = q.nvfp4_quantize_weight_shared([[w] for w in wts])
    off_arr = (ctypes.c_int64 * (E + 1))(*[int(v) for v in offs])
    ref = q.gemm_nvfp4_grouped_gather(xq, idx_dev, offs, tw.codes, tw.block_scales,
                                      tw.scales)
    C = Guarded(Mt * 2 * F * 4)
    ok(q, L.mxq_gemm_nvfp4_grouped_gather(
        xq.codes.data_ptr(), xq.block_scales.data_ptr(), xq.scales.data_ptr(), T_src,
        idx_dev.data_ptr(), ctypes.cast(off_arr, ctypes.c_void_p), E,
        tw.codes.data_ptr(), tw.block_scales.data_ptr(), tw.scales.data_ptr(), 2 * F,
        H, C.ptr, 2 * F, stream()), "grouped gather")
    C.check("C")
    same(C, ref, "C")
    ref2 = q.moe_gate_up_swiglu_gather(xq, idx_dev, offs, tw.codes, tw.block_scales,
                                       tw.scales)
    h = Guarded(Mt * F * 2)
    ok(q, L.mxq_moe_gate_up_swiglu_nvfp4_gather(
        xq.codes.data_ptr(), xq.block_scales.data_ptr(), xq.scales.data_ptr(), T_src,
        idx_dev.data_ptr(), ctypes.cast(off_arr, ctypes.c_void_p), E,
        tw.codes.data_ptr(), tw.block_scales.data_ptr(), tw.scales.data_ptr(), F, H,
        h.ptr, F, stream()), "swiglu gather")
    h.check("h")
    same(h, ref2, "h")
