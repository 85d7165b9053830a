"""GPU parity: libmxq kernels (called through the C ABI binding) against the
CPU oracle, byte for byte.

Codes, scales (every byte of the scale buffer, padding included), FP32
scales and dequantized bf16 must be identical to the oracle's.  Small
cases span several 128x128 tiles and a ragged tail; full-size cases use
the workload shapes with the launch configuration the benchmark times and
compare sampled rows/blocks (the oracle computes them one by one) plus
properties that hold at any size.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import assert_bytes_equal, dev_bf16, host_bits, host_u8

pytestmark = pytest.mark.gpu

LAYOUTS = ["swizzled", "linear"]


@pytest.fixture(scope="module")
def mxq():
    if not torch.cuda.is_available():
        pytest.fail("the GPU tests need a CUDA device")
    from nvfp4_quantizers_gb300 import build
    build.build()
    import nvfp4_quantizers_gb300 as q
    q.lib()
    return q


def exp_scales(logical: np.ndarray, lay: str) -> np.ndarray:
    return O.scale_swizzle(logical) if lay == "swizzled" else logical.reshape(-1)


def got_logical_scales(buf: torch.Tensor, R: int, C: int, lay: str):
    b = host_u8(buf).reshape(-1)
    if lay == "swizzled":
        return O.scale_unswizzle(b, R, C)
    return b.reshape(R, C)


# --------------------------------------------------------------------------
# MXFP8
# --------------------------------------------------------------------------
def check_mxfp8(q, x_bits, lay, rowwise=True, colwise=True, dequant=True,
                x_dev=None):
    x = dev_bf16(x_bits) if x_dev is None else x_dev
    r = q.mxfp8_quantize_rowcol(x, rowwise, colwise, lay)
    torch.cuda.synchronize()
    if rowwise:
        rc, rs = O.mxfp8_quantize_rowwise(x_bits)
        assert_bytes_equal(host_u8(r.row_codes), rc, f"row codes [{lay}]")
        assert_bytes_equal(host_u8(r.row_scales), exp_scales(rs, lay),
                           f"row scales [{lay}]")
        if dequant:
            y = q.dequantize_mxfp8(r.row_codes, r.row_scales, lay)
            assert_bytes_equal(host_bits(y), O.mxfp8_dequantize(rc, rs),
                               f"row dequant [{lay}]")
    else:
        assert r.row_codes is None
    if colwise:
        cc, cs = O.mxfp8_quantize_colwise(x_bits)
        assert_bytes_equal(host_u8(r.col_codes_t), cc, f"col codes [{lay}]")
        assert_bytes_equal(host_u8(r.col_scales_t), exp_scales(cs, lay),
                           f"col scales [{lay}]")
        if dequant:
            y = q.dequantize_mxfp8(r.col_codes_t, r.col_scales_t, lay)
            assert_bytes_equal(host_bits(y), O.mxfp8_dequantize(cc, cs),
                               f"col dequant [{lay}]")
    return r


@pytest.mark.parametrize("lay", LAYOUTS)
def test_mxfp8_dequant_every_code_and_scale(mxq, lay):
    """Dequantization of arbitrary bytes: all 256 codes (the E4M3 NaN pair
    included) under every E8M0 byte 0..255 (0xFF = NaN), 2^-127 subnormal
    and 2^127-overflow corners included.  Non-NaN outputs bit for bit, NaN
    where the oracle has NaN."""
    rows, cols = 256, 8192
    codes = np.tile(np.arange(256, dtype=np.uint8), (rows, cols // 256))
    codes = np.random.default_rng(31).permuted(codes, axis=1)
    scales = np.tile(np.arange(256, dtype=np.uint8)[:, None], (1, cols // 32))
    sdev = exp_scales(scales, lay)
    y = mxq.dequantize_mxfp8(torch.from_numpy(codes).cuda(),
                             torch.from_numpy(np.ascontiguousarray(sdev)).cuda(),
                             lay)
    torch.cuda.synchronize()
    got = host_bits(y)
    want = O.mxfp8_dequantize(codes, scales)
    nan_g = (got & 0x7FFF) > 0x7F80
    nan_w = (want & 0x7FFF) > 0x7F80
    assert np.array_equal(nan_g, nan_w)
    assert nan_w[255].all() and nan_w[:255][(codes[:255] & 0x7F) != 0x7F].sum() == 0
    assert_bytes_equal(np.where(nan_g, 0, got), np.where(nan_w, 0, want),
                       f"dequant of every code and scale [{lay}]")


@pytest.mark.parametrize("lay", LAYOUTS)
def test_mxfp8_small_case_rowwise(mxq, lay):
    """[256 x 512] N(0,1) with boundary / power-of-two / ulp-edge / zero /
    bf16-max rows; rowwise quantize + dequantize."""
    check_mxfp8(mxq, W.mxfp8_small(), lay, colwise=False)


@pytest.mark.parametrize("lay", LAYOUTS)
@pytest.mark.parametrize("cls", ["random", "boundary", "zeros", "maxes"])
def test_mxfp8_classes_ragged(mxq, cls, lay):
    """Four input classes on [416 x 352]: 3 full 128-row tiles + a 32-row
    tail, 2 full 128-column tiles + a 96-column tail."""
    x = W.MXFP8_CLASSES[cls](416, 352)
    check_mxfp8(mxq, x, lay)


def test_mxfp8_format_max(mxq):
    check_mxfp8(mxq, W.fmt_maxes(160, 224, 448.0), "swizzled")


def test_mxfp8_every_bf16_value(mxq):
    """Every finite bf16 value up to 448 in magnitude, 31 per block under a
    block max of 448 (scale 2^0): exhaustive over the E4M3 conversion the
    kernel performs (other scales only shift exponents by powers of two)."""
    bits = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    v = W.bits_to_f32(bits)
    keep = np.isfinite(v) & (np.abs(v) <= 448.0)
    vals = bits[keep]
    nblk = -(-vals.size // 31)
    pad = np.zeros(nblk * 31, np.uint16)
    pad[:vals.size] = vals
    blocks = np.zeros((nblk, 32), np.uint16)
    blocks[:, 0] = W.to_bf16_bits(np.float32(448.0))
    blocks[:, 1:] = pad.reshape(nblk, 31)
    cols = 512
    nrows = -(-nblk * 32 // cols)
    nrows = -(-nrows // 32) * 32
    flat = np.zeros(nrows * cols, np.uint16)
    flat[:nblk * 32] = blocks.reshape(-1)
    check_mxfp8(mxq, flat.reshape(nrows, cols), "swizzled")


@pytest.mark.parametrize("M", [1, 31, 100, 129])
def test_mxfp8_rowwise_only_any_rows(mxq, M):
    x = W.mxfp8_random(M, 160, seed=M)
    check_mxfp8(mxq, x, "swizzled", colwise=False)
    check_mxfp8(mxq, x, "linear", colwise=False)


def test_mxfp8_colwise_only(mxq):
    check_mxfp8(mxq, W.mxfp8_random(96, 64, seed=3), "swizzled", rowwise=False)


def test_mxfp8_strided_input(mxq):
    """A [256 x 192] view of a wider [256 x 320] buffer (ldx = 320)."""
    wide = W.mxfp8_random(256, 320, seed=5)
    dev = dev_bf16(wide)[:, 64:256]
    check_mxfp8(mxq, np.ascontiguousarray(wide[:, 64:256]), "swizzled",
                x_dev=dev)


def test_mxfp8_input_16_byte_aligned(mxq):
    """The input 16 bytes past a 32-byte boundary (the tensor maps need 16),
    with a ragged 96-row tail tile and a 32-column tail."""
    x = W.mxfp8_random(224, 416, seed=9)
    check_mxfp8(mxq, x, "swizzled", x_dev=_dev_bf16_shift16(x))
    check_mxfp8(mxq, x, "linear", x_dev=_dev_bf16_shift16(x))


def _bands(M, n, seed):
    rng = np.random.default_rng(seed)
    b = rng.choice(M // 32, n, replace=False)
    return sorted(set(b.tolist()) | {0, M // 32 - 1})


@pytest.mark.parametrize("cls", ["random", "boundary", "zeros", "maxes"])
def test_mxfp8_full_size_sampled(mxq, cls):
    """The 8192 x 4096 activation at full size (the benchmark's launch
    configuration), for each of the four input classes: sampled 32-row bands
    compared with the oracle for both copies and both dequantizations."""
    M, K = 8192, 4096
    x_bits = W.MXFP8_CLASSES[cls](M, K)
    x = dev_bf16(x_bits)
    r = mxq.mxfp8_quantize_rowcol(x, scale_layout="swizzled")
    yr = mxq.dequantize_mxfp8(r.row_codes, r.row_scales)
    yc = mxq.dequantize_mxfp8(r.col_codes_t, r.col_scales_t)
    torch.cuda.synchronize()
    rs_all = got_logical_scales(r.row_scales, M, K // 32, "swizzled")
    cs_all = got_logical_scales(r.col_scales_t, K, M // 32, "swizzled")
    rc_all, cc_all = host_u8(r.row_codes), host_u8(r.col_codes_t)
    yr_all, yc_all = host_bits(yr), host_bits(yc)
    for b in _bands(M, 6, 1):
        sl = slice(32 * b, 32 * b + 32)
        band = x_bits[sl]
        rc, rs = O.mxfp8_quantize_rowwise(band)
        cc, cs = O.mxfp8_quantize_colwise(band)
        assert_bytes_equal(rc_all[sl], rc, f"row codes band {b}")
        assert_bytes_equal(rs_all[sl], rs, f"row scales band {b}")
        assert_bytes_equal(cc_all[:, sl], cc, f"col codes band {b}")
        assert_bytes_equal(cs_all[:, b:b + 1], cs, f"col scales band {b}")
        assert_bytes_equal(yr_all[sl], O.mxfp8_dequantize(rc, rs), "row dq")
        assert_bytes_equal(yc_all[:, sl], O.mxfp8_dequantize(cc, cs), "col dq")


def test_mxfp8_colwise_is_rowwise_of_transpose_full_size(mxq):
    """Property at any size: the columnwise copy of X equals the rowwise
    copy of X^T, byte for byte, over the whole 8192 x 4096 tensor."""
    x = dev_bf16(W.mxfp8_random(8192, 4096, seed=7))
    a = mxq.mxfp8_quantize_rowcol(x, rowwise=False, colwise=True)
    b = mxq.mxfp8_quantize_rowcol(x.t().contiguous(), rowwise=True,
                                  colwise=False)
    torch.cuda.synchronize()
    assert torch.equal(a.col_codes_t, b.row_codes)
    assert torch.equal(a.col_scales_t, b.row_scales)


@pytest.mark.parametrize("shape,std", [((2048, 2048), 1.0),
                                       ((8192, 2048), 0.02)])
def test_mxfp8_linear_shapes_sampled(mxq, shape, std):
    M, K = shape
    x_bits = (W.linear_input(M, K) if std == 1.0 else W.linear_weight(M, K))
    x = dev_bf16(x_bits)
    r = mxq.mxfp8_quantize_rowcol(x, scale_layout="swizzled")
    torch.cuda.synchronize()
    rs_all = got_logical_scales(r.row_scales, M, K // 32, "swizzled")
    cs_all = got_logical_scales(r.col_scales_t, K, M // 32, "swizzled")
    for b in _bands(M, 4, 2):
        sl = slice(32 * b, 32 * b + 32)
        rc, rs = O.mxfp8_quantize_rowwise(x_bits[sl])
        cc, cs = O.mxfp8_quantize_colwise(x_bits[sl])
        assert_bytes_equal(host_u8(r.row_codes)[sl], rc, "row codes")
        assert_bytes_equal(rs_all[sl], rs, "row scales")
        assert_bytes_equal(host_u8(r.col_codes_t)[:, sl], cc, "col codes")
        assert_bytes_equal(cs_all[:, b:b + 1], cs, "col scales")


def test_mxfp8_repeatable(mxq):
    """Same bytes in, same bytes out, call after call."""
    x = dev_bf16(W.mxfp8_random(1024, 1024, seed=9))
    a = mxq.mxfp8_quantize_rowcol(x)
    b = mxq.mxfp8_quantize_rowcol(x)
    torch.cuda.synchronize()
    for u, v in zip(a[:4], b[:4]):
        assert torch.equal(u, v)
    assert mxq.get_last_error() == mxq.MXQ_OK


# --------------------------------------------------------------------------
# NVFP4 per token
# --------------------------------------------------------------------------
def check_nvfp4_tokens(q, x_bits, lay, x_dev=None, dequant=True):
    x = dev_bf16(x_bits) if x_dev is None else x_dev
    r = q.nvfp4_quantize_per_token(x, lay)
    torch.cuda.synchronize()
    codes, sc, S = O.nvfp4_quantize_per_token(x_bits)
    assert_bytes_equal(host_u8(r.codes), codes, f"codes [{lay}]")
    assert_bytes_equal(host_u8(r.block_scales), exp_scales(sc, lay),
                       f"block scales [{lay}]")
    assert_bytes_equal(r.scales.cpu().numpy().view(np.uint32),
                       S.view(np.uint32), f"token scales [{lay}]")
    if dequant:
        y = q.dequantize_nvfp4(r.codes, r.block_scales, r.scales, lay)
        assert_bytes_equal(host_bits(y), O.nvfp4_dequantize(codes, sc, S),
                           f"dequant [{lay}]")
    return r


@pytest.mark.parametrize("lay", LAYOUTS)
def test_nvfp4_ragged_batch(mxq, lay):
    x = W.ragged_tokens([5, 130, 1, 77, 300], H=2048)
    check_nvfp4_tokens(mxq, x, lay)


@pytest.mark.parametrize("H", [16, 48, 96, 768, 1040, 4096, 6144, 8192])
def test_nvfp4_hidden_sizes(mxq, H):
    x = W.ragged_tokens([37], H=H, seed=H)
    check_nvfp4_tokens(mxq, x, "swizzled")
    check_nvfp4_tokens(mxq, x, "linear")


@pytest.mark.parametrize("lay", LAYOUTS)
def test_nvfp4_tokens_16_byte_aligned(mxq, lay):
    """Tokens whose rows start 16 bytes past a 32-byte boundary (the
    16-byte load path), hidden 2048 and 768."""
    for H in (2048, 768):
        x = W.ragged_tokens([3, 130, 61], H=H)
        check_nvfp4_tokens(mxq, x, lay, x_dev=_dev_bf16_shift16(x))


@pytest.mark.parametrize("lay", LAYOUTS)
def test_nvfp4_edge_tokens(mxq, lay):
    """All-zero token, subnormal FP32 scale, all +-2688, all +-bf16 max,
    one huge channel (block scales that round to zero), E2M1 midpoints."""
    for H in (64, 256):
        check_nvfp4_tokens(mxq, W.tiny_token_rows(H=H), lay)


def test_nvfp4_block_scale_pairs(mxq):
    """Many (block amax, token amax) pairs: each token's first block holds
    the token max, the other 63 blocks carry smaller maxima spread over 40
    binades below it."""
    rng = np.random.default_rng(21)
    T, H = 4096, 1024
    at = np.ldexp(rng.uniform(1, 2, T), rng.integers(-60, 60, T))
    x = rng.uniform(-1, 1, (T, H)) * 0.999
    ratio = np.ldexp(rng.uniform(0.5, 1, (T, H // 16)),
                     -rng.integers(0, 40, (T, H // 16)))
    x = x * np.repeat(ratio, 16, axis=1) * at[:, None]
    x[:, 0] = at
    check_nvfp4_tokens(mxq, W.to_bf16_bits(x), "swizzled")


def _logical_token_bytes(q_res, T, H, lay):
    codes = host_u8(q_res.codes)
    sc = got_logical_scales(q_res.block_scales, T, H // 16, lay)
    S = q_res.scales.cpu().numpy().view(np.uint32)
    return codes, sc, S


def test_nvfp4_batch_invariance(mxq):
    """NVFP4 recipe: a token's bytes are the same quantized alone, in the
    batch, and in a shuffled batch (compared on logical bytes: the swizzled
    position of a scale legitimately depends on the row index)."""
    H = 2048
    x_bits = W.ragged_tokens([64, 200, 33], H=H)
    T = x_bits.shape[0]
    x = dev_bf16(x_bits)
    base = _logical_token_bytes(mxq.nvfp4_quantize_per_token(x), T, H, "swizzled")
    perm = np.random.default_rng(1).permutation(T)
    shuf = _logical_token_bytes(
        mxq.nvfp4_quantize_per_token(x[torch.from_numpy(perm).cuda()]), T, H,
        "swizzled")
    for a, b in zip(base, shuf):
        assert np.array_equal(a[perm], b)
    for t in (0, 5, 63, 64, 296):
        alone = _logical_token_bytes(mxq.nvfp4_quantize_per_token(x[t:t + 1]),
                                     1, H, "swizzled")
        for a, b in zip(base, alone):
            assert np.array_equal(a[t:t + 1], b)


def test_nvfp4_full_ragged_batch_sampled(mxq):
    """64 sequences with lengths U[128, 4096], H = 2048, t(4) values with
    sparse outliers, at full size; sampled tokens vs the oracle, and the
    same tokens quantized alone."""
    lengths = W.ragged_lengths()
    x_bits = W.ragged_tokens(lengths, H=2048)
    T = x_bits.shape[0]
    x = dev_bf16(x_bits)
    r = mxq.nvfp4_quantize_per_token(x, "swizzled")
    y = mxq.dequantize_nvfp4(r.codes, r.block_scales, r.scales)
    torch.cuda.synchronize()
    codes, sc, S = _logical_token_bytes(r, T, 2048, "swizzled")
    yb = host_bits(y)
    idx = np.random.default_rng(3).choice(T, 256, replace=False)
    idx = np.union1d(idx, [0, T - 1])
    oc, osc, oS = O.nvfp4_quantize_per_token(x_bits[idx])
    assert_bytes_equal(codes[idx], oc, "codes")
    assert_bytes_equal(sc[idx], osc, "scales")
    assert_bytes_equal(S[idx], oS.view(np.uint32), "S")
    assert_bytes_equal(yb[idx], O.nvfp4_dequantize(oc, osc, oS), "dequant")


# --------------------------------------------------------------------------
# NVFP4 weights with a shared FP32 scale
# --------------------------------------------------------------------------
def _dev_bf16_shift16(bits):
    """bits on the device 16 bytes past a 32-byte boundary (inside a
    larger allocation), so that 32-byte loads are not allowed."""
    rows, cols = bits.shape
    buf = torch.empty(rows * cols + 8, dtype=torch.bfloat16, device="cuda")
    view = buf[8:8 + rows * cols].view(rows, cols)
    view.copy_(dev_bf16(bits))
    assert view.data_ptr() % 32 == 16
    return view


def check_weight_groups(q, groups_bits, lay, S_in=None, shift16=False):
    place = _dev_bf16_shift16 if shift16 else dev_bf16
    groups = [[place(p) for p in g] for g in groups_bits]
    S_dev = None if S_in is None else torch.from_numpy(S_in).cuda()
    r = q.nvfp4_quantize_weight_shared(groups, S_dev, lay)
    y = q.dequantize_nvfp4(r.codes, r.block_scales, r.scales, lay)
    torch.cuda.synchronize()
    assert q.get_last_error() == q.MXQ_OK       # no bounded wait gave up
    codes, bs, S, yb = host_u8(r.codes), host_u8(r.block_scales), \
        r.scales.cpu().numpy(), host_bits(y)
    for g, parts in enumerate(groups_bits):
        oc, osc, oS = O.nvfp4_quantize_group(
            parts, None if S_in is None else S_in[g])
        assert_bytes_equal(codes[g], oc, f"group {g} codes [{lay}]")
        assert_bytes_equal(bs[g], exp_scales(osc, lay), f"group {g} scales")
        assert S[g].view(np.uint32) == np.float32(oS).view(np.uint32), g
        assert_bytes_equal(yb[g], O.nvfp4_dequantize(oc, osc, np.array([oS])),
                           f"group {g} dequant")
    return r


@pytest.mark.parametrize("lay", LAYOUTS)
def test_weight_gate_up_pairs_small(mxq, lay):
    experts = [W.moe_expert(e, hidden=256, ffn=64) for e in range(3)]
    r = check_weight_groups(mxq, [[g, u] for g, u, d in experts], lay)
    check_weight_groups(mxq, [[d] for g, u, d in experts], lay)
    # the shared scale: max of the two parts' amax / 2688
    for e, (g, u, d) in enumerate(experts):
        a = max(O.bf16_amax(g), O.bf16_amax(u))
        assert r.scales[e].item() == np.float32(np.float32(a) / np.float32(2688))


def test_weight_scale_passed_in(mxq):
    """Live update: quantizing gate alone with the stored pair scale gives
    the gate half of the fused pair."""
    experts = [W.moe_expert(e, hidden=128, ffn=64, seed=4) for e in range(2)]
    pair = mxq.nvfp4_quantize_weight_shared(
        [[dev_bf16(g), dev_bf16(u)] for g, u, d in experts])
    S = pair.scales.cpu().numpy()
    check_weight_groups(mxq, [[g] for g, u, d in experts], "swizzled", S_in=S)
    gate = mxq.nvfp4_quantize_weight_shared(
        [[dev_bf16(g)] for g, u, d in experts], pair.scales)
    torch.cuda.synchronize()
    assert torch.equal(gate.codes, pair.codes[:, :64])
    assert torch.equal(gate.scales, pair.scales)


@pytest.mark.parametrize("lay", LAYOUTS)
def test_weight_ragged_parts(mxq, lay):
    """Parts of 100 and 60 rows (160 rows per group: a partial 128-row
    scale tile) and K = 48 (3 blocks: a partial 4-column scale tile)."""
    rng = np.random.default_rng(8)
    groups = [[W.to_bf16_bits(rng.standard_normal((100, 48)) * s),
               W.to_bf16_bits(rng.standard_normal((60, 48)) * 2 * s)]
              for s in (1e-3, 1.0, 30.0)]
    check_weight_groups(mxq, groups, lay)


@pytest.mark.parametrize("lay", LAYOUTS)
def test_weight_odd_scale_rows(mxq, lay):
    """Parts of 99 and 60 rows with K = 48: 477 block scales per group, so
    the linear scale matrices of consecutive groups are not 4-byte aligned
    (byte stores), and the swizzled ones have a padding column."""
    rng = np.random.default_rng(13)
    groups = [[W.to_bf16_bits(rng.standard_normal((99, 48)) * s),
               W.to_bf16_bits(rng.standard_normal((60, 48)) * 3 * s)]
              for s in (1e-2, 1.0, 7.0, 0.3)]
    check_weight_groups(mxq, groups, lay)


@pytest.mark.parametrize("lay", LAYOUTS)
def test_weight_wide_rows_and_slices(mxq, lay):
    """K = 1552 (97 blocks per row: 16 KiB units start and end inside rows,
    and a partial 4-column scale tile), parts of 300 and 200 rows (units
    straddle the part boundary), three groups at three scales."""
    rng = np.random.default_rng(11)
    groups = [[W.to_bf16_bits(rng.standard_normal((300, 1552)) * s),
               W.to_bf16_bits(rng.standard_normal((200, 1552)) * 0.5 * s)]
              for s in (2e-3, 1.0, 50.0)]
    check_weight_groups(mxq, groups, lay)


@pytest.mark.parametrize("lay", LAYOUTS)
def test_weight_parts_16_byte_aligned(mxq, lay):
    """Parts whose base lies 16 bytes past a 32-byte boundary: every amax
    task takes the general path (a part lookup per 16-byte chunk) and every
    row the 16-byte loads; gate/up-like pairs (2048 values a row) and
    down-like parts (768 values a row, half-warp rows)."""
    rng = np.random.default_rng(13)
    pairs = [[W.to_bf16_bits(rng.standard_normal((200, 2048)) * s),
              W.to_bf16_bits(rng.standard_normal((300, 2048)) * 0.5 * s)]
             for s in (0.01, 3.0)]
    check_weight_groups(mxq, pairs, lay, shift16=True)
    downs = [[W.to_bf16_bits(rng.standard_normal((256, 768)) * s)]
             for s in (0.2, 40.0, 1e-3)]
    check_weight_groups(mxq, downs, lay, shift16=True)


def test_weight_windows(mxq):
    """Three gate/up pairs of [2048 x 4096] (32 MiB each, larger than a
    window): the task list spans three windows of one group each.  Every
    group scale is checked, and the first and the last group byte for
    byte."""
    rng = np.random.default_rng(12)
    groups_bits = [[W.to_bf16_bits(rng.standard_normal((2048, 4096)) * s),
                    W.to_bf16_bits(rng.standard_normal((2048, 4096)) * 2 * s)]
                   for s in (0.01, 1.0, 0.02)]
    groups = [[dev_bf16(x) for x in g] for g in groups_bits]
    r = mxq.nvfp4_quantize_weight_shared(groups)
    torch.cuda.synchronize()
    assert mxq.get_last_error() == mxq.MXQ_OK
    S = r.scales.cpu().numpy()
    for e, (a, b) in enumerate(groups_bits):
        assert S[e] == O.nvfp4_tensor_scale(max(O.bf16_amax(a), O.bf16_amax(b)))
    for e in (0, 2):
        oc, osc, oS = O.nvfp4_quantize_group(groups_bits[e])
        assert_bytes_equal(host_u8(r.codes[e]), oc, f"group {e} codes")
        assert_bytes_equal(host_u8(r.block_scales[e]), O.scale_swizzle(osc),
                           f"group {e} scales")


def test_weight_full_moe_layer_sampled(mxq):
    """128 Qwen3-30B-A3B-shaped experts at full size: gate/up fused pairs
    [1536 x 2048] under one scale each, down [2048 x 768] under its own.
    Every group scale is checked; three experts are checked byte for byte
    (codes, scales, and the dequantization of both)."""
    E = 128
    experts = [W.moe_expert(e) for e in range(E)]
    gu = mxq.nvfp4_quantize_weight_shared(
        [[dev_bf16(g), dev_bf16(u)] for g, u, d in experts])
    dn = mxq.nvfp4_quantize_weight_shared([[dev_bf16(d)] for g, u, d in experts])
    ygu = mxq.dequantize_nvfp4(gu.codes, gu.block_scales, gu.scales)
    ydn = mxq.dequantize_nvfp4(dn.codes, dn.block_scales, dn.scales)
    torch.cuda.synchronize()
    assert mxq.get_last_error() == mxq.MXQ_OK
    for e, (g, u, d) in enumerate(experts):
        a_gu = max(O.bf16_amax(g), O.bf16_amax(u))
        assert gu.scales[e].item() == O.nvfp4_tensor_scale(a_gu)
        assert dn.scales[e].item() == O.nvfp4_tensor_scale(O.bf16_amax(d))
    for e in (0, 77, E - 1):
        g, u, d = experts[e]
        oc, osc, oS = O.nvfp4_quantize_group([g, u])
        assert_bytes_equal(host_u8(gu.codes[e]), oc, f"expert {e} gate/up codes")
        assert_bytes_equal(host_u8(gu.block_scales[e]), O.scale_swizzle(osc),
                           f"expert {e} gate/up scales")
        assert_bytes_equal(host_bits(ygu[e]),
                           O.nvfp4_dequantize(oc, osc, np.array([oS])),
                           f"expert {e} gate/up dequant")
        oc, osc, oS = O.nvfp4_quantize_group([d])
        assert_bytes_equal(host_u8(dn.codes[e]), oc, f"expert {e} down codes")
        assert_bytes_equal(host_u8(dn.block_scales[e]), O.scale_swizzle(osc),
                           f"expert {e} down scales")
        assert_bytes_equal(host_bits(ydn[e]),
                           O.nvfp4_dequantize(oc, osc, np.array([oS])),
                           f"expert {e} down dequant")


# --------------------------------------------------------------------------
# Weight groups of many shapes: the MoE layer's gate/up pairs and down
# projections, small and odd part sizes, rows whose block count is not a
# multiple of 4, many groups, given scales right after computed ones.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("lay", LAYOUTS)
@pytest.mark.parametrize("rows,K,G", [
    ((768, 768), 2048, 3),      # gate/up pairs
    ((2048,), 768, 5),          # down projections, 48 blocks per row
    ((77, 30), 640, 3),         # 40 blocks per row: half-warp rows, odd row count
    ((5,), 528, 4),             # 33 blocks per row, 5 rows: one half idle
    ((200, 56), 512, 7),        # ~256 KiB groups, parts of 200 and 56 rows
    ((33,), 4096, 9),           # 33 rows of 4096: a partial scale tile
    ((1000,), 1552, 2),         # 97 blocks per row: byte scale stores
])
def test_weight_group_shapes(mxq, lay, rows, K, G):
    rng = np.random.default_rng(sum(rows) + K + G)
    groups = [[W.to_bf16_bits(rng.standard_normal((r, K)) * s * (1 + i))
               for i, r in enumerate(rows)]
              for s in np.geomspace(1e-3, 40.0, G)]
    check_weight_groups(mxq, groups, lay)


def test_weight_many_groups(mxq):
    """300 small groups (more than one launch's 256) and a zero group."""
    rng = np.random.default_rng(21)
    groups = [[W.to_bf16_bits(rng.standard_normal((32, 64)) * (g % 7 + 1))]
              for g in range(300)]
    groups[5] = [np.zeros((32, 64), np.uint16)]
    check_weight_groups(mxq, groups, "swizzled")


def test_weight_scale_in_after_amax(mxq):
    """A call with group_scales_in right after an amax call on the same
    workspace-sized groups: the given scales are used as they are."""
    experts = [W.moe_expert(e, hidden=2048, ffn=768, seed=6) for e in range(3)]
    gu = [[g, u] for g, u, d in experts]
    r = check_weight_groups(mxq, gu, "swizzled")
    S_in = (r.scales.cpu().numpy() * np.float32(1.5)).astype(np.float32)
    check_weight_groups(mxq, gu, "swizzled", S_in=S_in)
