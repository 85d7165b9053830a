"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle against something fixed outside it: values
worked by hand from the pages' format statements (tests/golden/*), library
casts that implement the same textbook formats (torch, optionally
ml_dtypes), closed forms, brute-force search written independently in
numpy, and invariants the pages state.  Sources are (page title, section).
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as W
from conftest import golden_lines

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# --------------------------------------------------------------------------
# Codec tables vs library decoders (standard format definitions).
# --------------------------------------------------------------------------
def test_e4m3_table_matches_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([orc.decode_e4m3(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(mine[~nan], ref[~nan])
    assert orc.decode_e4m3(0x7E) == 448.0 and orc.decode_e4m3(0x01) == 2.0 ** -9


def test_e8m0_table_matches_torch(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(
        torch.float8_e8m0fnu).to(torch.float64).numpy()
    mine = np.array([orc.decode_e8m0(c) for c in range(256)])
    assert np.isnan(mine[255]) and np.isnan(ref[255])
    assert np.array_equal(mine[:255], ref[:255])
    assert mine[127] == 1.0 and mine[0] == 2.0 ** -127


def test_bf16_decode_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(
        torch.float64).numpy()
    mine = np.array([orc.decode_bf16(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_e2m1_table_from_format_definition(orc):
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(8):
        assert orc.decode_e2m1(c) == mags[c]
        assert orc.decode_e2m1(c | 8) == -mags[c]
    assert math.copysign(1.0, orc.decode_e2m1(8)) == -1.0


def test_e2m1_table_matches_ml_dtypes(orc):
    mld = pytest.importorskip("ml_dtypes")
    # ml_dtypes stores one E2M1 value per byte in its low nibble
    ref = np.arange(16, dtype=np.uint8).view(mld.float4_e2m1fn).astype(
        np.float64)
    mine = np.array([orc.decode_e2m1(c) for c in range(16)])
    assert np.array_equal(mine, ref)


# --------------------------------------------------------------------------
# Round-to-nearest-even.
# --------------------------------------------------------------------------
def _torch_e4m3_rne(vals):
    t = torch.from_numpy(np.clip(vals, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_rne_matches_torch_on_all_bf16(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = W.bits_to_f32(bits).astype(np.float64)
    ok = np.isfinite(vals)
    vals = vals[ok]
    ref = _torch_e4m3_rne(vals)
    mine = np.array([orc.rne_e4m3(v) for v in vals], np.uint8)
    assert np.array_equal(mine, ref)


def test_e4m3_rne_matches_torch_near_midpoints(orc):
    rng = np.random.default_rng(123)
    mids = np.concatenate([W.E4M3_MIDPOINTS, -W.E4M3_MIDPOINTS])
    vals = []
    for m in mids:
        m32 = np.float32(m)
        vals += [m32, np.nextafter(m32, np.float32(0)),
                 np.nextafter(m32, np.float32(1e9) * np.sign(m32))]
    vals += list(rng.uniform(-500, 500, 20000).astype(np.float32))
    vals += list((rng.uniform(-1, 1, 20000) * 2.0 ** -8).astype(np.float32))
    vals = np.array(vals, np.float32).astype(np.float64)
    ref = _torch_e4m3_rne(vals)
    mine = np.array([orc.rne_e4m3(v) for v in vals], np.uint8)
    assert np.array_equal(mine, ref)


def test_e4m3_rne_saturates_and_keeps_sign(orc):
    assert orc.rne_e4m3(464.0) == 0x7E           # tie 448/480 -> even 448
    assert orc.rne_e4m3(1e30) == 0x7E
    assert orc.rne_e4m3(-1e30) == 0xFE
    assert orc.rne_e4m3(-1e-9) == 0x80
    assert orc.rne_e4m3(2.0 ** -10) == 0x00       # tie 0 / 2^-9 -> 0
    assert orc.rne_e4m3(1.5 * 2.0 ** -10) == 0x01


def test_e2m1_rne_golden(orc):
    for v, code in golden_lines("e2m1_rne.txt"):
        assert orc.rne_e2m1(float(v)) == int(code, 16), v


def test_e2m1_rne_matches_ml_dtypes(orc):
    mld = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(7)
    vals = np.concatenate([rng.uniform(-6, 6, 20000),
                           np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])])
    vals = vals.astype(np.float32).astype(np.float64)
    ref = vals.astype(mld.float4_e2m1fn).view(np.uint8) & 0xF
    mine = np.array([orc.rne_e2m1(v) for v in vals], np.uint8)
    assert np.array_equal(mine, ref)


def test_e2m1_rne_brute_force(orc):
    """Nearest magnitude by exhaustive distance over the 8 magnitudes (ties
    to the even code), written independently of the oracle."""
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rng = np.random.default_rng(8)
    vals = np.concatenate([rng.uniform(-7, 7, 5000),
                           (mags[:-1] + mags[1:]) / 2,
                           -(mags[:-1] + mags[1:]) / 2])
    for v in vals.astype(np.float32).astype(np.float64):
        a = min(abs(v), 6.0)
        d = np.abs(mags - a)
        best = np.nonzero(d == d.min())[0]
        c = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        c |= 8 if math.copysign(1.0, v) < 0 else 0
        assert orc.rne_e2m1(v) == c, v


def test_bf16_rne_matches_torch(orc):
    rng = np.random.default_rng(9)
    u = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)
    mine = np.array([orc.rne_bf16(float(v)) for v in f], np.uint16)
    assert np.array_equal(mine, ref)
    # ties and the overflow edge
    edge = np.array([3.3895313892515355e38, 3.3961775292304957e38,
                     3.4028234663852886e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8],
                    np.float32)
    ref = torch.from_numpy(edge).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)
    assert [orc.rne_bf16(float(v)) for v in edge] == list(ref)


# --------------------------------------------------------------------------
# E8M0 scale exponent (formats section: rounded up, block max not clipped).
# --------------------------------------------------------------------------
def _ceil_log2_ratio(a: float) -> int:
    """ceil(log2(a / 448)) in exact rational arithmetic."""
    q = Fraction(a) / 448
    k = math.frexp(float(q))[1]           # 2^(k-1) <= q < 2^k roughly
    while Fraction(2) ** (k - 1) >= q:
        k -= 1
    while Fraction(2) ** k < q:
        k += 1
    return k


def test_e8m0_exponent_exhaustive_over_bf16(orc):
    bits = np.arange(0, 0x7F80, dtype=np.uint16)       # all finite a >= 0
    vals = W.bits_to_f32(bits).astype(np.float64)
    for a in vals:
        k = orc.mxfp8_scale_exponent(a)
        if a == 0.0:
            assert k == -127
            continue
        expect = max(-127, _ceil_log2_ratio(a))
        assert k == expect, a
        # never clipped, and one step smaller would clip (unless clamped)
        assert a * 2.0 ** -k <= 448.0
        if k > -127:
            assert a * 2.0 ** -(k - 1) > 448.0


def test_e8m0_exponent_hand_values(orc):
    assert orc.mxfp8_scale_exponent(1.0) == -8
    assert orc.mxfp8_scale_exponent(448.0) == 0
    assert orc.mxfp8_scale_exponent(450.0) == 1
    assert orc.mxfp8_scale_exponent(3.3895313892515355e38) == 120
    assert orc.mxfp8_scale_exponent(2.0 ** -133) == -127


# --------------------------------------------------------------------------
# MXFP8 block encode / decode.
# --------------------------------------------------------------------------
def _golden_mxfp8_blocks():
    blocks, cur = [], None
    for tok in golden_lines("mxfp8_blocks.txt"):
        if tok[0] == "block":
            cur = {"name": tok[1], "scale": int(tok[2], 16), "rows": []}
            blocks.append(cur)
        else:
            cur["rows"].append((float(tok[0]), int(tok[1], 16),
                                int(tok[2], 16)))
    return blocks


def test_mxfp8_golden_blocks(orc):
    for blk in _golden_mxfp8_blocks():
        vals = np.zeros(32, np.float64)
        for i, (v, _, _) in enumerate(blk["rows"]):
            vals[i] = v
        x = W.to_bf16_bits(vals).reshape(1, 32)
        codes, scales = orc.mxfp8_quantize_rowwise(x)
        assert scales[0, 0] == blk["scale"], blk["name"]
        y = orc.mxfp8_dequantize(codes, scales)
        for i, (v, code, deq) in enumerate(blk["rows"]):
            assert codes[0, i] == code, (blk["name"], v)
            assert y[0, i] == deq, (blk["name"], v)
        n = len(blk["rows"])
        assert np.all(codes[0, n:] == 0) and np.all(y[0, n:] == 0)


def test_mxfp8_brute_force_small_blocks(orc):
    """Independent brute force: try every E8M0 scale from the smallest up,
    keep the first under which no element exceeds the E4M3 max, and pick
    each code as the argmin of |E4M3(c) * 2^k - x| over all 254 finite codes
    (ties to the even code)."""
    tab = torch.arange(256, dtype=torch.uint8).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = np.nonzero(np.isfinite(tab))[0]
    rng = np.random.default_rng(11)
    for trial in range(40):
        scale = 2.0 ** rng.integers(-30, 30)
        v = rng.standard_normal(32) * scale
        if trial % 5 == 0:
            v[rng.integers(32)] = 448.0 * 2.0 ** rng.integers(-20, 20)
        x = W.to_bf16_bits(v).reshape(1, 32)
        xv = W.bits_to_f32(x).astype(np.float64)[0]
        codes, scales = orc.mxfp8_quantize_rowwise(x)
        for e in range(255):
            if np.all(np.abs(xv) <= 448.0 * 2.0 ** (e - 127)):
                break
        assert scales[0, 0] == e
        for i in range(32):
            d = np.abs(tab[finite] * 2.0 ** (e - 127) - xv[i])
            best = finite[d == d.min()]
            # among equal magnitudes keep the sign of x; ties -> even code
            best = [b for b in best if (b >= 128) == (math.copysign(1, xv[i]) < 0)]
            c = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
            assert codes[0, i] == c, (trial, i, xv[i])


def test_mxfp8_block_max_never_clipped(orc):
    """Formats section: with the rounded-up scale the block maximum's code
    decodes to at least 224 (half of 448) unless the scale is clamped at its
    minimum, and no element is saturated."""
    x = W.mxfp8_random(256, 512, outlier_frac=1e-2)
    codes, scales = orc.mxfp8_quantize_rowwise(x)
    xv = W.bits_to_f32(x).astype(np.float64).reshape(256, 16, 32)
    tab = orc.e4m3_table()
    dec = tab[codes].reshape(256, 16, 32)
    k = scales.astype(np.int64) - 127
    amax = np.abs(xv).max(-1)
    assert np.all(amax * np.ldexp(1.0, -k) <= 448.0)
    idx = np.abs(xv).argmax(-1)
    top = np.abs(np.take_along_axis(dec, idx[..., None], -1)[..., 0])
    assert np.all((top >= 224.0) | (k == -127))


def test_mxfp8_roundtrip_error_bound(orc):
    """|dequant - x| <= half an E4M3 step at the scaled magnitude, times
    2^k (exact RNE with no saturation)."""
    x = W.mxfp8_random(128, 256)
    codes, scales = orc.mxfp8_quantize_rowwise(x)
    y = W.bits_to_f32(orc.mxfp8_dequantize(codes, scales)).astype(np.float64)
    xv = W.bits_to_f32(x).astype(np.float64)
    k = np.repeat(scales.astype(np.int64) - 127, 32, axis=1)
    s = np.abs(xv) * np.ldexp(1.0, -k)
    e = np.floor(np.log2(np.maximum(s, 2.0 ** -6)))
    half_step = np.ldexp(1.0, (e - 3).astype(np.int64)) / 2
    assert np.all(np.abs(y - xv) <= half_step * np.ldexp(1.0, k) * (1 + 1e-12))


def test_mxfp8_colwise_equals_rowwise_of_transpose(orc):
    """MXFP8 recipe section: the columnwise copy is quantized from the
    full-precision data in 32x1 blocks; stored transposed it must equal the
    rowwise quantization of X^T."""
    x = W.mxfp8_random(96, 160)
    ct, st = orc.mxfp8_quantize_colwise(x)
    cr, sr = orc.mxfp8_quantize_rowwise(np.ascontiguousarray(x.T))
    assert np.array_equal(ct, cr) and np.array_equal(st, sr)
    # and it differs from re-deriving columns out of the rowwise copy
    c_row, s_row = orc.mxfp8_quantize_rowwise(x)
    assert not np.array_equal(ct, np.ascontiguousarray(c_row.T))


def test_mxfp8_zero_and_max_classes(orc):
    z = W.mxfp8_zeros(64, 64)
    c, s = orc.mxfp8_quantize_rowwise(z)
    assert not c.any() and not s.any()
    assert not orc.mxfp8_dequantize(c, s).any()
    m = W.mxfp8_maxes(64, 64)
    c, s = orc.mxfp8_quantize_rowwise(m)
    assert np.all(s == 247) and np.all((c & 0x7F) == 0x78)
    y = orc.mxfp8_dequantize(c, s)
    assert np.all((y & 0x7FFF) == 0x7F80)          # 2^128 overflows to inf
    f = W.fmt_maxes(64, 64, 448.0)
    c, s = orc.mxfp8_quantize_rowwise(f)
    assert np.all(s == 127) and np.all((c & 0x7F) == 0x7E)


def test_mxfp8_dequant_exact_for_bf16_inputs(orc):
    """For codes made from bf16 data, E4M3(c) * 2^k always lies on the bf16
    grid, so the bf16 dequant equals the exact product (here checked
    against an exact float64 product of the torch-decoded tables)."""
    x = W.mxfp8_boundary(64, 128)
    c, s = orc.mxfp8_quantize_rowwise(x)
    y = W.bits_to_f32(orc.mxfp8_dequantize(c, s)).astype(np.float64)
    tab = torch.arange(256, dtype=torch.uint8).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    exact = tab[c] * np.ldexp(1.0, np.repeat(s.astype(np.int64) - 127, 32, 1))
    assert np.array_equal(y, exact)


# --------------------------------------------------------------------------
# NVFP4.
# --------------------------------------------------------------------------
def test_nvfp4_golden_token(orc):
    lines = list(golden_lines("nvfp4_token.txt"))
    S = float(lines[0][1])
    scales = [int(t, 16) for t in lines[1][1:]]
    vals = np.zeros(32)
    exp = {}
    for idx, v, code, deq in lines[2:]:
        vals[int(idx)] = float(v)
        exp[int(idx)] = (int(code, 16), int(deq, 16))
    x = W.to_bf16_bits(vals).reshape(1, 32)
    codes, sc, St = orc.nvfp4_quantize_per_token(x)
    assert St[0] == np.float32(S)
    assert list(sc[0]) == scales
    q = np.empty(32, np.uint8)
    q[0::2] = codes[0] & 0xF
    q[1::2] = codes[0] >> 4
    y = orc.nvfp4_dequantize(codes, sc, St)
    for i in range(32):
        c, d = exp.get(i, (0, 0))
        assert q[i] == c, i
        assert y[0, i] == d, i


def test_code_times_scale_worked_example(orc):
    """Code 3 under two different scales gives two different values."""
    rows = list(golden_lines("code_times_scale.txt"))
    vals = []
    for code, sb, value, bits in rows:
        codes = np.array([[int(code, 16) | (int(code, 16) << 4)] * 8], np.uint8)
        scales = np.array([[int(sb, 16)]], np.uint8)
        y = orc.nvfp4_dequantize(codes, scales, np.array([1.0], np.float32))
        assert y[0, 0] == int(bits, 16)
        assert W.bits_to_f32(y[0, :1])[0] == float(value)
        vals.append(float(value))
        assert orc.rne_e4m3({"1D": 0.1, "25": 0.2}[sb]) == int(sb, 16)
    assert vals[0] != vals[1] and vals[1] == 2 * vals[0]


def _nvfp4_unpack(codes):
    q = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    q[:, 0::2] = codes & 0xF
    q[:, 1::2] = codes >> 4
    return q


def test_nvfp4_scale_invariants(orc):
    """With S = amax/(6*448), the block holding a token's max gets block
    scale 448 (0x7E) and the max element gets code +-6; all-zero tokens get
    zero bytes and S = 0."""
    x = W.ragged_tokens([40, 25], H=256)
    x[3] = 0
    codes, sc, S = orc.nvfp4_quantize_per_token(x)
    xv = W.bits_to_f32(x)
    q = _nvfp4_unpack(codes)
    for t in range(x.shape[0]):
        a = np.abs(xv[t]).max()
        assert S[t] == np.float32(a) / np.float32(2688.0)
        if a == 0:
            assert S[t] == 0 and not sc[t].any() and not (q[t] & 7).any()
            continue
        assert sc[t].max() == 0x7E
        i = np.abs(xv[t]).argmax()
        assert (q[t, i] & 7) == 7
        assert (q[t, i] >> 3) == (xv[t, i] < 0)


def test_nvfp4_roundtrip_error_bound(orc):
    """dequant(quant(x)) lies within half an E2M1 step (of the scaled
    magnitude) of x, up to the binary32 rounding of the scales."""
    x = W.ragged_tokens([64], H=512)
    codes, sc, S = orc.nvfp4_quantize_per_token(x)
    y = W.bits_to_f32(orc.nvfp4_dequantize(codes, sc, S)).astype(np.float64)
    xv = W.bits_to_f32(x).astype(np.float64)
    d = np.repeat(orc.e4m3_table()[sc], 16, axis=1) * S[:, None]
    v = np.abs(xv) / np.where(d == 0, 1, d)
    step = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0))
    bound = np.where(d == 0, np.abs(xv), (step / 2) * d * (1 + 1e-5)
                     + np.abs(y) * 2.0 ** -8)
    assert np.all(np.abs(y - xv) <= bound)


def test_nvfp4_batch_invariance(orc):
    """NVFP4 recipe section: a per-token FP32 scale makes a token's bytes
    independent of the rest of the batch (alone, in batch, shuffled)."""
    x = W.ragged_tokens([30, 50, 17], H=128)
    c, s, S = orc.nvfp4_quantize_per_token(x)
    perm = np.random.default_rng(1).permutation(x.shape[0])
    cp, sp, Sp = orc.nvfp4_quantize_per_token(x[perm])
    assert np.array_equal(cp, c[perm]) and np.array_equal(sp, s[perm])
    assert np.array_equal(Sp, S[perm])
    for t in (0, 31, 96):
        c1, s1, S1 = orc.nvfp4_quantize_per_token(x[t:t + 1])
        assert np.array_equal(c1[0], c[t]) and np.array_equal(s1[0], s[t])
        assert S1[0] == S[t]
    # a per-tensor scale would not be batch invariant
    big = np.concatenate([x, W.to_bf16_bits(np.full((1, 128), 1e4))])
    cg, sg, _ = orc.nvfp4_quantize_group([big], None)
    assert not np.array_equal(cg[:x.shape[0]], c)


def test_nvfp4_gate_up_share_one_scale(orc):
    """NVFP4 recipe section: gate and up share one FP32 scale, so
    S = max(amax_gate, amax_up)/2688, and quantizing gate alone with that
    scale passed in reproduces the gate half of the fused result."""
    g, u, d = W.moe_expert(0, hidden=256, ffn=64)
    codes, sc, S = orc.nvfp4_quantize_group([g, u])
    ag, au = orc.bf16_amax(g), orc.bf16_amax(u)
    assert S == np.float32(np.float32(max(ag, au)) / np.float32(2688.0))
    cg, sg, Sg = orc.nvfp4_quantize_group([g], S_in=S)
    assert np.array_equal(cg, codes[:64]) and np.array_equal(sg, sc[:64])
    cu, su, _ = orc.nvfp4_quantize_group([u], S_in=S)
    assert np.array_equal(cu, codes[64:]) and np.array_equal(su, sc[64:])
    # separately scaled halves generally differ from the fused pair
    cg2, _, Sg2 = orc.nvfp4_quantize_group([g])
    cu2, _, Su2 = orc.nvfp4_quantize_group([u])
    assert Sg2 != Su2
    assert not (np.array_equal(cg2, codes[:64]) and np.array_equal(cu2, codes[64:]))


def test_nvfp4_edge_tokens(orc):
    x = W.tiny_token_rows(H=64)
    codes, sc, S = orc.nvfp4_quantize_per_token(x)
    q = _nvfp4_unpack(codes)
    assert S[0] == 0 and not sc[0].any() and not (q[0] & 7).any()
    # subnormal S: no flush to zero, the token still quantizes
    assert 0 < S[1] < np.finfo(np.float32).tiny
    assert sc[1].max() == 0x7E and (q[1] & 7).max() == 7
    # all +-2688 -> S = 1, block scales 448, codes +-6
    assert S[2] == 1.0 and np.all(sc[2] == 0x7E) and np.all((q[2] & 7) == 7)
    # all +-bf16 max: finite S, codes +-6
    assert np.isfinite(S[3]) and np.all((q[3] & 7) == 7)
    # one huge channel: blocks far below it get block scale 0 -> codes +-0
    assert (sc[4] == 0).sum() >= 1
    y = orc.nvfp4_dequantize(codes, sc, S)
    assert not (y[0] & 0x7FFF).any()


def test_nvfp4_quantize_then_gather(orc):
    """Token-local scaling: quantize-then-gather == gather-then-quantize."""
    x = W.ragged_tokens([40], H=64)
    idx = np.array([5, 1, 39, 5, 0])
    c, s, S = orc.nvfp4_quantize_per_token(x)
    c2, s2, S2 = orc.nvfp4_quantize_per_token(x[idx])
    assert np.array_equal(c[idx], c2) and np.array_equal(s[idx], s2)
    assert np.array_equal(S[idx], S2)


# --------------------------------------------------------------------------
# Swizzled scale layout.
# --------------------------------------------------------------------------
def test_swizzle_golden_positions(orc):
    for R, C, r, c, off in golden_lines("scale_swizzle.txt"):
        R, C, r, c, off = map(int, (R, C, r, c, off))
        logical = np.zeros((R, C), np.uint8)
        logical[r, c] = 0xAB
        swz = orc.scale_swizzle(logical)
        assert np.nonzero(swz)[0].tolist() == [off]


def test_swizzle_is_a_permutation_with_zero_padding(orc):
    rng = np.random.default_rng(3)
    for R, C in ((128, 4), (200, 6), (33, 17), (1, 1)):
        logical = rng.integers(1, 256, (R, C)).astype(np.uint8)
        swz = orc.scale_swizzle(logical)
        assert swz.size == -(-R // 128) * 128 * (-(-C // 4)) * 4
        assert (swz != 0).sum() == R * C
        assert np.array_equal(orc.scale_unswizzle(swz, R, C), logical)


# --------------------------------------------------------------------------
# GEMM oracle: closed forms.
# --------------------------------------------------------------------------
def test_gemm_oracle_closed_form(orc):
    """Small-integer operands are exact in E4M3; the MXFP8 GEMM oracle must
    reproduce the exact integer matmul."""
    rng = np.random.default_rng(4)
    A = rng.integers(-8, 9, (8, 64)).astype(np.float32)
    B = rng.integers(-8, 9, (64, 16)).astype(np.float32)
    A[:, 0] = 448                       # scale exponent 0 on every row block
    Bt = np.ascontiguousarray(B.T)
    Bt[:, 0] = 448
    Bt[:, 32] = 448
    A[:, 32] = 448
    ac, asc = orc.mxfp8_quantize_rowwise(W.to_bf16_bits(A))
    bc, bsc = orc.mxfp8_quantize_rowwise(W.to_bf16_bits(Bt))
    assert np.all(asc == 127) and np.all(bsc == 127)
    C = orc.gemm_mxfp8(ac, asc, bc, bsc)
    assert np.array_equal(C, A.astype(np.float64) @ Bt.T.astype(np.float64))


def test_gemm_nvfp4_grouped_closed_form(orc):
    """E2M1-representable operands with block scale 1 and S = 1/448 ...
    the grouped oracle must equal per-expert exact matmuls times S_a*S_w."""
    rng = np.random.default_rng(5)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4])
    a = rng.choice(mags, (6, 32)) * np.where(rng.random((6, 32)) < .5, -1, 1)
    w = rng.choice(mags, (2, 4, 32))
    a[:, 0] = 6.0
    a[:, 16] = 6.0
    w[:, :, 0] = 6.0
    w[:, :, 16] = 6.0
    S1 = np.array([1.0 / 448], np.float32)
    ac, asc = orc.nvfp4_encode_rows(W.to_bf16_bits(a), S1)
    assert np.all(asc == 0x7E)
    wc = np.stack([orc.nvfp4_encode_rows(W.to_bf16_bits(w[e]), S1)[0]
                   for e in range(2)])
    ws = np.stack([orc.nvfp4_encode_rows(W.to_bf16_bits(w[e]), S1)[1]
                   for e in range(2)])
    aS = np.full(6, 0.5, np.float32)
    wS = np.array([2.0, 0.25], np.float32)
    off = np.array([0, 4, 6])
    C = orc.gemm_nvfp4_grouped(ac, asc, aS, off, wc, ws, wS)
    # decoded operands are a*448 (block scale 448 x code) exactly
    ref = np.zeros((6, 4))
    ref[:4] = (a[:4] * 448) @ (w[0] * 448).T * 0.5 * 2.0
    ref[4:] = (a[4:] * 448) @ (w[1] * 448).T * 0.5 * 0.25
    assert np.array_equal(C, ref)


# --------------------------------------------------------------------------
# MoE gate/up + SwiGLU oracle: closed forms and structure.
# --------------------------------------------------------------------------
def test_silu_closed_forms(orc):
    """silu(0) = 0; sigmoid(ln 3) = 3/4; silu(-z) = silu(z) - z; silu(z)/z
    -> 1 and silu(-z) -> 0 for large z."""
    assert orc.silu(0.0) == 0.0
    assert abs(orc.silu(np.log(3.0)) - 0.75 * np.log(3.0)) < 1e-15
    z = np.random.default_rng(7).normal(0, 4, 1000)
    assert np.max(np.abs(orc.silu(-z) - (orc.silu(z) - z))) < 1e-12
    assert abs(orc.silu(40.0) / 40.0 - 1.0) < 1e-15
    assert abs(orc.silu(-40.0)) < 1e-15
    assert orc.silu(-1e4) == 0.0 and orc.silu(1e4) == 1e4


def test_gather_rows_pads_with_zero_rows(orc):
    x = np.arange(12, dtype=np.uint16).reshape(4, 3) + 1
    idx = np.array([2, -1, 0, 4, 3])
    g = orc.gather_rows(x, idx)
    assert np.array_equal(g, np.array([[7, 8, 9], [0, 0, 0], [1, 2, 3],
                                       [0, 0, 0], [10, 11, 12]]))


def test_moe_swiglu_structure(orc):
    """Exact small-integer operands: gate columns equal to 0 give h = 0;
    gate columns with a large positive value give h = g * u (silu(g) = g to
    1e-15); large negative give |h| < 1e-12 |u|; up columns equal to 0 give
    h = 0.  Swapping the gate and up halves changes h, and the two FP32
    scales multiply both halves before the activation."""
    rng = np.random.default_rng(8)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4])
    F, K = 4, 32
    a = rng.choice(mags, (6, K)) * np.where(rng.random((6, K)) < .5, -1, 1)
    a[:, 0] = 6.0
    a[:, 16] = 6.0
    w = rng.choice(mags, (2, 2 * F, K))
    w[:, :, 0] = 6.0
    w[:, :, 16] = 6.0
    w[:, 0, 1:16] = 0.0            # gate column 0: g = 6*6*448*448*S... > 0
    w[:, 0, 17:] = 0.0
    w[:, F + 1, :] = 0.0           # up column 1: u = 0
    S1 = np.array([1.0 / 448], np.float32)
    enc = [orc.nvfp4_encode_rows(W.to_bf16_bits(w[e]), S1) for e in range(2)]
    wc = np.stack([c for c, _ in enc])
    wsc = np.stack([s for _, s in enc])
    ac, asc = orc.nvfp4_encode_rows(W.to_bf16_bits(a), S1)
    aS = np.full(6, 0.5, np.float32)
    wS = np.array([2.0, 0.25], np.float32)
    off = np.array([0, 4, 6])
    h = orc.moe_gate_up_swiglu(ac, asc, aS, off, wc, wsc, wS)
    # exact gate/up products (decoded operands are value * 448)
    full = np.zeros((6, 2 * F))
    full[:4] = (a[:4] * 448) @ (w[0] * 448).T * 0.5 * 2.0
    full[4:] = (a[4:] * 448) @ (w[1] * 448).T * 0.5 * 0.25
    g, u = full[:, :F], full[:, F:]
    assert np.all(g[:, 0] > 1e5)
    assert np.allclose(h[:, 0], g[:, 0] * u[:, 0], rtol=1e-15, atol=0)
    assert np.all(h[:, 1] == 0)
    big_neg = g < -50
    assert np.all(np.abs(h[big_neg]) <= 1e-12 * np.abs(u[big_neg]))
    zero_g = g == 0
    assert np.all(h[zero_g] == 0)
    # In the O(1) range (tiny FP32 scales) silu is far from linear: swapping
    # the gate and up halves must change h.
    aS_small = np.full(6, 2.0 ** -11, np.float32)
    wS_small = np.array([2.0 ** -11, 2.0 ** -10], np.float32)
    swapped = np.concatenate([wc[:, F:], wc[:, :F]], axis=1)
    swapped_s = np.concatenate([wsc[:, F:], wsc[:, :F]], axis=1)
    h1 = orc.moe_gate_up_swiglu(ac, asc, aS_small, off, wc, wsc, wS_small)
    h2 = orc.moe_gate_up_swiglu(ac, asc, aS_small, off, swapped, swapped_s,
                                wS_small)
    assert 0.01 < np.median(np.abs(h1[:, 2:])) < 100
    assert not np.allclose(h1, h2, rtol=1e-3)


# --------------------------------------------------------------------------
# FP8 with FP32 block scales (DeepSeek-V3-style recipe, introduction of
# "Miles: end-to-end MXFP8 and per-token NVFP4 RL": 128x128 weight blocks,
# 1x128 activation tiles, online scales; MXFP8 recipe section: the backward
# conversion dequantizes and requantizes the 1x128 tiles).
# --------------------------------------------------------------------------
def _fp8blk_power_of_two_rows(rng, R, C):
    """Rows whose 1x128 tiles have amax exactly 448 * 2^j (one element per
    tile at +-448 * 2^j, the rest uniform below it)."""
    x = np.empty((R, C), np.float32)
    for r in range(R):
        for t in range(C // 128):
            j = int(rng.integers(-12, 12))
            v = rng.uniform(-448, 448, 128) * 2.0 ** j
            v[rng.integers(128)] = (448.0 if rng.random() < 0.5 else -448.0) * 2.0 ** j
            x[r, t * 128:(t + 1) * 128] = v
    return W.to_bf16_bits(x)


def test_fp8blk_power_of_two_scale_matches_torch_cast(orc):
    """amax = 448 * 2^j gives S = 2^j exactly, so x * fl(1/S) is exact and
    the codes are torch's E4M3 cast of x * 2^-j (all within +-448)."""
    rng = np.random.default_rng(31)
    x = _fp8blk_power_of_two_rows(rng, 8, 512)
    codes, S = orc.fp8_block_quantize(x, 1)
    xf = W.bits_to_f32(x).astype(np.float64)
    amax = np.abs(xf).reshape(8, 4, 128).max(axis=2)
    j = np.log2(amax / 448.0)
    assert np.array_equal(j, np.round(j))
    assert np.array_equal(S.astype(np.float64), 2.0 ** j)
    scaled = xf / np.repeat(2.0 ** j, 128, axis=1)
    assert np.abs(scaled).max() <= 448.0
    ref = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


def test_fp8blk_block_max_gets_the_format_max(orc):
    """In every non-zero block the element of largest magnitude encodes to
    +-448 (0x7E / 0xFE): a * fl(1/fl(a/448)) is within a few ulp of 448,
    far inside 448's rounding interval [432, 448].  A scale stored the other
    way round (encode instead of decode) or a wrong block extent breaks it."""
    rng = np.random.default_rng(32)
    x = W.to_bf16_bits(rng.standard_t(3, size=(256, 384)).astype(np.float32)
                       * 10.0 ** rng.uniform(-30, 30, size=(256, 1)).astype(np.float32))
    xf = np.abs(W.bits_to_f32(x))
    for br in (1, 128):
        codes, S = orc.fp8_block_quantize(x, br)
        blk = xf.reshape(256 // br, br, 3, 128).transpose(0, 2, 1, 3).reshape(
            256 // br, 3, -1)
        cb = codes.reshape(256 // br, br, 3, 128).transpose(0, 2, 1, 3).reshape(
            256 // br, 3, -1)
        arg = blk.argmax(axis=2)
        top = np.take_along_axis(cb, arg[..., None], axis=2)[..., 0]
        assert np.all((top & 0x7F) == 0x7E)
        assert np.all(S > 0)
        assert np.array_equal(S, (blk.max(axis=2) / np.float32(448)).astype(np.float32))


def test_fp8blk_zero_block_and_signs(orc):
    x = np.zeros((2, 256), np.uint16)
    x[1, :128] = 0x8000                       # -0 everywhere in one tile
    x[1, 200] = W.to_bf16_bits(np.array([3.0], np.float32))[0]
    codes, S = orc.fp8_block_quantize(x, 1)
    assert S[0, 0] == 0 and S[0, 1] == 0 and S[1, 0] == 0
    assert np.all(codes[0] == 0) and np.all(codes[1, :128] == 0x80)
    assert S[1, 1] == np.float32(3.0) / np.float32(448.0)
    assert codes[1, 200] == 0x7E
    y = orc.fp8_block_dequantize(codes, S, 1)
    assert np.all(y[0] == 0) and np.all(y[1, :128] == 0x8000)


def test_fp8blk_round_trip_within_half_a_step(orc):
    """dequant(quant(x)) is within half an E4M3 step of x (relative 2^-4 in
    the normal range, 2^-10 * S absolute in the subnormal range) plus the
    bf16 rounding of the result (relative 2^-8)."""
    rng = np.random.default_rng(33)
    x = W.to_bf16_bits(rng.standard_normal((128, 512)).astype(np.float32))
    xf = W.bits_to_f32(x).astype(np.float64)
    for br in (1, 128):
        codes, S = orc.fp8_block_quantize(x, br)
        y = W.bits_to_f32(orc.fp8_block_dequantize(codes, S, br)).astype(np.float64)
        s = np.repeat(np.repeat(S.astype(np.float64), br, axis=0), 128, axis=1)
        bound = np.abs(xf) * (2.0 ** -4 + 2.0 ** -8) * (1 + 1e-6) + s * 2.0 ** -10 * (1 + 2.0 ** -8)
        assert np.all(np.abs(y - xf) <= bound)


def test_fp8blk_block_geometry_brute_force(orc):
    """Raising one element changes the scale of exactly the block that holds
    it: 1x128 tiles run along rows, 128x128 blocks tile the matrix."""
    rng = np.random.default_rng(34)
    base = W.to_bf16_bits(rng.uniform(-1, 1, (256, 256)).astype(np.float32))
    for br in (1, 128):
        _, S0 = orc.fp8_block_quantize(base, br)
        for (r, c) in ((0, 0), (5, 130), (200, 127), (255, 255)):
            x = base.copy()
            x[r, c] = W.to_bf16_bits(np.array([1000.0], np.float32))[0]
            _, S1 = orc.fp8_block_quantize(x, br)
            changed = np.argwhere(S1 != S0)
            assert changed.tolist() == [[r // br, c // 128]]


def test_fp8blk_backward_conversion(orc):
    """Requantizing 1x128 tiles in the backward orientation is exact when the
    forward dequantization is (x built from E4M3 values times 2^j, so
    dequant(quant(x)) == x): then it equals quantizing x^T directly.  On
    generic data it is not: the dequantize-then-requantize path adds error
    on top of the direct 128x1 quantization (MXFP8 recipe section)."""
    rng = np.random.default_rng(35)
    e4 = np.array([orc.decode_e4m3(c) for c in range(0x7F)])
    M, K = 256, 256
    v = rng.choice(e4, size=(M, K)) * rng.choice([-1.0, 1.0], size=(M, K))
    j = rng.integers(-8, 8, size=(M, K // 128))
    v[:, ::128] = 448.0                       # every tile's amax is 448 * 2^j
    x = W.to_bf16_bits((v * np.repeat(2.0 ** j, 128, axis=1)).astype(np.float32))
    codes, S = orc.fp8_block_quantize(x, 1)
    assert np.array_equal(orc.fp8_block_dequantize(codes, S, 1), x)
    ct, st = orc.fp8_block_requantize_transpose(codes, S)
    dt, sd = orc.fp8_block_quantize(np.ascontiguousarray(x.T), 1)
    assert np.array_equal(ct, dt) and np.array_equal(st, sd)
    # generic data: the conversion differs from the direct quantization
    g = W.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    codes, S = orc.fp8_block_quantize(g, 1)
    ct, st = orc.fp8_block_requantize_transpose(codes, S)
    dt, sd = orc.fp8_block_quantize(np.ascontiguousarray(g.T), 1)
    assert (ct != dt).any()
    gf = W.bits_to_f32(np.ascontiguousarray(g.T)).astype(np.float64)
    err_conv = np.abs(W.bits_to_f32(orc.fp8_block_dequantize(ct, st, 1)) - gf).mean()
    err_direct = np.abs(W.bits_to_f32(orc.fp8_block_dequantize(dt, sd, 1)) - gf).mean()
    assert err_conv > err_direct


def test_fp8blk_subnormal_scale(orc):
    """A block whose amax is ~1e-37 has a subnormal S = fl(amax / 448) (no
    flush to zero) whose reciprocal overflows, so enc = FLT_MAX: S must be
    numpy's binary32 quotient and the codes torch's E4M3 cast of
    fl(x * FLT_MAX)."""
    rng = np.random.default_rng(36)
    v = (rng.uniform(-1, 1, (3, 256)) * 1e-37).astype(np.float32)
    x = W.to_bf16_bits(v)
    codes, S = orc.fp8_block_quantize(x, 1)
    amax = np.abs(W.bits_to_f32(x)).reshape(3, 2, 128).max(axis=2)
    ref = (amax.astype(np.float32) / np.float32(448.0)).astype(np.float32)
    assert np.all(ref < np.finfo(np.float32).tiny) and np.all(ref > 0)
    assert np.array_equal(S.view(np.uint32), ref.view(np.uint32))
    xf = W.bits_to_f32(x).astype(np.float32)
    prod = (xf * np.float32(np.finfo(np.float32).max)).astype(np.float64)
    exp = torch.from_numpy(np.clip(prod, -448, 448).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, exp)


# --------------------------------------------------------------------------
# NVFP4 with the pretraining recipe's stabilizers (NVFP4 recipe section:
# stochastic rounding for unbiased quantized gradients, Random Hadamard
# Transforms to disperse block outliers).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("key,counter", [((0, 0), (0, 0, 0, 0)),
                                         ((0x0123456789abcdef, 0xfedcba9876543210), (5, 0, 0, 0)),
                                         ((2**64 - 1, 2**64 - 1), (2**64 - 2, 7, 9, 2**64 - 1))])
def test_philox4x64_matches_numpy(orc, key, counter):
    """The oracle's Philox4x64-10 against numpy's own implementation of the
    same published generator (numpy steps the counter once before each
    block of four outputs)."""
    bg = np.random.Philox(counter=np.array(counter, np.uint64),
                          key=np.array(key, np.uint64))
    raw = bg.random_raw(8)
    c = list(counter)
    for blk in range(2):
        # counter + 1 with carry across the four 64-bit words
        i = 0
        while True:
            c[i] = (c[i] + 1) % 2 ** 64
            if c[i] != 0 or i == 3:
                break
            i += 1
        assert np.array_equal(orc.philox4x64(c, key), raw[4 * blk:4 * blk + 4])


def _sylvester16():
    H = np.array([[1.0]])
    for _ in range(4):
        H = np.kron(np.array([[1.0, 1.0], [1.0, -1.0]]), H)
    return H


def test_rht16_is_the_sylvester_transform(orc):
    """On small integers every butterfly sum is exact, so the binary32
    transform equals (1/4) H16 (s * x) in float64, H16 built by Kronecker
    products; (1/4) H16 is orthonormal, so applying it twice with all signs
    + returns x."""
    rng = np.random.default_rng(51)
    H = _sylvester16()
    assert np.allclose(H @ H.T / 16, np.eye(16))
    for seed in (0, 1, 12345):
        s = np.array([-1.0 if (orc.rht_signs(seed) >> i) & 1 else 1.0
                      for i in range(16)])
        for _ in range(20):
            x = rng.integers(-8, 9, 16).astype(np.float32)
            y = orc.rht16(x, orc.rht_signs(seed))
            assert np.array_equal(y.astype(np.float64), H @ (s * x) / 4)
    x = rng.integers(-8, 9, 16).astype(np.float32)
    assert np.array_equal(orc.rht16(orc.rht16(x, 0), 0), x)


def test_rht_sr_reduce_to_per_token(orc):
    """Without RHT and SR the path is the per-token quantizer; with RHT on
    inputs whose transforms are bf16 values, it is the per-token quantizer
    of the transformed rows."""
    x = W.ragged_tokens([5, 3], H=256)
    assert all(np.array_equal(a, b) for a, b in zip(
        orc.nvfp4_quantize_rht_sr(x, 9, 0), orc.nvfp4_quantize_per_token(x)))
    rng = np.random.default_rng(52)
    xi = rng.integers(-8, 9, (6, 64)).astype(np.float32)
    xb = W.to_bf16_bits(xi)
    signs = orc.rht_signs(3)
    y = np.stack([np.concatenate([orc.rht16(row[b * 16:(b + 1) * 16], signs)
                                  for b in range(4)]) for row in xi])
    yb = W.to_bf16_bits(y)
    assert np.array_equal(W.bits_to_f32(yb), y)          # exact in bf16
    got = orc.nvfp4_quantize_rht_sr(xb, 3, orc.RHT)
    exp = orc.nvfp4_quantize_per_token(yb)
    assert all(np.array_equal(a, b) for a, b in zip(got, exp))


def test_sr_is_unbiased_and_keeps_grid_values(orc):
    """A block whose maximum is 2688 has S = 1, block scale 448 and
    enc = 1/448, so x = 1008 scales to exactly 2.25: stochastic rounding
    gives 2 or 3 with mean 2.25 (4096 independent positions), while
    x = 1344 (exactly 3.0) always gives 3."""
    R = 4096
    row = np.zeros(16, np.float32)
    row[0] = 2688.0
    row[1] = 1008.0
    row[2] = 1344.0
    x = W.to_bf16_bits(np.tile(row, (R, 1)))
    codes, sc, S = orc.nvfp4_quantize_rht_sr(x, 77, orc.SR)
    assert np.all(S == 1.0) and np.all(sc[:, 0] == 0x7E)
    e2 = np.array([orc.decode_e2m1(c) for c in range(16)])
    v1 = e2[codes[:, 0] >> 4]
    v2 = e2[codes[:, 1] & 0xF]
    assert set(np.unique(v1)) == {2.0, 3.0}
    assert abs(v1.mean() - 2.25) < 0.03
    assert np.all(v2 == 3.0)
    again = orc.nvfp4_quantize_rht_sr(x, 77, orc.SR)[0]
    other = orc.nvfp4_quantize_rht_sr(x, 78, orc.SR)[0]
    assert np.array_equal(codes, again) and not np.array_equal(codes, other)


def test_gemm_bf16_mxfp8_closed_form(orc):
    """One non-zero code in B^T: column n of C is column k of A times that
    code's value E4M3(c) * 2^(s - 127); everything else is zero."""
    rng = np.random.default_rng(61)
    A = W.to_bf16_bits(rng.standard_normal((4, 64)).astype(np.float32))
    codes = np.zeros((3, 64), np.uint8)
    scales = np.full((3, 2), 127, np.uint8)
    codes[1, 40] = 0x46                      # E4M3 1.75 * 2 = 3.5
    scales[1, 1] = 127 + 5                   # block 1 of row 1: 2^5
    C = orc.gemm_bf16_mxfp8(A, codes, scales)
    af = W.bits_to_f32(A).astype(np.float64)
    assert orc.decode_e4m3(0x46) == 3.5
    exp = np.zeros((4, 3))
    exp[:, 1] = af[:, 40] * 3.5 * 32
    assert np.array_equal(C, exp)
