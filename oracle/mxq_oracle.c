/*
 * mxq_oracle.c -- plain, slow, scalar CPU oracle for the MXFP8 / NVFP4
 * quantizer contract.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library and its Python binding) never calls it, links it or
 * shares any code, header, table or constant generator with it.
 *
 * Sources (page title, section):
 *  - "Miles: end-to-end MXFP8 and per-token NVFP4 RL", formats section:
 *      MXFP8 = E4M3 elements, 32 consecutive values share one E8M0
 *      (power-of-two) scale, 1-D blocks; the decoded scale is rounded up so
 *      the block maximum is not clipped.
 *      NVFP4 = E2M1 elements with one E4M3 scale per 16 values, rounded to
 *      the nearest representable value, plus one FP32 scale over a larger
 *      tensor scope (two-level hierarchy).
 *  - same page, MXFP8 recipe section: rowwise 1x32 and columnwise 32x1
 *      blocks are quantized independently from the full-precision data.
 *  - same page, NVFP4 recipe section: one FP32 activation scale per token,
 *      computed online; gate/up weights share one FP32 scale.
 *  - same page, backward-mode section: dequantized backward consumes BF16
 *      dequantizations of the exact forward low-precision operands.
 *  - "Using Quantization in RL", section "Two Ways to Configure Training
 *      and Inference": a stored value is interpreted as code x scale.
 *
 * Design rules of this file:
 *  - Every format is decoded from its bit pattern (sign / exponent /
 *    mantissa fields), and every rounding is a brute-force nearest search
 *    over the decoded table with ties resolved to the even code.  No bit
 *    tricks are used to round.
 *  - MXFP8 arithmetic is exact: block amax, the power-of-two scale and the
 *    scaled element x * 2^-k are computed in binary64, where all of them are
 *    exact for bf16 inputs.
 *  - NVFP4 arithmetic is binary32, because the pages fix the second-level
 *    scale as an FP32 number; every step is one IEEE binary32 operation
 *    with round-to-nearest-even (compiled with -ffp-contract=off, no fast
 *    math, FLT_EVAL_METHOD == 0).
 *  - Readings of points the pages leave open (listed in the design notes):
 *      scale exponent k = smallest integer with 448 * 2^k >= amax, clamped
 *      to [-127, 127] (an all-zero block gets k = -127, scale byte 0x00);
 *      NVFP4 FP32 scale is a decode scale S = amax / (6 * 448);
 *      block scale sb = RNE_E4M3(amax_b / (6 * S)); element encode factor
 *      enc = 1 / (E4M3(sb) * S) (0 when that product is 0, FLT_MAX-clamped);
 *      packed E2M1: lower-index element in the low nibble.
 *
 * Logical layouts produced here (row-major, no padding, no swizzle):
 *  - MXFP8 rowwise: codes [R x C], scales [R x C/32] (block j of row r at
 *    r*(C/32)+j).
 *  - MXFP8 columnwise of X [M x K]: codes stored transposed [K x M] (byte
 *    (k, m) at k*M+m) and scales [K x M/32].
 *  - NVFP4: codes [R x C/2] (two per byte), block scales [R x C/16].
 *  - Swizzled scale layout: oracle_scale_swizzle() maps the logical matrix
 *    to the 128x4-tile layout; it is a pure permutation with zero padding.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs binary32 arithmetic evaluated in binary32"
#endif

/* ------------------------------------------------------------------------ */
/* Format decoders, from the bit fields.                                     */
/* ------------------------------------------------------------------------ */

/* bf16: 1 sign, 8 exponent (bias 127), 7 mantissa bits. */
static double bf16_decode(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int m = b & 0x7F;
    double v;
    if (e == 0xFF) return m ? NAN : (sign ? -INFINITY : INFINITY);
    if (e == 0) v = ldexp((double)m / 128.0, -126);           /* subnormal */
    else v = ldexp(1.0 + (double)m / 128.0, e - 127);
    return sign ? -v : v;
}

/* E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa; S.1111.111 = NaN;
 * no infinities; max finite 448. */
static double e4m3_decode(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa; no NaN/inf; max 6. */
static double e2m1_decode(uint8_t c) {
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 0x3;
    int m = c & 0x1;
    double v;
    if (e == 0) v = (double)m * 0.5;
    else v = ldexp(1.0 + (double)m / 2.0, e - 1);
    return sign ? -v : v;
}

/* E8M0 (unsigned): 2^(e-127) for e in [0, 254]; 0xFF = NaN. */
static double e8m0_decode(uint8_t c) {
    if (c == 0xFF) return NAN;
    return ldexp(1.0, (int)c - 127);
}

/* ------------------------------------------------------------------------ */
/* Tables built by enumerating every code once.                              */
/* ------------------------------------------------------------------------ */
static double T_E4M3[256];
static double T_E2M1[16];
static int g_tables_ready = 0;

static void build_tables(void) {
    if (g_tables_ready) return;
    for (int c = 0; c < 256; ++c) T_E4M3[c] = e4m3_decode((uint8_t)c);
    for (int c = 0; c < 16; ++c) T_E2M1[c] = e2m1_decode((uint8_t)c);
    g_tables_ready = 1;
}

/* ------------------------------------------------------------------------ */
/* Round-to-nearest-even by brute force over the non-negative codes.          */
/* Saturate first (|v| > max -> max), then pick the nearest magnitude; on a   */
/* tie the code with a 0 least-significant bit wins.  The sign bit of the    */
/* input is kept, so a negative value that rounds to zero gives -0.          */
/* ------------------------------------------------------------------------ */
static uint8_t rne_e4m3(double v) {
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    if (a > 448.0) a = 448.0;
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {          /* 0x7F is NaN */
        double d = fabs(T_E4M3[c] - a);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)(best | (neg << 7));
}

static uint8_t rne_e2m1(double v) {
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    if (a > 6.0) a = 6.0;
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 7; ++c) {
        double d = fabs(T_E2M1[c] - a);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)(best | (neg << 3));
}

/* Round a finite binary32 value to bf16, nearest, ties to even mantissa:
 * the two candidates are the bf16 values that bracket it (truncation toward
 * zero and the next bf16 away from zero); the nearer one wins, exactly
 * compared in binary64.  Overflow past the largest bf16 goes to infinity
 * as IEEE rounding does (the candidate above 0x7F7F is 0x7F80 = inf, and
 * the halfway point to it is 2^128 - 2^119). */
static uint16_t rne_bf16_from_f32(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u) {       /* inf / nan pass through */
        uint16_t hi = (uint16_t)(u >> 16);
        if (u & 0x007FFFFFu) hi |= 0x40;          /* keep NaN a NaN */
        return hi;
    }
    uint16_t lo = (uint16_t)(u >> 16);            /* toward zero */
    uint16_t up = (uint16_t)(lo + 1);             /* away from zero */
    double x = fabs((double)f);
    double vlo = fabs(bf16_decode(lo));
    double vup;
    if ((up & 0x7FFF) == 0x7F80) vup = ldexp(1.0, 128);  /* next step is inf */
    else vup = fabs(bf16_decode(up));
    double dlo = x - vlo, dup = vup - x;
    if (dlo < dup) return lo;
    if (dup < dlo) return up;
    return (lo & 1) ? up : lo;
}

/* ------------------------------------------------------------------------ */
/* Exported codec probes (used by the pin tests).                            */
/* ------------------------------------------------------------------------ */
double oracle_decode_bf16(uint16_t b) { return bf16_decode(b); }
double oracle_decode_e4m3(uint8_t c) { return e4m3_decode(c); }
double oracle_decode_e2m1(uint8_t c) { return e2m1_decode(c); }
double oracle_decode_e8m0(uint8_t c) { return e8m0_decode(c); }
uint8_t oracle_rne_e4m3(double v) { build_tables(); return rne_e4m3(v); }
uint8_t oracle_rne_e2m1(double v) { build_tables(); return rne_e2m1(v); }
uint16_t oracle_rne_bf16(float f) { return rne_bf16_from_f32(f); }

/* ------------------------------------------------------------------------ */
/* MXFP8 (formats section + MXFP8 recipe section).                           */
/* ------------------------------------------------------------------------ */

/* E8M0 scale exponent for a block maximum a >= 0: the smallest k in
 * [-127, 127] with 448 * 2^k >= a, i.e. the power-of-two scale "rounded
 * up" so that a / 2^k never exceeds the E4M3 maximum.  Brute force over
 * every representable scale. */
static int mxfp8_scale_exponent(double a) {
    for (int k = -127; k <= 127; ++k)
        if (448.0 * ldexp(1.0, k) >= a) return k;
    return 127;
}

int oracle_mxfp8_scale_exponent(double a) { return mxfp8_scale_exponent(a); }

/* Encode one block of n values, read with a stride: returns the E8M0 byte
 * and writes n E4M3 codes to out (contiguous). */
static uint8_t mxfp8_encode_block(const uint16_t* x, int64_t stride, int n,
                                  uint8_t* out) {
    double a = 0.0;
    for (int i = 0; i < n; ++i) {
        double v = fabs(bf16_decode(x[(int64_t)i * stride]));
        if (v > a) a = v;
    }
    int k = mxfp8_scale_exponent(a);
    double inv = ldexp(1.0, -k);                /* exact power of two */
    for (int i = 0; i < n; ++i)
        out[i] = rne_e4m3(bf16_decode(x[(int64_t)i * stride]) * inv);
    return (uint8_t)(k + 127);
}

/* Rowwise 1x32 blocks of X [R x C] (row stride ldx elements).
 * codes [R x C], scales [R x C/32].  Returns 0, or -1 on a bad shape. */
int oracle_mxfp8_quantize_rowwise(const uint16_t* x, int64_t R, int64_t C,
                                  int64_t ldx, uint8_t* codes,
                                  uint8_t* scales) {
    if (C % 32 != 0 || R < 0 || ldx < C) return -1;
    build_tables();
    int64_t nb = C / 32;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t j = 0; j < nb; ++j)
            scales[r * nb + j] = mxfp8_encode_block(
                x + r * ldx + j * 32, 1, 32, codes + r * C + j * 32);
    return 0;
}

/* Columnwise 32x1 blocks of X [M x K], quantized from X itself (never from
 * the rowwise copy).  Output is stored transposed: codes_t [K x M] with
 * byte (k, m) at k*M+m, scales_t [K x M/32].  Returns 0 or -1. */
int oracle_mxfp8_quantize_colwise(const uint16_t* x, int64_t M, int64_t K,
                                  int64_t ldx, uint8_t* codes_t,
                                  uint8_t* scales_t) {
    if (M % 32 != 0 || M < 0 || ldx < K) return -1;
    build_tables();
    int64_t nb = M / 32;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < nb; ++j)
            scales_t[k * nb + j] = mxfp8_encode_block(
                x + (j * 32) * ldx + k, ldx, 32, codes_t + k * M + j * 32);
    return 0;
}

/* Dequantize MXFP8: y = bf16( fl32( E4M3(code) * 2^(e-127) ) ), blocks of
 * 32 along each row of codes [R x C]; scales [R x C/32] (logical layout).
 * The binary32 product is formed exactly in binary64 and then rounded to
 * binary32 (one rounding, as a binary32 multiply does), then to bf16. */
int oracle_mxfp8_dequantize(const uint8_t* codes, const uint8_t* scales,
                            int64_t R, int64_t C, uint16_t* y) {
    if (C % 32 != 0) return -1;
    int64_t nb = C / 32;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            double s = e8m0_decode(scales[r * nb + c / 32]);
            float p = (float)(e4m3_decode(codes[r * C + c]) * s);
            y[r * C + c] = rne_bf16_from_f32(p);
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* NVFP4 (formats section + NVFP4 recipe section).                           */
/* ------------------------------------------------------------------------ */

/* max |x| over R rows of C values (exact; bf16 values are exact floats). */
float oracle_bf16_amax(const uint16_t* x, int64_t R, int64_t C, int64_t ldx) {
    double a = 0.0;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            double v = fabs(bf16_decode(x[r * ldx + c]));
            if (v > a) a = v;
        }
    return (float)a;                      /* exact: a is a bf16 value */
}

/* Second-level FP32 scale: a decode scale, S = amax / (6 * 448). */
float oracle_nvfp4_tensor_scale(float amax) {
    const float fp4_max_times_e4m3_max = 2688.0f;  /* 6 * 448, exact */
    return amax / fp4_max_times_e4m3_max;
}

/* Encode one 16-value block given the FP32 scale S.  Writes 16 E2M1 codes
 * (one per byte, unpacked) and returns the E4M3 block-scale byte. */
static uint8_t nvfp4_encode_block(const uint16_t* x, float S,
                                  uint8_t* codes16) {
    float ab = 0.0f;
    for (int i = 0; i < 16; ++i) {
        float v = fabsf((float)bf16_decode(x[i]));
        if (v > ab) ab = v;
    }
    uint8_t sb;
    if (S == 0.0f) {
        sb = 0x00;
    } else {
        float six_s = 6.0f * S;
        float t = ab / six_s;
        sb = rne_e4m3((double)t);
    }
    float d = (float)T_E4M3[sb] * S;   /* E4M3 value is exact in binary32 */
    float enc;
    if (d == 0.0f) {
        enc = 0.0f;
    } else {
        enc = 1.0f / d;
        if (enc > FLT_MAX) enc = FLT_MAX;
    }
    for (int i = 0; i < 16; ++i) {
        float v = (float)bf16_decode(x[i]) * enc;
        codes16[i] = rne_e2m1((double)v);
    }
    return sb;
}

/* Encode R rows of C values (C % 16 == 0) with FP32 scales: row r uses
 * S[r * s_stride] (s_stride = 1: one scale per row, 0: one shared scale).
 * codes [R x C/2] packed, lower-index element in the low nibble;
 * scales [R x C/16]. */
int oracle_nvfp4_encode_rows(const uint16_t* x, int64_t R, int64_t C,
                             int64_t ldx, const float* S, int64_t s_stride,
                             uint8_t* codes, uint8_t* scales) {
    if (C % 16 != 0) return -1;
    build_tables();
    int64_t nb = C / 16;
    uint8_t q[16];
    for (int64_t r = 0; r < R; ++r) {
        float s = S[r * s_stride];
        for (int64_t j = 0; j < nb; ++j) {
            scales[r * nb + j] = nvfp4_encode_block(x + r * ldx + j * 16, s, q);
            for (int i = 0; i < 8; ++i)
                codes[r * (C / 2) + j * 8 + i] =
                    (uint8_t)((q[2 * i] & 0xF) | ((q[2 * i + 1] & 0xF) << 4));
        }
    }
    return 0;
}

/* Per-token quantization: S_t = amax(row t) / 2688, then encode the row. */
int oracle_nvfp4_quantize_per_token(const uint16_t* x, int64_t T, int64_t H,
                                    int64_t ldx, uint8_t* codes,
                                    uint8_t* scales, float* token_scales) {
    if (H % 16 != 0) return -1;
    for (int64_t t = 0; t < T; ++t)
        token_scales[t] =
            oracle_nvfp4_tensor_scale(oracle_bf16_amax(x + t * ldx, 1, H, H));
    return oracle_nvfp4_encode_rows(x, T, H, ldx, token_scales, 1, codes,
                                    scales);
}

/* Dequantize NVFP4: y = bf16( fl32( fl32(E2M1(c) * E4M3(sb)) * S ) ).
 * codes [R x C/2], scales [R x C/16]; row r uses S[r * s_stride]. */
int oracle_nvfp4_dequantize(const uint8_t* codes, const uint8_t* scales,
                            const float* S, int64_t s_stride, int64_t R,
                            int64_t C, uint16_t* y) {
    if (C % 16 != 0) return -1;
    int64_t nb = C / 16;
    for (int64_t r = 0; r < R; ++r) {
        float s = S[r * s_stride];
        for (int64_t c = 0; c < C; ++c) {
            uint8_t byte = codes[r * (C / 2) + c / 2];
            uint8_t q = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
            float bs = (float)e4m3_decode(scales[r * nb + c / 16]);
            float p = (float)e2m1_decode(q) * bs;  /* exact (<= 6 bits) */
            float v = p * s;
            y[r * C + c] = rne_bf16_from_f32(v);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Swizzled scale layout (not on the pages: the 128x4-tile layout that      */
/* block-scaled tensor-core MMA reads).  Logical scale matrix [R x C] ->    */
/* tiles of 128 rows x 4 columns, 512 bytes each, tile (rt, ct) at byte     */
/* (rt * ceil(C/4) + ct) * 512; inside a tile, element (r, c) sits at        */
/* (r % 32) * 16 + (r / 32) * 4 + c.  Padding bytes are 0x00.                */
/* ------------------------------------------------------------------------ */
int64_t oracle_swizzled_scale_bytes(int64_t R, int64_t C) {
    int64_t rt = (R + 127) / 128, ct = (C + 3) / 4;
    return rt * ct * 512;
}

int oracle_scale_swizzle(const uint8_t* logical, int64_t R, int64_t C,
                         uint8_t* out) {
    int64_t ct_n = (C + 3) / 4;
    memset(out, 0, (size_t)oracle_swizzled_scale_bytes(R, C));
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            int64_t tile = (r / 128) * ct_n + (c / 4);
            int64_t rr = r % 128, cc = c % 4;
            out[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cc] =
                logical[r * C + c];
        }
    return 0;
}

int oracle_scale_unswizzle(const uint8_t* swz, int64_t R, int64_t C,
                           uint8_t* logical) {
    int64_t ct_n = (C + 3) / 4;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            int64_t tile = (r / 128) * ct_n + (c / 4);
            int64_t rr = r % 128, cc = c % 4;
            logical[r * C + c] =
                swz[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cc];
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 with one FP32 scale per block: the DeepSeek-V3-style recipe of  */
/* "Miles: end-to-end MXFP8 and per-token NVFP4 RL", introduction (weights  */
/* in 128x128 blocks, activations in 1x128 tiles, scales computed online    */
/* per tile or block) and MXFP8 recipe section (that recipe stores forward  */
/* activations in 1x128 tiles and, before the backward GEMM, dequantizes    */
/* and requantizes them in the backward orientation).  The pages give no    */
/* formula for the scale; the reading used here is the one the NVFP4        */
/* second level uses, with 448 (the E4M3 maximum) as the code range:        */
/*   a = max |x| over the block (exact),                                     */
/*   S = fl(a / 448)              (a decode scale: value = code * S),        */
/*   enc = fl(1 / S), FLT_MAX-clamped; 0 when S = 0,                         */
/*   code = RNE_E4M3(fl(x * enc)), saturating at 448, sign kept;             */
/*   dequant y = RNE_bf16(fl(E4M3(code) * S)).                               */
/* Blocks are br x bc (1 x 128 tiles or 128 x 128 blocks); R % br == 0 and  */
/* C % bc == 0.  codes [R x C]; scales [R/br x C/bc] row-major.             */
/* ------------------------------------------------------------------------ */
float oracle_fp8blk_scale(float amax) {
    const float e4m3_max = 448.0f;
    return amax / e4m3_max;
}

int oracle_fp8blk_quantize(const uint16_t* x, int64_t R, int64_t C,
                           int64_t ldx, int64_t br, int64_t bc,
                           uint8_t* codes, float* scales) {
    if (R < 0 || C < 0 || br < 1 || bc < 1 || R % br || C % bc || ldx < C)
        return 1;
    build_tables();
    const int64_t nbc = C / bc;
    for (int64_t bi = 0; bi < R / br; ++bi)
        for (int64_t bj = 0; bj < nbc; ++bj) {
            float a = 0.0f;
            for (int64_t r = bi * br; r < (bi + 1) * br; ++r)
                for (int64_t c = bj * bc; c < (bj + 1) * bc; ++c) {
                    float v = fabsf((float)bf16_decode(x[r * ldx + c]));
                    if (v > a) a = v;
                }
            float s = oracle_fp8blk_scale(a);
            /* Stored before enc is derived: gcc -O2 otherwise concludes
             * from "1/s > FLT_MAX" that s is 0 and stores 0 for a
             * subnormal s (whose reciprocal overflows). */
            scales[bi * nbc + bj] = s;
            float enc;
            if (s == 0.0f) {
                enc = 0.0f;
            } else {
                enc = 1.0f / s;
                if (enc > FLT_MAX) enc = FLT_MAX;
            }
            for (int64_t r = bi * br; r < (bi + 1) * br; ++r)
                for (int64_t c = bj * bc; c < (bj + 1) * bc; ++c) {
                    float v = (float)bf16_decode(x[r * ldx + c]) * enc;
                    codes[r * C + c] = rne_e4m3((double)v);
                }
        }
    return 0;
}

int oracle_fp8blk_dequantize(const uint8_t* codes, const float* scales,
                             int64_t R, int64_t C, int64_t br, int64_t bc,
                             uint16_t* y) {
    if (R < 0 || C < 0 || br < 1 || bc < 1 || R % br || C % bc) return 1;
    const int64_t nbc = C / bc;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            float s = scales[(r / br) * nbc + c / bc];
            float v = (float)e4m3_decode(codes[r * C + c]) * s;
            y[r * C + c] = rne_bf16_from_f32(v);
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* NVFP4 with the stabilizers of the original NVFP4 pretraining recipe     */
/* ("Miles: end-to-end MXFP8 and per-token NVFP4 RL", NVFP4 recipe         */
/* section: that recipe adds stochastic rounding, applied to gradients to  */
/* make the quantized values unbiased, and Random Hadamard Transforms,     */
/* which disperse block-level outliers of weight-gradient GEMM inputs).    */
/* The pages give no formulas; the readings used here:                     */
/*  - random bits: Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel    */
/*    random numbers: as easy as 1, 2, 3", SC 2011), a counter-based        */
/*    generator, so every element's bits depend only on (seed, position);  */
/*  - RHT: each 16-value block x (along the row) becomes                   */
/*    y = (1/4) H16 (s * x), H16 the Sylvester Hadamard matrix, s the 16   */
/*    signs given by the low 16 bits of word 0 of Philox(counter 0, key    */
/*    (seed, 1)) (bit i set -> s_i = -1); evaluated in binary32 as the     */
/*    four butterfly stages h = 1, 2, 4, 8 ((a, b) -> (a + b, a - b) on    */
/*    elements i, i + h with i & h == 0), then times 1/4 (exact);          */
/*  - the per-token FP32 scale and the E4M3 block scales follow Algorithm  */
/*    2 on the (transformed) binary32 values;                              */
/*  - SR: element (r, c) takes u = (w >> 8) * 2^-24, w the 32-bit word     */
/*    c % 8 of Philox(counter (r, c / 8, 0, 0), key (seed, 2)) (word j is  */
/*    the low half of output j / 2 for even j, the high half for odd j);   */
/*    |v| = |fl(y * enc)| saturated at 6 rounds up to the next E2M1        */
/*    magnitude iff u < (|v| - lo) / (hi - lo), lo <= |v| < hi the         */
/*    bracketing magnitudes (that ratio is exact in binary32: hi - lo is a */
/*    power of two and |v| - lo is exact); values on the grid stay; sign   */
/*    kept.                                                                */
/* ------------------------------------------------------------------------ */
static uint64_t mulhi64(uint64_t a, uint64_t b, uint64_t* lo) {
    /* 64 x 64 -> 128 bits from four 32 x 32 products */
    uint64_t a0 = a & 0xffffffffu, a1 = a >> 32;
    uint64_t b0 = b & 0xffffffffu, b1 = b >> 32;
    uint64_t p00 = a0 * b0, p01 = a0 * b1, p10 = a1 * b0, p11 = a1 * b1;
    uint64_t mid = (p00 >> 32) + (p01 & 0xffffffffu) + (p10 & 0xffffffffu);
    *lo = (mid << 32) | (p00 & 0xffffffffu);
    return p11 + (p01 >> 32) + (p10 >> 32) + (mid >> 32);
}

void oracle_philox4x64(const uint64_t ctr_in[4], const uint64_t key_in[2],
                       uint64_t out[4]) {
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    uint64_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t lo0, lo1;
        uint64_t hi0 = mulhi64(M0, c[0], &lo0);
        uint64_t hi1 = mulhi64(M1, c[2], &lo1);
        uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
        k0 += W0;
        k1 += W1;
    }
    for (int i = 0; i < 4; ++i) out[i] = c[i];
}

static uint32_t philox_word(uint64_t seed, uint64_t stream, uint64_t c0,
                            uint64_t c1, int j) {
    const uint64_t ctr[4] = {c0, c1, 0, 0}, key[2] = {seed, stream};
    uint64_t out[4];
    oracle_philox4x64(ctr, key, out);
    uint64_t w = out[j / 2];
    return (uint32_t)((j & 1) ? (w >> 32) : (w & 0xffffffffu));
}

/* The 16 RHT signs of a seed, bit i set -> s_i = -1. */
uint32_t oracle_rht_signs(uint64_t seed) {
    return philox_word(seed, 1, 0, 0, 0) & 0xffffu;
}

/* y = (1/4) H16 (s * x) in binary32, butterfly order as stated above. */
void oracle_rht16(const float* x, uint32_t signs, float* y) {
    float v[16];
    for (int i = 0; i < 16; ++i) v[i] = ((signs >> i) & 1) ? -x[i] : x[i];
    for (int h = 1; h < 16; h <<= 1)
        for (int i = 0; i < 16; ++i)
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
    for (int i = 0; i < 16; ++i) y[i] = v[i] * 0.25f;
}

/* E2M1 code of v with stochastic rounding by u in [0, 1). */
static uint8_t sr_e2m1(float v, float u) {
    int neg = signbit(v) ? 1 : 0;
    float a = fabsf(v);
    if (a > 6.0f) a = 6.0f;
    int lo = 0;                                  /* largest magnitude <= a */
    for (int c = 0; c <= 7; ++c)
        if (T_E2M1[c] <= (double)a) lo = c;
    int code = lo;
    if ((double)a != T_E2M1[lo]) {
        float frac = (a - (float)T_E2M1[lo]) /
                     ((float)T_E2M1[lo + 1] - (float)T_E2M1[lo]);
        if (u < frac) code = lo + 1;
    }
    return (uint8_t)(code | (neg << 3));
}

/* Per-token NVFP4 of x [R x C] (C % 16 == 0) with the optional RHT (flags
 * bit 0) and SR (bit 1); row r of x is row row0 + r of the tensor (the SR
 * counters use that index).  codes [R x C/2] packed, low nibble = lower
 * index; scales [R x C/16] logical; S [R]. */
int oracle_nvfp4_rht_sr_rows(const uint16_t* x, int64_t R, int64_t C,
                             int64_t ldx, uint64_t seed, int flags,
                             int64_t row0, uint8_t* codes, uint8_t* scales,
                             float* S_out) {
    if (R < 0 || C < 0 || C % 16 || ldx < C) return 1;
    build_tables();
    const uint32_t signs = oracle_rht_signs(seed);
    const int64_t nb = C / 16;
    float* y = (float*)malloc(sizeof(float) * (size_t)(C > 0 ? C : 1));
    if (!y) return 2;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            float xb[16];
            for (int i = 0; i < 16; ++i)
                xb[i] = (float)bf16_decode(x[r * ldx + b * 16 + i]);
            if (flags & 1) oracle_rht16(xb, signs, &y[b * 16]);
            else memcpy(&y[b * 16], xb, sizeof(xb));
        }
        float at = 0.0f;
        for (int64_t c = 0; c < C; ++c)
            if (fabsf(y[c]) > at) at = fabsf(y[c]);
        const float S = at / 2688.0f;
        S_out[r] = S;
        for (int64_t b = 0; b < nb; ++b) {
            float ab = 0.0f;
            for (int i = 0; i < 16; ++i)
                if (fabsf(y[b * 16 + i]) > ab) ab = fabsf(y[b * 16 + i]);
            uint8_t sb = 0x00;
            if (S != 0.0f) sb = rne_e4m3((double)(ab / (6.0f * S)));
            scales[r * nb + b] = sb;
            float d = (float)T_E4M3[sb] * S;
            float enc;
            if (d == 0.0f) {
                enc = 0.0f;
            } else {
                enc = 1.0f / d;
                if (enc > FLT_MAX) enc = FLT_MAX;
            }
            uint8_t q[16];
            for (int i = 0; i < 16; ++i) {
                float v = y[b * 16 + i] * enc;
                if (flags & 2) {
                    const int64_t c = b * 16 + i;
                    const uint32_t w = philox_word(seed, 2, (uint64_t)(row0 + r),
                                                   (uint64_t)(c / 8), (int)(c % 8));
                    const float u = (float)(w >> 8) * 0x1p-24f;
                    q[i] = sr_e2m1(v, u);
                } else {
                    q[i] = rne_e2m1((double)v);
                }
            }
            for (int i = 0; i < 8; ++i)
                codes[r * (C / 2) + b * 8 + i] =
                    (uint8_t)(q[2 * i] | (q[2 * i + 1] << 4));
        }
    }
    free(y);
    return 0;
}
