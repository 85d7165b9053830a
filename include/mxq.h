/*
 * mxq.h -- C ABI of libmxq, the GB300 (sm_103a) MXFP8 / NVFP4 quantizer
 * library.
 *
 * Sources are cited as (page title, section):
 *   [MILES]  "Miles: end-to-end MXFP8 and per-token NVFP4 RL"
 *   [RLQ]    "Using Quantization in RL"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are plain pointers.  Unless stated otherwise every tensor
 *    pointer is a DEVICE pointer on the current CUDA device; bf16 data is
 *    passed as `const void*` holding IEEE bfloat16 values.  Only the
 *    pointer table of nvfp4_quantize_weight_shared and its part_rows array
 *    live in HOST memory.
 *  - Every device pointer must be 16-byte aligned (MXQ_ERR_ALIGN).
 *  - The caller owns every buffer.  The library never allocates or frees
 *    memory and keeps no per-call state.  Calls that need scratch take a
 *    caller-provided workspace and have a *_workspace_size query.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *    work is enqueued on it; no entry point synchronizes.
 *  - Arguments are validated on the host before anything is launched; a
 *    rejected call writes nothing and returns a non-zero mxq_status.  No
 *    C++ exception crosses this ABI.
 *  - Inputs must be finite bf16 values (NaN / Inf inputs are outside the
 *    contract).
 *  - Results are deterministic and bit-exact with respect to the algorithm
 *    stated at each entry point: the same input bytes always give the same
 *    output bytes, on any launch configuration.
 *  - Bounded device waits: the kernels of the entry points marked
 *    "[bounded waits]" wait on the GPU (for data copies in flight, for
 *    other CTAs); every such wait gives up after about one second, skips
 *    the rest of the kernel's work and records an error word.  The call
 *    itself has already returned MXQ_OK by then, and its outputs are
 *    incomplete: the failure is reported only by the next
 *    mxq_get_last_error() (which synchronizes the device).  Callers that
 *    must know check it after the work has completed.
 *
 * Scale layouts (argument `scale_layout`)
 * ---------------------------------------
 *  MXQ_SCALE_LINEAR:   the logical scale matrix [R x C] (one byte per
 *                      block), row-major, no padding.
 *  MXQ_SCALE_SWIZZLED: the 128x4-tile layout that block-scaled tensor-core
 *                      MMA reads: R padded to a multiple of 128, C to a
 *                      multiple of 4; tile (rt, ct) of 512 bytes at byte
 *                      (rt * ceil(C/4) + ct) * 512; element (r, c) inside
 *                      its tile at (r % 32) * 16 + ((r % 128) / 32) * 4 +
 *                      (c % 4).  Padding bytes are written as 0x00.
 *  mxq_scale_bytes() gives the buffer size of either layout.
 */
#ifndef MXQ_H
#define MXQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int mxq_status;

#define MXQ_OK            0  /* success                                    */
#define MXQ_ERR_NULL      1  /* a required pointer is NULL                 */
#define MXQ_ERR_SHAPE     2  /* a size is negative or not a block multiple */
#define MXQ_ERR_ALIGN     3  /* a pointer or a leading dimension is not
                                16-byte aligned                            */
#define MXQ_ERR_LAYOUT    4  /* unknown scale_layout / scale mode          */
#define MXQ_ERR_WORKSPACE 5  /* workspace NULL or smaller than required    */
#define MXQ_ERR_CUDA      6  /* a CUDA call or kernel launch failed        */
#define MXQ_ERR_TIMEOUT   7  /* a bounded device-side wait gave up         */
#define MXQ_ERR_ARG       8  /* any other invalid argument                 */

#define MXQ_SCALE_LINEAR   0
#define MXQ_SCALE_SWIZZLED 1

/* FP32 scale modes of dequantize_nvfp4. */
#define MXQ_S_PER_ROW   0    /* S[b * rows + r]: one scale per row (token)  */
#define MXQ_S_PER_BATCH 1    /* S[b]: one scale per batch entry (group)     */

/* Human-readable name of a status code (static string, never NULL). */
const char* mxq_status_string(mxq_status s);

/* Library version, as 10000 * major + 100 * minor + patch. */
int mxq_version(void);

/* Bytes of a scale buffer for a logical [rows x cols] scale matrix in the
 * given layout; -1 for a bad layout or negative size. */
int64_t mxq_scale_bytes(int64_t rows, int64_t cols, int scale_layout);

/* Returns and clears the error word that bounded device-side waits set
 * when they give up (MXQ_ERR_TIMEOUT), then the last CUDA runtime error
 * (MXQ_ERR_CUDA); MXQ_OK if neither is set.  Synchronizes the device. */
mxq_status mxq_get_last_error(void);

/* Self-test of the device-side failure detection (the pages have no
 * counterpart; it exists so that tests can check the path without making
 * the GPU fault or hang).  Launches one CTA whose bounded mbarrier wait --
 * the same wait the kernels use -- waits on a barrier nothing completes;
 * after 20 ms it gives up and records the error word, so the next
 * mxq_get_last_error returns MXQ_ERR_TIMEOUT and the context stays usable.
 * Returns MXQ_ERR_CUDA if the launch fails. */
mxq_status mxq_selftest_wait_timeout(void* stream);

/* Host-side fault injection for tests of the error paths: mode 0 = off,
 * 1 = every entry point fails its launch with MXQ_ERR_CUDA without
 * launching, 2 = argument checks fail with MXQ_ERR_ARG.  Also read once
 * from the environment variable MXQ_FAULT_INJECT ("launch" / "argcheck").
 * Nothing faults on the GPU. */
void mxq_set_fault_inject(int mode);

/* --------------------------------------------------------------------- */
/* MXFP8 quantize, rowwise and columnwise copies in one pass.             */
/*                                                                       */
/* [MILES] formats section: E4M3 elements, every 32 consecutive values    */
/* share one E8M0 (power-of-two) scale, the block is one-dimensional, and */
/* the decoded scale is rounded up so the block maximum is not clipped.   */
/* [MILES] MXFP8 recipe section: rowwise 1x32 and columnwise 32x1 blocks  */
/* are numerically different and are each quantized from the full-        */
/* precision data; both copies are materialized by one quantization.      */
/*                                                                       */
/* Per block B (32 values): a = max|x|; k = smallest integer in           */
/* [-127, 127] with 448 * 2^k >= a (a = 0 gives k = -127); scale byte =   */
/* k + 127; code_i = E4M3 round-to-nearest-even of x_i * 2^-k (exact      */
/* product, never saturates).                                             */
/*                                                                       */
/* x            bf16 [M x K], row stride ldx elements (ldx >= K,           */
/*              ldx % 8 == 0).                                            */
/* row_codes    u8 [M x K] (row stride K): blocks along K.                 */
/* row_scales   E8M0, logical [M x K/32], in scale_layout.                 */
/* col_codes_t  u8 [K x M]: the columnwise copy stored TRANSPOSED, byte    */
/*              (k, m) at k * M + m, so each 32x1 block is 32 contiguous   */
/*              bytes (the K-major operand of the backward GEMMs).         */
/* col_scales_t E8M0, logical [K x M/32], in scale_layout.                 */
/* Either pair may be NULL (both pointers of the pair) to skip that copy;  */
/* at least one pair must be given.  K % 32 == 0; M % 32 == 0 when the     */
/* columnwise copy is requested.  M == 0 or K == 0 is a no-op.            */
/* [bounded waits]: a device-side wait that gives up is reported by the   */
/* next mxq_get_last_error(), not by this call's status.                  */
/* --------------------------------------------------------------------- */
mxq_status mxfp8_quantize_rowcol(const void* x, int64_t M, int64_t K,
                                 int64_t ldx, uint8_t* row_codes,
                                 uint8_t* row_scales, uint8_t* col_codes_t,
                                 uint8_t* col_scales_t, int scale_layout,
                                 void* stream);

/* --------------------------------------------------------------------- */
/* NVFP4 quantize with one FP32 scale per token.                          */
/*                                                                       */
/* [MILES] formats section: E2M1 elements, one E4M3 scale per 16 values   */
/* rounded to the nearest representable value, and an FP32 scale over a   */
/* larger scope.  [MILES] NVFP4 recipe section: that FP32 scale is one    */
/* per token, computed online inside the same call that emits the packed  */
/* FP4 values and the E4M3 block scales, so a token's bytes never depend  */
/* on the rest of the batch.                                              */
/*                                                                       */
/* Per token t (all IEEE binary32, round-to-nearest-even, no FTZ):        */
/*   S_t  = amax_t / 2688                        (2688 = 6 * 448)         */
/*   sb   = E4M3_RNE( amax_b / (6 * S_t) )  per 16-block b (0 if S_t = 0) */
/*   enc  = 1 / (E4M3(sb) * S_t)   (0 if that product is 0, else clamped  */
/*                                  to FLT_MAX)                           */
/*   code = E2M1_RNE( x * enc ), saturating at +-6, sign kept              */
/* Two codes per byte, the lower-index element in the LOW nibble.         */
/*                                                                       */
/* x            bf16 [T x H], row stride ldx (ldx >= H, ldx % 8 == 0);     */
/*              a ragged batch is passed flattened.                        */
/* codes        u8 [T x H/2].                                              */
/* block_scales E4M3, logical [T x H/16], in scale_layout.                 */
/* token_scales f32 [T] (the decode scales S_t).                           */
/* H % 16 == 0.  T == 0 is a no-op.                                       */
/* --------------------------------------------------------------------- */
mxq_status nvfp4_quantize_per_token(const void* x, int64_t T, int64_t H,
                                    int64_t ldx, uint8_t* codes,
                                    uint8_t* block_scales,
                                    float* token_scales, int scale_layout,
                                    void* stream);

/* --------------------------------------------------------------------- */
/* NVFP4 per-token quantize of gathered rows (routing gather fused in).    */
/*                                                                       */
/* [MILES] NVFP4 recipe section (SwiGLU MoE layers: the tokens routed to  */
/* an expert form that expert's rows of the gate/up GEMM) and experiments */
/* section (per-token NVFP4 activation quantize): output row t is the     */
/* per-token quantization of x row row_index[t], exactly as               */
/* nvfp4_quantize_per_token would produce it for that row.                 */
/*                                                                       */
/* x            bf16 [T_src x H] (row stride ldx), device.                */
/* row_index    int32 [T], device (4-byte aligned).  An index outside     */
/*              [0, T_src) gives a zero row (codes 0, block scales 0,     */
/*              token scale 0): the padding rows of an expert group.      */
/* codes, block_scales, token_scales: as nvfp4_quantize_per_token, for T  */
/*              output rows.                                              */
/* --------------------------------------------------------------------- */
mxq_status nvfp4_quantize_per_token_gather(
    const void* x, int64_t T_src, int64_t H, int64_t ldx,
    const int32_t* row_index, int64_t T, uint8_t* codes,
    uint8_t* block_scales, float* token_scales, int scale_layout,
    void* stream);

/* --------------------------------------------------------------------- */
/* NVFP4 weight quantize with one FP32 scale shared by a group of parts.  */
/*                                                                       */
/* [MILES] NVFP4 recipe section: NVFP4 targets MoE expert weights; the    */
/* gate and up projections are fused into one GEMM, so both must share    */
/* the same FP32 scale during conversion and live weight update; the pair */
/* is quantized together.                                                 */
/*                                                                       */
/* Group g consists of num_parts parts; part p is a bf16 [part_rows[p] x  */
/* K] row-major matrix (row stride K) at device address                   */
/* parts[g * num_parts + p].  S_g = max over all its parts of |x| / 2688  */
/* (or group_scales_in[g] when that pointer is not NULL: a live update    */
/* reusing a stored scale), then each row is encoded exactly as in        */
/* nvfp4_quantize_per_token with S_g.  The output rows of a group are the */
/* parts' rows concatenated (R = sum part_rows).                          */
/*   gate/up pair: num_parts = 2, part_rows = {768, 768};                  */
/*   down:         a second call with num_parts = 1.                      */
/*                                                                       */
/* parts          HOST array of num_groups * num_parts device pointers.    */
/* part_rows      HOST array [num_parts].                                  */
/* codes          u8 [num_groups x R x K/2].                                */
/* block_scales   num_groups consecutive scale matrices, each logical      */
/*                [R x K/16] in scale_layout, mxq_scale_bytes(R, K/16)     */
/*                bytes apart.                                             */
/* group_scales   f32 [num_groups] (out).                                  */
/* group_scales_in f32 [num_groups] or NULL.                               */
/* ws / ws_bytes  device workspace of at least                             */
/*                nvfp4_quantize_weight_shared_workspace_size() bytes.     */
/* K % 16 == 0; 1 <= num_parts <= 4.                                       */
/* [bounded waits]: a device-side wait that gives up is reported by the   */
/* next mxq_get_last_error(), not by this call's status.                  */
/* --------------------------------------------------------------------- */
size_t nvfp4_quantize_weight_shared_workspace_size(int64_t num_groups);

mxq_status nvfp4_quantize_weight_shared(
    int64_t num_groups, int num_parts, const void* const* parts,
    const int64_t* part_rows, int64_t K, uint8_t* codes,
    uint8_t* block_scales, float* group_scales, const float* group_scales_in,
    int scale_layout, void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------- */
/* NVFP4 weight quantize with a shared FP32 scale, allocating nothing.    */
/*                                                                       */
/* The pages have no counterpart to this entry point: it exists for       */
/* callers that cannot allocate device memory -- plug-ins inside a host   */
/* framework that owns every device allocation and offers no allocator,   */
/* and latency-critical loops where a cudaMalloc (which may synchronize   */
/* the device) is not allowed -- and so cannot provide the workspace of   */
/* nvfp4_quantize_weight_shared.                                          */
/*                                                                       */
/* Same arguments, layouts and results as nvfp4_quantize_weight_shared,   */
/* without ws / ws_bytes: the per-group scratch lives in a fixed device   */
/* array inside the library (32.25 KiB, held on every GPU that loads the  */
/* library until the process exits).                                      */
/*  - num_groups must not exceed                                          */
/*    nvfp4_quantize_weight_shared_noalloc_max_groups() (4096); larger    */
/*    requests are rejected with MXQ_ERR_SHAPE before anything runs.      */
/*  - The first call on a device looks up the array's device address      */
/*    (cudaGetSymbolAddress) with that device current, and a call that    */
/*    finds the device's context replaced (cudaDeviceReset) looks it up   */
/*    again; make the first call on a device, and the first after a       */
/*    reset, before any stream capture on the device.                     */
/*  - Honours the host-side fault injection of mxq_set_fault_inject like  */
/*    every other entry point.                                            */
/*  - Every call shares the array.  A call clears the words it uses on    */
/*    its own stream before using them, so back-to-back calls on one      */
/*    stream are correct; calls whose work overlaps on the GPU (unordered */
/*    streams) race on the array.                                         */
/*  - Calls no cudaMalloc, cudaFree or allocating routine.                */
/* [bounded waits]: a device-side wait that gives up is reported by the   */
/* next mxq_get_last_error(), not by this call's status.                  */
/* --------------------------------------------------------------------- */
int64_t nvfp4_quantize_weight_shared_noalloc_max_groups(void);

mxq_status nvfp4_quantize_weight_shared_noalloc(
    int64_t num_groups, int num_parts, const void* const* parts,
    const int64_t* part_rows, int64_t K, uint8_t* codes,
    uint8_t* block_scales, float* group_scales, const float* group_scales_in,
    int scale_layout, void* stream);

/* --------------------------------------------------------------------- */
/* MXFP8 dequantize to bf16.                                              */
/*                                                                       */
/* [MILES] backward-mode section: dequantized backward feeds the BF16     */
/* backward GEMMs with BF16 dequantizations of the exact low-precision    */
/* operands of the forward pass.  [RLQ] "Two Ways to Configure Training   */
/* and Inference": a stored value is code x scale.                        */
/*                                                                       */
/* y = bf16_RNE( fp32( E4M3(code) * 2^(scale - 127) ) ), blocks of 32      */
/* along each row.  Exact for codes produced from bf16 data, except that  */
/* a block of bf16-max magnitude overflows to +-inf (2^128).  The E8M0   */
/* NaN byte 0xFF and the E4M3 NaN codes 0x7F / 0xFF decode to NaN.        */
/* codes u8 [rows x cols]; scales logical [rows x cols/32] in              */
/* scale_layout; y bf16 [rows x cols].  Dequantize the columnwise copy by */
/* passing (col_codes_t, col_scales_t, K, M): the result is X^T.          */
/* cols % 32 == 0.                                                        */
/* --------------------------------------------------------------------- */
mxq_status dequantize_mxfp8(const uint8_t* codes, const uint8_t* scales,
                            int64_t rows, int64_t cols, int scale_layout,
                            void* y, void* stream);

/* --------------------------------------------------------------------- */
/* NVFP4 dequantize to bf16.                                              */
/*                                                                       */
/* Same sources as dequantize_mxfp8.                                      */
/* y = bf16_RNE( fp32( fp32(E2M1(c) * E4M3(sb)) * S ) ); the inner        */
/* product is exact.  `batch` matrices of [rows x cols], stored back to   */
/* back: codes [batch x rows x cols/2], block_scales batch consecutive    */
/* scale matrices of mxq_scale_bytes(rows, cols/16) bytes, y [batch x rows */
/* x cols].  S: s_mode MXQ_S_PER_ROW -> S[b * rows + r] (per-token data,  */
/* batch = 1); MXQ_S_PER_BATCH -> S[b] (one weight group per batch        */
/* entry).  cols % 16 == 0.                                                */
/* --------------------------------------------------------------------- */
mxq_status dequantize_nvfp4(const uint8_t* codes, const uint8_t* block_scales,
                            const float* S, int s_mode, int64_t batch,
                            int64_t rows, int64_t cols, int scale_layout,
                            void* y, void* stream);

/* --------------------------------------------------------------------- */
/* NVFP4 per-token quantize with the stabilizers of the original NVFP4    */
/* pretraining recipe.                                                    */
/*                                                                       */
/* [MILES] NVFP4 recipe section: that recipe uses stochastic rounding      */
/* (SR, applied to gradients so the quantized values are unbiased) and    */
/* Random Hadamard Transforms (RHT, dispersing block-level outliers of    */
/* weight-gradient GEMM inputs); the RL recipe leaves both out.           */
/*                                                                       */
/* Same outputs and layouts as nvfp4_quantize_per_token.  flags:          */
/*   MXQ_NVFP4_RHT: each 16-value block x becomes (1/4) H16 (s * x)        */
/*     before quantization (H16 the Sylvester Hadamard matrix, s 16 signs  */
/*     drawn from the seed); S and the block scales are those of the      */
/*     transformed values, and dequantization returns transformed values  */
/*     (the inverse transform belongs to the consumer, where H cancels    */
/*     between two operands transformed with the same signs).             */
/*   MXQ_NVFP4_SR: E2M1 codes by stochastic rounding: |x * enc| rounds up  */
/*     to the next E2M1 magnitude with probability equal to its distance  */
/*     from the one below, over their spacing.                            */
/* Random bits: Philox4x64-10 keyed by seed, so the result depends only   */
/* on (seed, input); flags = 0 gives nvfp4_quantize_per_token's bytes.    */
/* H % 16 == 0, ldx % 8 == 0.                                             */
/* --------------------------------------------------------------------- */
#define MXQ_NVFP4_RHT 1
#define MXQ_NVFP4_SR  2
mxq_status nvfp4_quantize_per_token_rht_sr(const void* x, int64_t T,
                                           int64_t H, int64_t ldx,
                                           uint64_t seed, int flags,
                                           uint8_t* codes,
                                           uint8_t* block_scales,
                                           float* token_scales,
                                           int scale_layout, void* stream);

/* --------------------------------------------------------------------- */
/* FP8 E4M3 with one FP32 scale per block (the DeepSeek-V3-style recipe). */
/*                                                                       */
/* [MILES] introduction: that recipe scales weights in 128x128 blocks and */
/* activations in 1x128 tiles, one FP32 scale per tile or block computed  */
/* online.  [MILES] MXFP8 recipe section: it stores forward activations   */
/* in 1x128 tiles and converts them to the backward orientation by        */
/* dequantizing and requantizing before the backward GEMM.                */
/*   S = amax / 448 (FP32 decode scale), enc = 1 / S (0 when S = 0,       */
/*   FLT_MAX-clamped), code = RNE_E4M3(x * enc) saturating at +-448,      */
/*   dequant y = RNE_bf16(E4M3(code) * S); binary32 throughout.           */
/*                                                                       */
/* fp8_block_quantize: x bf16 [rows x cols], row stride ldx elements      */
/* (ldx >= cols, ldx % 8 == 0).  block_rows = 1: 1x128 tiles along rows;  */
/* block_rows = 128: 128x128 blocks (rows % 128 == 0).  cols % 128 == 0.  */
/* codes u8 [rows x cols]; scales f32 [rows/block_rows x cols/128],       */
/* row-major.  All pointers 16-byte aligned.                              */
/* [bounded waits] (block_rows = 128): a device-side wait that gives up   */
/* is reported by the next mxq_get_last_error(), not by this call's       */
/* status.                                                               */
/* --------------------------------------------------------------------- */
mxq_status fp8_block_quantize(const void* x, int64_t rows, int64_t cols,
                              int64_t ldx, int block_rows, uint8_t* codes,
                              float* scales, void* stream);

/* fp8_block_dequantize: bf16 y [rows x cols] from codes [rows x cols] and */
/* scales [rows/block_rows x cols/128]; same shape rules.                 */
mxq_status fp8_block_dequantize(const uint8_t* codes, const float* scales,
                                int64_t rows, int64_t cols, int block_rows,
                                void* y, void* stream);

/* fp8_block_requantize_transpose: the backward-orientation conversion of  */
/* 1x128-tile activations X [rows x cols] (codes, scales as produced by    */
/* fp8_block_quantize with block_rows = 1): X is dequantized to bf16       */
/* exactly as fp8_block_dequantize does and its transpose X^T [cols x rows] */
/* is quantized in 1x128 tiles: codes_t u8 [cols x rows], scales_t f32     */
/* [cols x rows/128].  rows % 128 == 0, cols % 128 == 0.                   */
mxq_status fp8_block_requantize_transpose(const uint8_t* codes,
                                          const float* scales, int64_t rows,
                                          int64_t cols, uint8_t* codes_t,
                                          float* scales_t, void* stream);

/* --------------------------------------------------------------------- */
/* Block-scaled GEMM consumers (5th-generation tensor cores).             */
/*                                                                       */
/* [MILES] MXFP8 recipe section: forward, weight-gradient and data-       */
/* gradient GEMMs consume the MXFP8 copies.  [MILES] experiments section: */
/* the per-token NVFP4 GEMM applies the per-token FP32 scale in the       */
/* kernel epilogue rather than as a separate operation.                   */
/*                                                                       */
/* mxq_gemm_mxfp8: C[m, n] = sum_k A[m, k] * B[k, n] with fp32             */
/* accumulation, where A is the rowwise MXFP8 copy of an [M x K] tensor    */
/* (a_codes [M x K], a_scales swizzled E8M0 [M x K/32]) and B is given as  */
/* B^T [N x K]: the columnwise copy of a [K x N] tensor (col_codes_t,      */
/* col_scales_t), or the rowwise copy of an [N x K] weight.  Scales must   */
/* be in MXQ_SCALE_SWIZZLED layout.  C is fp32 [M x N], row stride ldc    */
/* (ldc >= N, ldc % 4 == 0).  M % 128 == 0, N % 128 == 0, K % 128 == 0.    */
/* [bounded waits]: a device-side wait that gives up is reported by the   */
/* next mxq_get_last_error(), not by this call's status.                  */
/* --------------------------------------------------------------------- */
mxq_status mxq_gemm_mxfp8(const uint8_t* a_codes, const uint8_t* a_scales,
                          const uint8_t* bt_codes, const uint8_t* bt_scales,
                          int64_t M, int64_t N, int64_t K, float* C,
                          int64_t ldc, void* stream);

/* mxq_gemm_bf16_mxfp8: the dequantized-backward GEMM ([MILES] backward-  */
/* mode section: BF16 backward GEMMs on BF16 dequantizations of the exact  */
/* forward operands) without a bf16 copy of the quantized operand in HBM:  */
/*   C[m, n] = sum_k A[m, k] * Bq[k, n],                                  */
/* A bf16 [M x K] (row stride lda elements, lda >= K, lda % 8 == 0), B    */
/* given as B^T [N x K]: MXFP8 codes (bt_codes, row stride K) and swizzled */
/* E8M0 scales (bt_scales, 1x32 blocks along K) -- the columnwise copy of */
/* a [K x N] forward tensor; Bq = bf16_RNE(E4M3(code) * 2^(s - 127)),    */
/* bit-identical to dequantize_mxfp8 (exact unless the product leaves     */
/* bf16's normal range; the E8M0 byte 0xFF and E4M3 NaN codes give NaN).  */
/* The bf16 values of B are formed in shared memory only.  fp32            */
/* accumulation, fp32 C [M x N] (ldc >= N, ldc % 4 == 0).                  */
/* M % 128 == 0, N % 128 == 0, K % 64 == 0.                               */
/* [bounded waits]: a device-side wait that gives up is reported by the   */
/* next mxq_get_last_error(), not by this call's status.                  */
mxq_status mxq_gemm_bf16_mxfp8(const void* a, int64_t lda,
                               const uint8_t* bt_codes,
                               const uint8_t* bt_scales, int64_t M, int64_t N,
                               int64_t K, float* C, int64_t ldc, void* stream);

/* mxq_gemm_nvfp4_grouped: expert-grouped NVFP4 GEMM.  A holds the routed  */
/* activations of all groups, grouped contiguously: rows                  */
/* group_offsets[g] .. group_offsets[g+1] (HOST array of num_groups + 1    */
/* entries, group_offsets[0] == 0, every entry a multiple of 128: pad each */
/* group) use weight W_g.  a_codes [M_total x K/2], a_scales swizzled E4M3 */
/* [M_total x K/16], a_token_scales f32 [M_total] (as produced by          */
/* nvfp4_quantize_per_token).  w_codes [num_groups x N x K/2], w_scales    */
/* num_groups swizzled scale matrices of mxq_scale_bytes(N, K/16) bytes,   */
/* w_group_scales f32 [num_groups] (as produced by                         */
/* nvfp4_quantize_weight_shared).                                          */
/*   C[r, n] = a_token_scales[r] * w_group_scales[g] *                     */
/*             sum_k (E2M1 x E4M3)(a[r, k]) * (E2M1 x E4M3)(w_g[n, k])     */
/* with fp32 accumulation; C fp32 [M_total x N], row stride ldc.           */
/* N % 128 == 0, K % 256 == 0, num_groups <= 256.                          */
/* [bounded waits]: a device-side wait that gives up is reported by the   */
/* next mxq_get_last_error(), not by this call's status.                  */
/* --------------------------------------------------------------------- */
mxq_status mxq_gemm_nvfp4_grouped(
    const uint8_t* a_codes, const uint8_t* a_scales, const float* a_token_scales,
    const int64_t* group_offsets, int64_t num_groups, const uint8_t* w_codes,
    const uint8_t* w_scales, const float* w_group_scales, int64_t N, int64_t K,
    float* C, int64_t ldc, void* stream);

/* --------------------------------------------------------------------- */
/* MoE expert forward up to the activation: grouped NVFP4 gate/up GEMM    */
/* with SwiGLU in the epilogue.                                           */
/*                                                                       */
/* [MILES] NVFP4 recipe section: in SwiGLU MoE layers the gate and up     */
/* projections are one GEMM whose two halves share an FP32 weight scale;  */
/* experiments section: the per-token FP32 scale is applied in the GEMM   */
/* epilogue.  SwiGLU is its standard form, silu(gate) * up with           */
/* silu(z) = z / (1 + e^-z).                                              */
/*                                                                       */
/*   rows off[e] .. off[e+1] of A use expert e; with                       */
/*   s = S_tok[r] * S_w[e], g = s * (a . gate_e[j]), u = s * (a . up_e[j]): */
/*   h[r, j] = bf16( silu(g) * u ),  j < F.                               */
/*                                                                       */
/* a_*            per-token NVFP4 operand (e.g. from                       */
/*                nvfp4_quantize_per_token_gather), swizzled scales,      */
/*                rows = group_offsets[num_groups].                       */
/* group_offsets  HOST int64 [num_groups + 1], ascending multiples of 128. */
/* w_codes        u8 [num_groups x 2F x K/2]: per expert the F gate rows  */
/*                then the F up rows (nvfp4_quantize_weight_shared with   */
/*                parts {gate, up}); w_scales: per expert a swizzled      */
/*                [2F x K/16] matrix, mxq_scale_bytes(2F, K/16) apart;    */
/*                w_group_scales f32 [num_groups].                         */
/* h              bf16 [rows x F], row stride ldh elements (ldh % 8 == 0). */
/* F % 128 == 0, K % 256 == 0, num_groups <= 256.                         */
/* binary32 arithmetic before the bf16 rounding; silu uses a fast         */
/* exponential and divide (relative error below 2^-20, far inside bf16).  */
/* [bounded waits]: a device-side wait that gives up is reported by the   */
/* next mxq_get_last_error(), not by this call's status.                  */
/* --------------------------------------------------------------------- */
mxq_status mxq_moe_gate_up_swiglu_nvfp4(
    const uint8_t* a_codes, const uint8_t* a_scales, const float* a_token_scales,
    const int64_t* group_offsets, int64_t num_groups, const uint8_t* w_codes,
    const uint8_t* w_scales, const float* w_group_scales, int64_t F, int64_t K,
    void* h, int64_t ldh, void* stream);

/* --------------------------------------------------------------------- */
/* The grouped NVFP4 GEMM and the MoE gate/up + SwiGLU GEMM with the      */
/* routing gather in the GEMM's operand load.                             */
/*                                                                       */
/* [MILES] NVFP4 recipe section (SwiGLU MoE layers, gate and up fused     */
/* into one GEMM under one FP32 weight scale) and experiments section     */
/* (the per-token scale applied in the GEMM rather than as a separate     */
/* operation).  Per-token quantization does not depend on the batch, so   */
/* the unique tokens are quantized once (nvfp4_quantize_per_token with    */
/* MXQ_SCALE_LINEAR) and the GEMM gathers each routed row's codes (TMA    */
/* gather of four rows per instruction) and block scales as it loads A;   */
/* no routed copy of the tokens is written.                               */
/*                                                                       */
/* x_codes        u8 [T_src x K/2], x_scales its LINEAR E4M3 block scales */
/*                [T_src x K/16], x_token_scales f32 [T_src].              */
/* row_index      int32 [group_offsets[num_groups]] (device): routed row r */
/*                is token row_index[r]; an index outside [0, T_src) is a  */
/*                padding row, whose outputs are +0.                       */
/* Everything else, and every result byte, as mxq_gemm_nvfp4_grouped and */
/* mxq_moe_gate_up_swiglu_nvfp4 on the gathered operand that             */
/* nvfp4_quantize_per_token_gather writes.                                */
/* [bounded waits]: a device-side wait that gives up is reported by the   */
/* next mxq_get_last_error(), not by this call's status.                  */
/* --------------------------------------------------------------------- */
mxq_status mxq_gemm_nvfp4_grouped_gather(
    const uint8_t* x_codes, const uint8_t* x_scales, const float* x_token_scales,
    int64_t T_src, const int32_t* row_index, const int64_t* group_offsets,
    int64_t num_groups, const uint8_t* w_codes, const uint8_t* w_scales,
    const float* w_group_scales, int64_t N, int64_t K, float* C, int64_t ldc,
    void* stream);

mxq_status mxq_moe_gate_up_swiglu_nvfp4_gather(
    const uint8_t* x_codes, const uint8_t* x_scales, const float* x_token_scales,
    int64_t T_src, const int32_t* row_index, const int64_t* group_offsets,
    int64_t num_groups, const uint8_t* w_codes, const uint8_t* w_scales,
    const float* w_group_scales, int64_t F, int64_t K, void* h, int64_t ldh,
    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H */
