// nvfp4.cu -- NVFP4 quantize: E2M1 codes, one E4M3 scale per 16 values and
// one FP32 scale per token (activations) or per weight group (MoE weights,
// gate/up sharing one scale).
//
// "Miles: end-to-end MXFP8 and per-token NVFP4 RL", formats section: E2M1
// values with one E4M3 scale per 16-value block rounded to the nearest
// representable value, plus an FP32 scale over a larger scope.  NVFP4
// recipe section: the FP32 activation scale is one per token, computed
// online in the same call that emits the packed FP4 values and the block
// scales; gate and up weights share one FP32 scale and are quantized
// together.
//
// Arithmetic (IEEE binary32, round-to-nearest-even, no FTZ, no FMA):
//   S   = amax / 2688                 (2688 = 6 * 448; a decode scale)
//   sb  = E4M3_RNE( amax_b / (6 S) )  (0 when S = 0)
//   enc = 1 / (E4M3(sb) S)            (0 when that product is 0, clamped to
//                                      FLT_MAX otherwise)
//   q   = E2M1_RNE( x enc )           (saturating at +-6, sign kept)
//
// Design (sm_103a): HBM-streaming.  Per-token rows: one lane per 16-value
// block, R blocks per lane with all of a lane's loads in flight at once
// (non-allocating 16-byte loads), WPR warps per row joined by a named
// barrier for the row amax; the block's scale and codes come from binary32
// IEEE intrinsics and cvt.rn.satfinite.e2m1x2; one 8-byte code store per
// block, four block scales gathered by shuffles into one 32-bit store (four
// consecutive scale columns are contiguous in both layouts).  Weight groups
// use one persistent task-list kernel (see below): the amax tasks of a
// window of groups run ahead of that window's encode tasks, so the second
// read of a group is served from L2.
#include <float.h>

#include "common.cuh"
#include "launch.h"

namespace mxq {

namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int CTA_WARPS = 8;                 // 256 threads per CTA

struct RowOut {
  uint8_t* codes_row;   // H/2 bytes of this row
  uint8_t* scales;      // base of this row's scale matrix
  int64_t row;          // row index within the scale matrix
  int64_t col_tiles;    // swizzled: ceil(nblocks / 4)
  int64_t nblocks;      // H / 16
  int swizzled;
  int wide;             // rows 32-byte aligned: one 32-byte load per block
  uint8_t* stage;       // non-NULL: block scales go to this shared row
};

// 16 bf16 values of one block (two 16-byte chunks).
struct Blk {
  uint4 a, b;
};

// max |x| of the 16 values of a block, as a bf16 bit pattern (the sign
// bit left by max.xorsign.abs is cleared at the end).
__device__ __forceinline__ uint32_t block_absmax(const Blk& v) {
  const uint32_t m =
      bf16x2_maxabs(bf16x2_maxabs(bf16x2_maxabs(v.a.x, v.a.y),
                                  bf16x2_maxabs(v.a.z, v.a.w)),
                    bf16x2_maxabs(bf16x2_maxabs(v.b.x, v.b.y),
                                  bf16x2_maxabs(v.b.z, v.b.w)));
  return bf16x2_hmax(m & 0x7FFF7FFFu);
}

__device__ __forceinline__ uint32_t chunk_absmax(const uint4& v) {
  return bf16x2_hmax(bf16x2_maxabs(bf16x2_maxabs(v.x, v.y),
                                   bf16x2_maxabs(v.z, v.w)) &
                     0x7FFF7FFFu);
}

__device__ __forceinline__ uint32_t warp_max(uint32_t a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(FULL, a, o));
  return a;
}

// Maximum over each half of the warp (lanes 0-15 and 16-31 separately).
__device__ __forceinline__ uint32_t half_warp_max(uint32_t a) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(FULL, a, o));
  return a;
}

// pol != 0: the rows are read for the last time (the weight quantizer's
// second pass): their lines are marked first to evict in L2.
__device__ __forceinline__ void load_block(Blk& v, const uint16_t* row,
                                           int64_t b, bool valid, bool wide,
                                           uint64_t pol = 0) {
  if (valid && pol) {
    if (wide) {
      ld_last_v8(row + b * 16, v.a, v.b, pol);
    } else {
      v.a = ld_last_v4(row + b * 16, pol);
      v.b = ld_last_v4(row + b * 16 + 8, pol);
    }
  } else if (valid) {
    if (wide) {
      ld_stream_v8(row + b * 16, v.a, v.b);
    } else {
      v.a = ld_stream_v4(row + b * 16);
      v.b = ld_stream_v4(row + b * 16 + 8);
    }
  } else {
    v.a = make_uint4(0, 0, 0, 0);
    v.b = v.a;
  }
}

// Encode one 16-value block whose amax (bf16 bits) is `a` with FP32 scale
// S (six_s = fl(6 S)); returns the packed codes (lo: values 0-7, hi:
// values 8-15) and the E4M3 block-scale byte.
__device__ __forceinline__ void encode_block(const Blk& v, uint32_t a, float S,
                                             float six_s, uint32_t& lo,
                                             uint32_t& hi, uint32_t& sb) {
  sb = 0;
  if (S != 0.0f)
    sb = cvt_e4m3x2(__fdiv_rn(__uint_as_float(a << 16), six_s), 0.0f) & 0xFFu;
  const float d = __fmul_rn(e4m3_to_f32(sb), S);
  float enc = 0.0f;
  if (d != 0.0f) enc = fminf(__frcp_rn(d), FLT_MAX);
  float q[8];
  fmul2(bf16lo_to_f32(v.a.x), bf16hi_to_f32(v.a.x), enc, enc, q[0], q[1]);
  fmul2(bf16lo_to_f32(v.a.y), bf16hi_to_f32(v.a.y), enc, enc, q[2], q[3]);
  fmul2(bf16lo_to_f32(v.a.z), bf16hi_to_f32(v.a.z), enc, enc, q[4], q[5]);
  fmul2(bf16lo_to_f32(v.a.w), bf16hi_to_f32(v.a.w), enc, enc, q[6], q[7]);
  lo = cvt_e2m1x8(q);
  fmul2(bf16lo_to_f32(v.b.x), bf16hi_to_f32(v.b.x), enc, enc, q[0], q[1]);
  fmul2(bf16lo_to_f32(v.b.y), bf16hi_to_f32(v.b.y), enc, enc, q[2], q[3]);
  fmul2(bf16lo_to_f32(v.b.z), bf16hi_to_f32(v.b.z), enc, enc, q[4], q[5]);
  fmul2(bf16lo_to_f32(v.b.w), bf16hi_to_f32(v.b.w), enc, enc, q[6], q[7]);
  hi = cvt_e2m1x8(q);
}

// Store a lane's block: 8 bytes of codes, and (lanes 0, 4, 8, ...) the
// 32-bit word holding the scales of blocks b0..b0+3 gathered from the
// four consecutive lanes that own them.  `b` is the lane's block index;
// all 32 lanes of the warp must call this together.
__device__ __forceinline__ void store_block(const RowOut& o, int64_t b,
                                            bool write_codes, uint32_t lo,
                                            uint32_t hi, uint32_t sb, int lane) {
  if (write_codes && b < o.nblocks) st_v2(o.codes_row + b * 8, lo, hi);
  if (o.stage) {                          // uniform over the CTA
    if (b < 4 * o.col_tiles) o.stage[b] = (uint8_t)sb;
    return;
  }
  // lanes 4i .. 4i+3 hold four consecutive block scales: two shuffles
  // assemble them, lowest block in the lowest byte, in lane 4i
  const uint32_t pair = sb | (__shfl_down_sync(FULL, sb, 1) << 8);
  const uint32_t word = pair | (__shfl_down_sync(FULL, pair, 2) << 16);
  if ((lane & 3) == 0 && o.scales) {      // no scales: a row past the matrix
    if (o.swizzled) {
      if (b < ((o.nblocks + 3) & ~int64_t(3)))
        *reinterpret_cast<uint32_t*>(o.scales +
                                     swz_offset(o.row, b, o.col_tiles)) = word;
    } else if ((o.nblocks & 3) == 0) {
      if (b < o.nblocks)
        *reinterpret_cast<uint32_t*>(o.scales + o.row * o.nblocks + b) = word;
    } else {
      for (int j = 0; j < 4; ++j)
        if (b + j < o.nblocks)
          o.scales[o.row * o.nblocks + b + j] = (uint8_t)(word >> (8 * j));
    }
  }
}

// One row of H values is spread over WPR warps; warp w of the row owns
// blocks [w*R*32, (w+1)*R*32), lane l the blocks w*R*32 + r*32 + l.  The
// row's amax is combined across its warps through shared memory and a
// named barrier (id 1 + row slot, 32*WPR threads).  LPR = 16: each half of
// the warp takes its own row (WPR = 1), lane l of a half the blocks
// r*16 + l (rows of 33 to 48 blocks: 3 blocks a lane, no idle lanes).
template <int R, int WPR, int LPR = 32>
__device__ __forceinline__ void encode_row_warps(
    const uint16_t* row, bool load, bool write, float S_given, bool use_given,
    const RowOut& o, int row_slot, int wpart, int lane, uint32_t* red,
    float* S_used, uint64_t pol = 0) {
  static_assert(LPR == 32 || (LPR == 16 && WPR == 1), "lanes per row");
  const int l = lane & (LPR - 1);
  const int64_t blk0 = (int64_t)wpart * R * LPR;
  Blk v[R];
  uint32_t am[R];
  uint32_t a = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t b = blk0 + r * LPR + l;
    load_block(v[r], row, b, load && b < o.nblocks, o.wide, pol);
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    am[r] = block_absmax(v[r]);
    a = max(a, am[r]);
  }
  float S = S_given;
  if (!use_given) {
    a = LPR == 32 ? warp_max(a) : half_warp_max(a);
    if (WPR > 1) {
      if (lane == 0) red[row_slot * WPR + wpart] = a;
      named_barrier_sync(1 + row_slot, 32 * WPR);
      for (int w = 0; w < WPR; ++w) a = max(a, red[row_slot * WPR + w]);
    }
    S = __fdiv_rn(__uint_as_float(a << 16), kNvfp4ScaleDenom);
  }
  const float six_s = __fmul_rn(6.0f, S);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (blk0 + r * LPR >= o.nblocks) break;            // warp-uniform
    uint32_t lo, hi, sb;
    encode_block(v[r], am[r], S, six_s, lo, hi, sb);
    store_block(o, blk0 + r * LPR + l, write, lo, hi, sb, lane);
  }
  *S_used = S;
}

// ---------------------------------------------------------------------------
// Per-token activations.
// ---------------------------------------------------------------------------
// With swizzled scales and 4 or 8 rows per CTA, a CTA takes rows of one
// 128-row scale tile that share swizzled segments (rows k + 32q, or
// 2k + d + 32q for 8 rows), stages their block scales in shared memory and
// writes each column tile's segment with one 16- or 32-byte store instead
// of one 4-byte store per row.
template <int R, int WPR>
__global__ void __launch_bounds__(CTA_WARPS * 32)
    nvfp4_token_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t T_pad,
                       int64_t H, int64_t ldx,
                       const int32_t* __restrict__ row_index, int64_t T_src,
                       uint8_t* __restrict__ codes,
                       uint8_t* __restrict__ scales, float* __restrict__ S_out,
                       int swizzled, int wide, int sc_wide) {
  constexpr int ROWS = CTA_WARPS / WPR;
  constexpr bool kStageable = ROWS == 4 || ROWS == 8;
  __shared__ uint32_t red[CTA_WARPS];
  __shared__ __align__(16) uint8_t s_sc[kStageable ? ROWS : 1]
                                       [kStageable ? 1024 / ROWS : 4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = warp / WPR, wpart = warp % WPR;
  const bool staged = kStageable && swizzled;
  constexpr int64_t P = 128 / ROWS;               // CTAs per 128-row tile
  const int64_t rt = blockIdx.x / P, k = blockIdx.x % P;
  const int64_t t =
      !staged ? (int64_t)blockIdx.x * ROWS + slot
              : rt * 128 + (ROWS == 8 ? 2 * k + (slot & 1) + 32 * (slot >> 1)
                                      : k + 32 * slot);
  const int64_t col_tiles = ((H >> 4) + 3) >> 2;
  pdl_wait();
  if (t < T_pad) {                        // uniform over the row's warps
    const bool real = t < T;
    int64_t src = t;
    bool load = real;
    if (row_index && real) {              // gather: row t <- x[row_index[t]]
      src = row_index[t];
      load = src >= 0 && src < T_src;     // other indices: a zero row
    }
    RowOut o{codes + t * (H >> 1), scales, t, col_tiles, H >> 4,
             swizzled, wide, staged ? s_sc[slot] : nullptr};
    float S;
    encode_row_warps<R, WPR>(load ? x + src * ldx : x, load, real, 0.0f,
                             false, o, slot, wpart, lane, red, &S);
    if (real && wpart == 0 && lane == 0) S_out[t] = S;
  }
  if (staged) {
    // T_pad is a multiple of 128 here, so every row of the CTA exists.
    __syncthreads();
    uint8_t* tile0 = scales + rt * col_tiles * 512;
    for (int64_t ct = threadIdx.x; ct < col_tiles; ct += CTA_WARPS * 32) {
      const int64_t c4 = ct * 4;
      if (ROWS == 4) {
        const uint4 v = make_uint4(*reinterpret_cast<const uint32_t*>(&s_sc[0][c4]),
                                   *reinterpret_cast<const uint32_t*>(&s_sc[1 % ROWS][c4]),
                                   *reinterpret_cast<const uint32_t*>(&s_sc[2 % ROWS][c4]),
                                   *reinterpret_cast<const uint32_t*>(&s_sc[3 % ROWS][c4]));
        st_v4(tile0 + ct * 512 + k * 16, v);
      } else {
        const uint4 a = make_uint4(*reinterpret_cast<const uint32_t*>(&s_sc[0][c4]),
                                   *reinterpret_cast<const uint32_t*>(&s_sc[2 % ROWS][c4]),
                                   *reinterpret_cast<const uint32_t*>(&s_sc[4 % ROWS][c4]),
                                   *reinterpret_cast<const uint32_t*>(&s_sc[6 % ROWS][c4]));
        const uint4 b = make_uint4(*reinterpret_cast<const uint32_t*>(&s_sc[1 % ROWS][c4]),
                                   *reinterpret_cast<const uint32_t*>(&s_sc[3 % ROWS][c4]),
                                   *reinterpret_cast<const uint32_t*>(&s_sc[5 % ROWS][c4]),
                                   *reinterpret_cast<const uint32_t*>(&s_sc[7 % ROWS][c4]));
        st_32B(tile0 + ct * 512 + k * 32, a, b, sc_wide);
      }
    }
  }
  pdl_launch_dependents();
}

// Rows longer than 8 warps x 2048 values: one CTA per row, an amax pass and
// a second (cache-served) pass that encodes.
__global__ void __launch_bounds__(CTA_WARPS * 32)
    nvfp4_token_long_kernel(const uint16_t* __restrict__ x, int64_t T,
                            int64_t H, int64_t ldx,
                            const int32_t* __restrict__ row_index,
                            int64_t T_src, uint8_t* __restrict__ codes,
                            uint8_t* __restrict__ scales,
                            float* __restrict__ S_out, int swizzled,
                            int wide) {
  __shared__ uint32_t red[CTA_WARPS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = blockIdx.x;
  const bool real = t < T;
  int64_t src = t;
  bool load = real;
  if (row_index && real) {                // gather: row t <- x[row_index[t]]
    src = row_index[t];
    load = src >= 0 && src < T_src;
  }
  const uint16_t* row = load ? x + src * ldx : x;
  pdl_wait();
  RowOut o{codes + t * (H >> 1), scales, t, ((H >> 4) + 3) >> 2, H >> 4,
           swizzled, wide, nullptr};
  const int64_t span = CTA_WARPS * 32;
  uint32_t a = 0;
  for (int64_t b0 = 0; b0 < o.nblocks; b0 += span) {
    const int64_t b = b0 + threadIdx.x;
    Blk v;
    load_block(v, row, b, load && b < o.nblocks, o.wide);
    a = max(a, block_absmax(v));
  }
  a = warp_max(a);
  if (lane == 0) red[warp] = a;
  __syncthreads();
  for (int w = 0; w < CTA_WARPS; ++w) a = max(a, red[w]);
  const float S = __fdiv_rn(__uint_as_float(a << 16), kNvfp4ScaleDenom);
  const float six_s = __fmul_rn(6.0f, S);
  for (int64_t b0 = 0; b0 < o.nblocks; b0 += span) {
    if (b0 + warp * 32 >= o.nblocks) continue;         // warp-uniform
    const int64_t b = b0 + threadIdx.x;
    Blk v;
    load_block(v, row, b, load && b < o.nblocks, o.wide);
    uint32_t lo, hi, sb;
    encode_block(v, block_absmax(v), S, six_s, lo, hi, sb);
    store_block(o, b, real, lo, hi, sb, lane);
  }
  if (real && threadIdx.x == 0) S_out[t] = S;
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Weight groups: one persistent kernel working through a task list.  Per
// group g there are nA amax tasks (64 to 256 KiB of the group each) and
// nE encode tasks (2 or 4 sets of ROWS rows); an encode task needs its
// group's S, i.e. every amax task of the group.  Groups are taken in windows of about
// 12 MB of input, and the list runs A(0) .. A(L-1), then A(w+L) E(w) for
// w = 0, 1, ...: the amax tasks L windows ahead of the encode tasks, with
// L windows making about 36 MB (128 gate/up pairs: 12 MB x 3 or 6 MB x 6
// 224 us; 24 MB x 1 230 us, 6 MB x 5 249 us, 12 MB x 4 231 us: a shorter
// lead leaves encode tasks waiting for S, a longer one overflows L2).
// CTAs take tasks in list order from an atomic counter, so an encode task
// only ever waits (bounded) for amax tasks that running CTAs already hold,
// and by the time it is handed out L windows of amax and encode tasks
// separate it from its group's; the windows in flight stay in
// the 126 MB L2, so the encode tasks read their rows back from L2 however
// many groups a call holds (those reads mark the lines first to evict, so
// lines still waiting for their second read outlive the ones read twice).
//
// Workspace: [1 + launch] the task counter of each launch; [64 + g] the
// amax of group g (float bits, merged with atomicMax); [64 + G + g] the
// number of group g's amax tasks that have merged their maximum (a release
// add after the maximum).  Plain single-shot atomics: a compare-and-swap loop on
// one word per group serialises the hundreds of CTAs that finish together.
// ---------------------------------------------------------------------------
constexpr int kMaxGroupsPerLaunch = 256;
// An amax task covers a whole number of rounds of kRoundChunks (one 32-byte
// load pair per thread per round), about 1/kAmaxTasksPerGroup of its
// group, from 2 to 8 rounds (64 to 256 KiB): fewer, longer amax tasks mean
// fewer task claims and CTA barriers (128 gate/up pairs: 64 KiB tasks 255
// us, 128 KiB 240, 256 KiB 234, 512 KiB 310; down: 126, 121, 127, 163).
constexpr int64_t kRoundChunks = CTA_WARPS * 32 * 8;
constexpr int64_t kAmaxTasksPerGroup = 24;
constexpr int64_t kMinAmaxTasks = 1024;
// Encode task: RowSets(R, WPR) sets of ROWS rows (ROWS = 8 / WPR, or 16
// with half-warp rows).  Rows of at most 1024 values on full warps (R <= 2
// blocks per lane) take 4 sets, 32 rows (short rows would otherwise make
// small tasks whose fixed cost dominates); longer rows take 2, and so do
// half-warp rows (2 x 16 = 32 rows: the down projections); 4 sets measured
// slower at 2048 values, and with WPR = 2 the 8 rows of 2 sets fill whole
// swizzled scale sectors.
__host__ __device__ constexpr int RowSets(int r, int wpr) {
  return (wpr == 1 && r <= 2) ? 4 : 2;
}
constexpr int kWsHeaderWords = 64;            // [1 + launch] = task counters
constexpr int64_t kWindowBytes = 12ll << 20;  // input bytes per window
constexpr int64_t kLeadBytes = 36ll << 20;    // amax lead, L windows

// Error word of the bounded waits of this translation unit.
__device__ unsigned int g_nvfp4_wait_error = 0;

struct GroupTable {
  const uint16_t* part[kMaxGroupsPerLaunch][kMaxParts];
};

struct GroupParams {
  int num_parts;
  int64_t part_row0[kMaxParts + 1];   // prefix sums of the parts' rows
  int64_t part_chunk0[kMaxParts + 1]; // prefix sums of the parts' 16-byte chunks
  int64_t R, R_pad, K;
  int64_t g0;                         // global index of local group 0
  int ng;                             // groups in this launch
  int64_t nA, nE;                     // amax / encode tasks per group
  int64_t win;                        // groups per window (>= 1)
  int64_t lead;                       // windows of amax tasks ahead, L
  uint8_t* codes;                     // group g at g * R * K/2
  uint8_t* scales;                    // group g at g * scale_stride
  int64_t scale_stride;
  float* group_scales;
  const float* S_in;                  // NULL: S from amax
  uint32_t* ws;                       // [64 + g] amax words
  uint32_t* counter;                  // this launch's task counter
  uint32_t* done;                     // finished amax tasks per group
  int wide;                           // all parts 32-byte aligned
  int sc_wide;                        // scale matrices 32-byte aligned
  int swizzled;
};

__device__ __forceinline__ const uint16_t* chunk_ptr(const GroupTable& tab,
                                                     const GroupParams& p,
                                                     int gl, int64_t q) {
  int pi = 0;
  while (pi + 1 < p.num_parts && q >= p.part_chunk0[pi + 1]) ++pi;
  return tab.part[gl][pi] + (q - p.part_chunk0[pi]) * 8;
}

// Task t of the list -> (is_amax, local group, index within the group).
// With S given there are only encode tasks, group-major.  Otherwise the
// list is A(0) .. A(L-1), then for w = 0, 1, ...: A(w+L) (if window w+L
// exists) and E(w); A(w) holds nA tasks per group of window w, E(w) nE per
// group, and every window but the last holds `win` groups.  The amax tasks
// of a group thus run L windows of amax work and L - 1 windows of encode
// work before its encode tasks, which is the time its slowest amax task
// has to become visible, while the L2 holds about L + 1 windows of input.
__device__ __forceinline__ void task_of(const GroupParams& p, int64_t t,
                                        bool* is_a, int* gl, int64_t* idx) {
  if (p.S_in) {
    *is_a = false;
    *gl = (int)(t / p.nE);
    *idx = t - (int64_t)*gl * p.nE;
    return;
  }
  // Closed form (no loop over windows: the decode is on every task's
  // path).  Every window but the last is full (W groups): a = W nA amax
  // and e = W nE encode tasks; the last has `last` groups.
  const int64_t W = p.win;
  const int64_t nw = (p.ng + W - 1) / W;
  const int64_t last = p.ng - (nw - 1) * W;
  const int64_t L = p.lead < nw ? p.lead : nw;
  const int64_t a = W * p.nA, e = W * p.nE;
  const int64_t a_last = last * p.nA, e_last = last * p.nE;
  auto amax_task = [&](int64_t w, int64_t r) {
    *is_a = true;
    *gl = (int)(w * W + r / p.nA);
    *idx = r % p.nA;
  };
  auto enc_task = [&](int64_t w, int64_t r) {
    *is_a = false;
    *gl = (int)(w * W + r / p.nE);
    *idx = r % p.nE;
  };
  // 1. A(0) .. A(L-1)
  if (L < nw) {
    if (t < L * a) return amax_task(t / a, t % a);
    t -= L * a;
  } else {
    if (t < (nw - 1) * a) return amax_task(t / a, t % a);
    t -= (nw - 1) * a;
    if (t < a_last) return amax_task(nw - 1, t);
    t -= a_last;
  }
  int64_t w_tail = 0;                              // first window of step 3
  if (L < nw) {
    // 2. pairs A(w+L) E(w), w = 0 .. nw-L-1; the last pair's A is the
    //    last window
    const int64_t full_pairs = nw - L - 1;
    if (t < full_pairs * (a + e)) {
      const int64_t w = t / (a + e), r = t % (a + e);
      if (r < a) return amax_task(w + L, r);
      return enc_task(w, r - a);
    }
    t -= full_pairs * (a + e);
    if (t < a_last) return amax_task(nw - 1, t);
    t -= a_last;
    if (t < e) return enc_task(nw - L - 1, t);
    t -= e;
    w_tail = nw - L;
  }
  // 3. E(w) for the remaining windows, the last one possibly partial
  const int64_t full_tail = (nw - 1) - w_tail;     // full windows before the last
  if (t < full_tail * e) return enc_task(w_tail + t / e, t % e);
  t -= full_tail * e;
  if (t < e_last) return enc_task(nw - 1, t);
  *is_a = false;                                   // past the list's end
  *gl = 0;
  *idx = 0;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v)
               : "memory");
}

// Half-warp rows (the down projections) run 5 CTAs per SM at 48 registers
// (137 -> 126 us at 128 experts); the full-warp shapes 4 at 56 (5 measured
// slower: gate/up 255 -> 292 us; the 64 registers of 4 CTAs per SM spilled
// 16-24 bytes in the encode loop, 56 spill none at 2048 values a row: 128
// gate/up pairs 234.7 -> 229.6 us).
template <int R, int WPR, int LPR, int NR>
__global__ void __maxnreg__(LPR == 16 ? 48 : 56)
    nvfp4_weight_kernel(const __grid_constant__ GroupTable tab,
                        const __grid_constant__ GroupParams p) {
  constexpr int ROWS = CTA_WARPS / WPR * (32 / LPR);  // rows per row set
  constexpr int64_t kTaskChunks = NR * kRoundChunks;  // per amax task
  __shared__ uint32_t red[CTA_WARPS];
  __shared__ int s_abort;
  __shared__ int64_t s_task[2];
  // Encode tasks of 8 rows with swizzled scales: the rows 2k + d + 32q of
  // one 128-row tile, whose block scales fill whole 32-byte sectors of the
  // swizzled tiles; staged here, written as one 32-byte store per tile.
  constexpr int kRowSetsPerTask = RowSets(R, WPR);
  constexpr bool kStage8 = ROWS * kRowSetsPerTask == 8;
  __shared__ __align__(16) uint8_t s_sc[kStage8 ? 8 : 1][kStage8 ? 256 : 4];
  __shared__ float s_S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // LPR = 16: the two halves of a warp take rows 2 warp and 2 warp + 1
  const int slot = LPR == 32 ? warp / WPR : 2 * warp + (lane >> 4);
  const int wpart = LPR == 32 ? warp % WPR : 0;
  if (threadIdx.x == 0) s_abort = 0;
  __syncthreads();
  pdl_wait();
  const int64_t group_chunks = p.part_chunk0[p.num_parts];
  uint32_t* amax = p.ws + kWsHeaderWords;      // unused when S_in is given
  const int64_t total = (int64_t)p.ng * (p.S_in ? p.nE : p.nA + p.nE);
  int64_t t_static = blockIdx.x;
  // The next task's index is fetched while the current task runs (slot
  // buf ^ 1); the barrier that ends every task publishes it.
  if (!p.S_in && threadIdx.x == 0) s_task[0] = (int64_t)atomicAdd(p.counter, 1u);
  __syncthreads();
  int buf = 0;
  const uint64_t pol_last = l2_policy_evict_first();
  while (true) {
    int64_t t;
    if (p.S_in) {
      t = t_static;                   // no amax: a static round robin
      t_static += gridDim.x;
    } else {
      t = s_task[buf];
      if (t < total && threadIdx.x == 0)
        s_task[buf ^ 1] = (int64_t)atomicAdd(p.counter, 1u);
      buf ^= 1;
    }
    if (t >= total) break;
    bool is_a;
    int gl;
    int64_t idx;
    task_of(p, t, &is_a, &gl, &idx);
    if (is_a) {
      // ---- amax of one task (2, 4 or 8 rounds, 64 to 256 KiB) of group gl ----
      uint32_t a = 0;
      const int64_t q0 = idx * kTaskChunks;
      // The task's chunks usually lie in one part: then one base pointer
      // and 32-byte loads (pairs of chunks); otherwise a part lookup per
      // 16-byte chunk.
      int pi = 0;
      while (pi + 1 < p.num_parts && q0 >= p.part_chunk0[pi + 1]) ++pi;
      const bool one_part = p.wide && q0 + kTaskChunks <= p.part_chunk0[pi + 1];
      if (one_part && !s_abort) {
        const uint16_t* base = tab.part[gl][pi] + (q0 - p.part_chunk0[pi]) * 8;
        // NR rounds of 32-byte loads, a round's loads issued before its
        // reduction.  NR is a template parameter and the loop is written
        // here rather than in a helper: either change alone measured 181
        // instead of 174 us for the encode tasks at 128 gate/up pairs with
        // the scales given (a different register allocation of the loop).
#pragma unroll
        for (int rr = 0; rr < NR; ++rr) {
          uint4 v[8];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
            ld_stream_v8(base + ((int64_t)(rr * 4 + jj) * (CTA_WARPS * 32) +
                                 threadIdx.x) * 16,
                         v[2 * jj], v[2 * jj + 1]);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) a = max(a, chunk_absmax(v[jj]));
        }
      } else {
#pragma unroll
        for (int rr = 0; rr < NR; ++rr) {
          uint4 v[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int64_t q = q0 + (int64_t)(rr * 8 + jj) * (CTA_WARPS * 32) +
                              threadIdx.x;
            v[jj] = (q < group_chunks && !s_abort)
                        ? ld_stream_v4(chunk_ptr(tab, p, gl, q))
                        : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) a = max(a, chunk_absmax(v[jj]));
        }
      }
      const uint32_t m = warp_max(a);
      if (lane == 0) red[warp] = m;
      __syncthreads();
      if (threadIdx.x == 0) {
        uint32_t mm = red[0];
        for (int w = 1; w < CTA_WARPS; ++w) mm = max(mm, red[w]);
        if (mm) atomicMax(&amax[p.g0 + gl], mm << 16);
        red_release_add(&p.done[p.g0 + gl], 1u);   // after the maximum
      }
      __syncthreads();
      continue;
    }
    // ---- encode ROWS rows of group gl ----
    const int64_t g = p.g0 + gl;
    if (threadIdx.x == 0) {
      float S = 0.0f;
      if (p.S_in) {
        S = p.S_in[g];
      } else {
        // wait until every amax task of the group has merged its maximum
        // Poll with relaxed loads and a back-off (acquire loads in a tight
        // loop slow down the streaming loads of the other CTAs on the SM),
        // then one acquire fence.
        const uint64_t t0 = global_timer_ns();
        while (true) {
          const uint32_t nd = *reinterpret_cast<volatile uint32_t*>(&p.done[g]);
          if ((int64_t)nd >= p.nA || s_abort) break;
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_nvfp4_wait_error, 1u);
            s_abort = 1;
            break;
          }
          __nanosleep(256);
        }
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        S = __fdiv_rn(
            __uint_as_float(*reinterpret_cast<volatile uint32_t*>(&amax[g])),
            kNvfp4ScaleDenom);
      }
      s_S = S;
    }
    __syncthreads();
    const float S = s_S;
    const bool staged = kStage8 && p.swizzled && (p.K >> 4) <= 256;
    for (int rs = 0; rs < kRowSetsPerTask; ++rs) {
    const int s8 = rs * ROWS + slot;
    const int64_t r = staged ? (idx >> 4) * 128 + 2 * (idx & 15) + (s8 & 1) +
                                   32 * (s8 >> 1)
                             : (idx * kRowSetsPerTask + rs) * ROWS + slot;
    // uniform over the row; with half-warp rows the two halves may
    // differ, so a warp with one row in range runs the other half idle
    // (no loads, no stores)
    const bool active = r < p.R_pad && !s_abort;
    if (LPR == 32 ? active : __any_sync(FULL, active)) {
      const bool real = active && r < p.R;
      const uint16_t* row = nullptr;
      if (real) {
        int pi = 0;
        while (pi + 1 < p.num_parts && r >= p.part_row0[pi + 1]) ++pi;
        row = tab.part[gl][pi] + (r - p.part_row0[pi]) * p.K;
      }
      if (active && r == 0 && wpart == 0 && (lane & (LPR - 1)) == 0)
        p.group_scales[g] = S;
      RowOut o{p.codes + (g * p.R + r) * (p.K >> 1),
               active ? p.scales + g * p.scale_stride : nullptr, r,
               ((p.K >> 4) + 3) >> 2, p.K >> 4, p.swizzled, p.wide,
               staged ? s_sc[s8 % (kStage8 ? 8 : 1)] : nullptr};
      float S_used;
      encode_row_warps<R, WPR, LPR>(row, real, real, S, true, o, slot, wpart,
                                    lane, red, &S_used,
                                    p.S_in ? 0 : pol_last);
    }
    }
    if (staged) {
      __syncthreads();
      // R_pad is a multiple of 128 here: all 8 rows exist
      const int64_t col_tiles = ((p.K >> 4) + 3) >> 2;
      uint8_t* tile0 = p.scales + g * p.scale_stride +
                       (idx >> 4) * col_tiles * 512 + (idx & 15) * 32;
      for (int64_t ct = threadIdx.x; ct < col_tiles; ct += CTA_WARPS * 32) {
        const int64_t c4 = ct * 4;
        const uint4 a = make_uint4(
            *reinterpret_cast<const uint32_t*>(&s_sc[0][c4]),
            *reinterpret_cast<const uint32_t*>(&s_sc[2 % (kStage8 ? 8 : 1)][c4]),
            *reinterpret_cast<const uint32_t*>(&s_sc[4 % (kStage8 ? 8 : 1)][c4]),
            *reinterpret_cast<const uint32_t*>(&s_sc[6 % (kStage8 ? 8 : 1)][c4]));
        const uint4 b = make_uint4(
            *reinterpret_cast<const uint32_t*>(&s_sc[1 % (kStage8 ? 8 : 1)][c4]),
            *reinterpret_cast<const uint32_t*>(&s_sc[3 % (kStage8 ? 8 : 1)][c4]),
            *reinterpret_cast<const uint32_t*>(&s_sc[5 % (kStage8 ? 8 : 1)][c4]),
            *reinterpret_cast<const uint32_t*>(&s_sc[7 % (kStage8 ? 8 : 1)][c4]));
        st_32B(tile0 + ct * 512, a, b, p.sc_wide);
      }
    }
    __syncthreads();                  // s_S and red are reused by the next task
  }
  pdl_launch_dependents();
}

// Launch shape of the row encoders: R blocks per lane (R * 512 values per
// warp) and WPR warps per row; 0 = rows too long (one CTA per row).
struct RowShape {
  int R, WPR;
  int LPR = 32;           // lanes per row (16: two rows per warp)
};
RowShape pick_shape(int64_t H) {
  const int64_t nb = H >> 4;
  if (nb <= 32) return {1, 1};
  if (nb <= 64) return {2, 1};
  if (nb <= 128) return {4, 1};
  if (nb <= 256) return {4, 2};
  if (nb <= 512) return {4, 4};
  if (nb <= 1024) return {4, 8};
  return {0, 0};
}
// The weight quantizer's encode: rows of 33 to 48 blocks take half a warp
// each, 3 blocks a lane (with a full warp and 2 blocks a lane a quarter of
// the lanes idled in the second pass: 128 down projections [2048 x 768]).
RowShape pick_weight_shape(int64_t K) {
  const int64_t nb = K >> 4;
  if (nb > 32 && nb <= 48) return {3, 1, 16};
  return pick_shape(K);
}

}  // namespace

cudaError_t launch_nvfp4_per_token(const void* x, int64_t T, int64_t H,
                                   int64_t ldx, const int32_t* row_index,
                                   int64_t T_src, uint8_t* codes,
                                   uint8_t* scales, float* token_scales,
                                   int swizzled, cudaStream_t stream) {
  const int64_t T_pad = swizzled ? (T + 127) / 128 * 128 : T;
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  // every block starts a multiple of 32 bytes from x when ldx % 16 == 0
  const int wide = (reinterpret_cast<uintptr_t>(x) & 31u) == 0 && ldx % 16 == 0;
  const int sc_wide = (reinterpret_cast<uintptr_t>(scales) & 31u) == 0;
  const RowShape sh = pick_shape(H);
  if (sh.R == 0) {
    return launch_pdl(nvfp4_token_long_kernel, dim3((unsigned)T_pad),
                      dim3(CTA_WARPS * 32), 0, stream, false, xs, T, H, ldx,
                      row_index, T_src, codes, scales, token_scales, swizzled,
                      wide);
  }
  const int rows_per_cta = CTA_WARPS / sh.WPR;
  const unsigned grid = (unsigned)((T_pad + rows_per_cta - 1) / rows_per_cta);
#define MXQ_TOKEN_LAUNCH(R_, W_)                                          \
  launch_pdl(nvfp4_token_kernel<R_, W_>, dim3(grid), dim3(CTA_WARPS * 32), \
             0, stream, false, xs, T, T_pad, H, ldx, row_index, T_src,     \
             codes, scales, token_scales, swizzled, wide, sc_wide)
  if (sh.R == 1) return MXQ_TOKEN_LAUNCH(1, 1);
  if (sh.R == 2) return MXQ_TOKEN_LAUNCH(2, 1);
  if (sh.WPR == 1) return MXQ_TOKEN_LAUNCH(4, 1);
  if (sh.WPR == 2) return MXQ_TOKEN_LAUNCH(4, 2);
  if (sh.WPR == 4) return MXQ_TOKEN_LAUNCH(4, 4);
  return MXQ_TOKEN_LAUNCH(4, 8);
#undef MXQ_TOKEN_LAUNCH
}

size_t nvfp4_weight_ws_bytes(int64_t num_groups) {
  return (size_t)(((kWsHeaderWords + 2 * num_groups) * 4 + 255) / 256 * 256);
}

cudaError_t nvfp4_take_wait_error(unsigned int* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_nvfp4_wait_error, sizeof(*word));
  if (e != cudaSuccess || *word == 0) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_nvfp4_wait_error, &zero, sizeof(zero));
}

namespace {

template <int R, int WPR, int LPR, int NR>
cudaError_t launch_weight_nr(const GroupTable& tab, const GroupParams& p,
                             int dev, cudaStream_t stream) {
  static int occ[64] = {};
  int n = (dev >= 0 && dev < 64) ? occ[dev] : 0;
  if (n == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &n, nvfp4_weight_kernel<R, WPR, LPR, NR>, CTA_WARPS * 32, 0);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) occ[dev] = n;
  }
  const unsigned grid = (unsigned)(n * sm_count(dev));
  // No co-residency is needed: a CTA only waits for tasks that running
  // CTAs hold.
  return launch_pdl(nvfp4_weight_kernel<R, WPR, LPR, NR>, dim3(grid),
                    dim3(CTA_WARPS * 32), 0, stream, false, tab, p);
}

// rounds: 2, 4 or 8 rounds of kRoundChunks per amax task
template <int R, int WPR, int LPR = 32>
cudaError_t launch_weight_tasks(const GroupTable& tab, const GroupParams& p,
                                int rounds, int dev, cudaStream_t stream) {
  if (rounds == 8) return launch_weight_nr<R, WPR, LPR, 8>(tab, p, dev, stream);
  if (rounds == 4) return launch_weight_nr<R, WPR, LPR, 4>(tab, p, dev, stream);
  return launch_weight_nr<R, WPR, LPR, 2>(tab, p, dev, stream);
}

}  // namespace

cudaError_t launch_nvfp4_weight_shared(
    int64_t num_groups, int num_parts, const void* const* parts,
    const int64_t* part_rows, int64_t K, uint8_t* codes, uint8_t* scales,
    float* group_scales, const float* group_scales_in, int swizzled,
    uint32_t* ws, cudaStream_t stream) {
  const RowShape sh = pick_weight_shape(K);
  if (sh.R == 0) return cudaErrorInvalidValue;   // K > 16384: not supported
  GroupParams p;
  p.num_parts = num_parts;
  p.part_row0[0] = 0;
  p.part_chunk0[0] = 0;
  for (int i = 0; i < num_parts; ++i) {
    p.part_row0[i + 1] = p.part_row0[i] + part_rows[i];
    p.part_chunk0[i + 1] = p.part_chunk0[i] + part_rows[i] * K / 8;
  }
  for (int i = num_parts + 1; i <= kMaxParts; ++i) {
    p.part_row0[i] = p.part_row0[num_parts];
    p.part_chunk0[i] = p.part_chunk0[num_parts];
  }
  p.R = p.part_row0[num_parts];
  p.R_pad = swizzled ? (p.R + 127) / 128 * 128 : p.R;
  p.K = K;
  int64_t rounds;
  {
    // 2, 4 or 8 rounds: about kAmaxTasksPerGroup tasks per group, but at
    // least kMinAmaxTasks in the call (a small call needs many tasks to
    // fill the GPU)
    const int64_t gc = p.part_chunk0[num_parts];
    rounds = 8;
    while (rounds > 2 && (gc / (rounds * kRoundChunks) < kAmaxTasksPerGroup ||
                          num_groups * ((gc + rounds * kRoundChunks - 1) /
                                        (rounds * kRoundChunks)) <
                              kMinAmaxTasks))
      rounds /= 2;
    p.nA = (gc + rounds * kRoundChunks - 1) / (rounds * kRoundChunks);
  }
  const int64_t rows_per_task =
      RowSets(sh.R, sh.WPR) * (CTA_WARPS / sh.WPR) * (32 / sh.LPR);
  p.nE = (p.R_pad + rows_per_task - 1) / rows_per_task;
  p.win = kWindowBytes / (p.R * K * 2);
  if (p.win < 1) p.win = 1;
  // a call whose whole input stays in L2 runs as one window (8 gate/up
  // pairs of [1024 x 2048], 64 MB: 44.6 -> 40.8 us)
  if (num_groups * p.R * K * 2 <= (64ll << 20)) p.win = num_groups;
  p.lead = kLeadBytes / (p.win * p.R * K * 2);
  if (p.lead < 1) p.lead = 1;
  p.done = ws ? ws + kWsHeaderWords + num_groups : nullptr;
  p.codes = codes;
  p.scales = scales;
  p.scale_stride = scale_bytes(p.R, K / 16, swizzled);
  p.group_scales = group_scales;
  p.S_in = group_scales_in;
  p.ws = ws;
  p.swizzled = swizzled;
  p.sc_wide = (reinterpret_cast<uintptr_t>(scales) & 31u) == 0 &&
              p.scale_stride % 32 == 0;
  p.wide = 1;
  for (int64_t i = 0; i < num_groups * num_parts; ++i)
    if (reinterpret_cast<uintptr_t>(parts[i]) & 31u) p.wide = 0;

  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int64_t n_launch =
      (num_groups + kMaxGroupsPerLaunch - 1) / kMaxGroupsPerLaunch;
  if (!group_scales_in) {
    if (n_launch > kWsHeaderWords - 1) return cudaErrorInvalidValue;
    // Zero the task counters and every group's amax and count words.
    err = cudaMemsetAsync(ws, 0, (kWsHeaderWords + 2 * num_groups) * 4, stream);
    if (err != cudaSuccess) return err;
  }
  GroupTable tab;
  for (int64_t g0 = 0; g0 < num_groups; g0 += kMaxGroupsPerLaunch) {
    const int ng = (int)((num_groups - g0) < kMaxGroupsPerLaunch
                             ? (num_groups - g0)
                             : kMaxGroupsPerLaunch);
    for (int gl = 0; gl < kMaxGroupsPerLaunch; ++gl)
      for (int pi = 0; pi < kMaxParts; ++pi)
        tab.part[gl][pi] =
            (gl < ng && pi < num_parts)
                ? static_cast<const uint16_t*>(parts[(g0 + gl) * num_parts + pi])
                : nullptr;
    p.g0 = g0;
    p.ng = ng;
    p.counter = ws ? ws + 1 + g0 / kMaxGroupsPerLaunch : nullptr;
    if (sh.LPR == 16) err = launch_weight_tasks<3, 1, 16>(tab, p, (int)rounds, dev, stream);
    else if (sh.R == 1) err = launch_weight_tasks<1, 1>(tab, p, (int)rounds, dev, stream);
    else if (sh.R == 2) err = launch_weight_tasks<2, 1>(tab, p, (int)rounds, dev, stream);
    else if (sh.WPR == 1) err = launch_weight_tasks<4, 1>(tab, p, (int)rounds, dev, stream);
    else if (sh.WPR == 2) err = launch_weight_tasks<4, 2>(tab, p, (int)rounds, dev, stream);
    else if (sh.WPR == 4) err = launch_weight_tasks<4, 4>(tab, p, (int)rounds, dev, stream);
    else err = launch_weight_tasks<4, 8>(tab, p, (int)rounds, dev, stream);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace mxq
