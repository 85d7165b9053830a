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
// Design (sm_103a): HBM-streaming, one warp per row.  A lane loads 16-byte
// chunks (8 bf16) with coalesced non-allocating loads, all chunks of the
// row in flight at once (H = 2048: 8 loads of 16 B per lane); the row
// amax is a 5-step xor-shuffle reduction and a 16-block's amax one more
// shuffle between the two lanes that hold it.  Each lane emits one 32-bit
// word of packed codes per chunk (the warp writes 128 contiguous bytes per
// step); four block scales are gathered by shuffles into one 32-bit store
// (four consecutive scale columns are contiguous in both layouts).
// Weight groups use one persistent cooperative kernel (see below): an amax
// phase and an encode phase per L2-sized chunk of groups, separated by a
// bounded grid barrier, so the second read of a chunk is served from L2.
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

__device__ __forceinline__ void load_block(Blk& v, const uint16_t* row,
                                           int64_t b, bool valid) {
  if (valid) {
    v.a = ld_stream_v4(row + b * 16);
    v.b = ld_stream_v4(row + b * 16 + 8);
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
  const uint32_t s1 = __shfl_down_sync(FULL, sb, 1);
  const uint32_t s2 = __shfl_down_sync(FULL, sb, 2);
  const uint32_t s3 = __shfl_down_sync(FULL, sb, 3);
  if ((lane & 3) == 0) {
    const uint32_t word = sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
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
// named barrier (id 1 + row slot, 32*WPR threads).
template <int R, int WPR>
__device__ __forceinline__ void encode_row_warps(
    const uint16_t* row, bool real, float S_given, bool use_given,
    const RowOut& o, int row_slot, int wpart, int lane, uint32_t* red,
    float* S_used) {
  const int64_t blk0 = (int64_t)wpart * R * 32;
  Blk v[R];
  uint32_t am[R];
  uint32_t a = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t b = blk0 + r * 32 + lane;
    load_block(v[r], row, b, real && b < o.nblocks);
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    am[r] = block_absmax(v[r]);
    a = max(a, am[r]);
  }
  float S = S_given;
  if (!use_given) {
    a = warp_max(a);
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
    if (blk0 + r * 32 >= o.nblocks) break;             // warp-uniform
    uint32_t lo, hi, sb;
    encode_block(v[r], am[r], S, six_s, lo, hi, sb);
    store_block(o, blk0 + r * 32 + lane, real, lo, hi, sb, lane);
  }
  *S_used = S;
}

// ---------------------------------------------------------------------------
// Per-token activations.
// ---------------------------------------------------------------------------
template <int R, int WPR>
__global__ void __launch_bounds__(CTA_WARPS * 32)
    nvfp4_token_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t T_pad,
                       int64_t H, int64_t ldx, uint8_t* __restrict__ codes,
                       uint8_t* __restrict__ scales, float* __restrict__ S_out,
                       int swizzled) {
  constexpr int ROWS = CTA_WARPS / WPR;
  __shared__ uint32_t red[CTA_WARPS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = warp / WPR, wpart = warp % WPR;
  const int64_t t = (int64_t)blockIdx.x * ROWS + slot;
  pdl_wait();
  if (t >= T_pad) return;                 // uniform over the row's warps
  const bool real = t < T;
  RowOut o{codes + t * (H >> 1), scales, t, ((H >> 4) + 3) >> 2, H >> 4,
           swizzled};
  float S;
  encode_row_warps<R, WPR>(x + t * ldx, real, 0.0f, false, o, slot, wpart,
                           lane, red, &S);
  if (real && wpart == 0 && lane == 0) S_out[t] = S;
  pdl_launch_dependents();
}

// Rows longer than 8 warps x 2048 values: one CTA per row, an amax pass and
// a second (cache-served) pass that encodes.
__global__ void __launch_bounds__(CTA_WARPS * 32)
    nvfp4_token_long_kernel(const uint16_t* __restrict__ x, int64_t T,
                            int64_t H, int64_t ldx,
                            uint8_t* __restrict__ codes,
                            uint8_t* __restrict__ scales,
                            float* __restrict__ S_out, int swizzled) {
  __shared__ uint32_t red[CTA_WARPS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = blockIdx.x;
  const bool real = t < T;
  const uint16_t* row = x + t * ldx;
  pdl_wait();
  RowOut o{codes + t * (H >> 1), scales, t, ((H >> 4) + 3) >> 2, H >> 4,
           swizzled};
  const int64_t span = CTA_WARPS * 32;
  uint32_t a = 0;
  for (int64_t b0 = 0; b0 < o.nblocks; b0 += span) {
    const int64_t b = b0 + threadIdx.x;
    Blk v;
    load_block(v, row, b, real && b < o.nblocks);
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
    load_block(v, row, b, real && b < o.nblocks);
    uint32_t lo, hi, sb;
    encode_block(v, block_absmax(v), S, six_s, lo, hi, sb);
    store_block(o, b, real, lo, hi, sb, lane);
  }
  if (real && threadIdx.x == 0) S_out[t] = S;
  pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// Weight groups: one persistent cooperative kernel.  For each chunk of
// groups small enough to stay in L2: phase A reduces every group's amax
// (64 KiB work units, CTA partial maxima combined with an integer atomicMax
// on the float bits, exact for non-negative values); a grid-wide barrier;
// phase B encodes the chunk's rows with their group's S, re-reading the
// chunk from L2.  A CTA that finishes phase B of one chunk goes straight to
// phase A of the next.
// ---------------------------------------------------------------------------
constexpr int kMaxGroupsPerLaunch = 256;
constexpr int64_t kAmaxUnitChunks = 1024;     // 16-byte chunks per unit (16 KiB)
constexpr int kWsHeaderWords = 64;            // [0] = barrier counter

// Error word of the bounded grid barrier of this translation unit.
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
  int chunk;                          // groups per L2-sized chunk
  int64_t units_per_group;            // phase-A units per group
  uint8_t* codes;                     // group g at g * R * K/2
  uint8_t* scales;                    // group g at g * scale_stride
  int64_t scale_stride;
  float* group_scales;
  const float* S_in;                  // NULL: S from amax
  uint32_t* ws;                       // [0] barrier, [64 + g] amax of group g
  int swizzled;
};

// Grid-wide barrier for a cooperative launch: every CTA adds 1 to *ctr and
// waits (bounded, ~1 s) until it reaches `target`.  On timeout it records 1
// in g_nvfp4_wait_error, sets *abort and returns false; all threads of the
// CTA still pass the same __syncthreads calls.
__device__ __forceinline__ bool grid_barrier(uint32_t* ctr, uint32_t target,
                                             volatile int* abort) {
  __syncthreads();
  if (threadIdx.x == 0 && !*abort) {
    __threadfence();
    atomicAdd(ctr, 1u);
    const uint64_t t0 = global_timer_ns();
    while (true) {
      uint32_t v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];"
                   : "=r"(v)
                   : "l"(ctr)
                   : "memory");
      if (v >= target) break;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicOr(&g_nvfp4_wait_error, 1u);
        *abort = 1;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
  return !*abort;
}

__device__ __forceinline__ const uint16_t* chunk_ptr(const GroupTable& tab,
                                                     const GroupParams& p,
                                                     int gl, int64_t q) {
  int pi = 0;
  while (pi + 1 < p.num_parts && q >= p.part_chunk0[pi + 1]) ++pi;
  return tab.part[gl][pi] + (q - p.part_chunk0[pi]) * 8;
}

template <int R, int WPR>
__global__ void __launch_bounds__(CTA_WARPS * 32, 4)
    nvfp4_weight_kernel(const __grid_constant__ GroupTable tab,
                        const __grid_constant__ GroupParams p) {
  constexpr int ROWS = CTA_WARPS / WPR;
  __shared__ uint32_t red[CTA_WARPS];
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = warp / WPR, wpart = warp % WPR;
  if (threadIdx.x == 0) s_abort = 0;
  __syncthreads();
  pdl_wait();
  const int64_t group_chunks = p.part_chunk0[p.num_parts];
  uint32_t* amax = p.ws + kWsHeaderWords;
  uint32_t gen = 0;
  for (int c0 = 0; c0 < p.ng; c0 += p.chunk) {
    const int nc = (p.ng - c0) < p.chunk ? (p.ng - c0) : p.chunk;
    if (!p.S_in) {
      // Phase A: amax of every group of the chunk.  Each CTA takes a
      // contiguous range of 16 KiB units (so it spans at most a few groups),
      // keeps a running max in registers and combines it across the CTA
      // only when the group changes and at the end of its range.
      const int64_t n_units = (int64_t)nc * p.units_per_group;
      const int64_t u_begin = n_units * blockIdx.x / gridDim.x;
      const int64_t u_end = n_units * (blockIdx.x + 1) / gridDim.x;
      int cur = -1;
      uint32_t a = 0;
      for (int64_t u = u_begin; u < u_end; ++u) {
        const int gl = c0 + (int)(u / p.units_per_group);
        const int64_t q0 = (u % p.units_per_group) * kAmaxUnitChunks;
        uint4 v[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int64_t q = q0 + threadIdx.x + (int64_t)jj * 256;
          v[jj] = q < group_chunks ? ld_stream_v4(chunk_ptr(tab, p, gl, q))
                                   : make_uint4(0, 0, 0, 0);
        }
        if (gl != cur) {                                   // CTA-uniform
          if (cur >= 0) {
            const uint32_t m = warp_max(a);
            if (lane == 0) red[warp] = m;
            __syncthreads();
            if (threadIdx.x == 0) {
              uint32_t mm = red[0];
              for (int w = 1; w < CTA_WARPS; ++w) mm = max(mm, red[w]);
              if (mm) atomicMax(&amax[p.g0 + cur], mm << 16);
            }
            __syncthreads();
          }
          cur = gl;
          a = 0;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) a = max(a, chunk_absmax(v[jj]));
      }
      if (cur >= 0) {                                      // CTA-uniform
        const uint32_t m = warp_max(a);
        if (lane == 0) red[warp] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
          uint32_t mm = red[0];
          for (int w = 1; w < CTA_WARPS; ++w) mm = max(mm, red[w]);
          if (mm) atomicMax(&amax[p.g0 + cur], mm << 16);
        }
        __syncthreads();
      }
      ++gen;
      grid_barrier(p.ws, gen * gridDim.x, &s_abort);
    }
    // Phase B: encode the chunk's rows (and the scale-tile padding rows).
    const int64_t nrows = (int64_t)nc * p.R_pad;
    for (int64_t base = (int64_t)blockIdx.x * ROWS; base < nrows;
         base += (int64_t)gridDim.x * ROWS) {
      const int64_t w = base + slot;
      if (w >= nrows || s_abort) continue;             // uniform over the row
      const int gl = c0 + (int)(w / p.R_pad);
      const int64_t r = w - (int64_t)(gl - c0) * p.R_pad;
      const int64_t g = p.g0 + gl;
      const bool real = r < p.R;
      const uint16_t* row = nullptr;
      if (real) {
        int pi = 0;
        while (pi + 1 < p.num_parts && r >= p.part_row0[pi + 1]) ++pi;
        row = tab.part[gl][pi] + (r - p.part_row0[pi]) * p.K;
      }
      const float S = p.S_in ? p.S_in[g]
                             : __fdiv_rn(__uint_as_float(__ldcg(&amax[g])),
                                         kNvfp4ScaleDenom);
      if (r == 0 && wpart == 0 && lane == 0) p.group_scales[g] = S;
      RowOut o{p.codes + (g * p.R + r) * (p.K >> 1),
               p.scales + g * p.scale_stride, r, ((p.K >> 4) + 3) >> 2,
               p.K >> 4, p.swizzled};
      float S_used;
      encode_row_warps<R, WPR>(row, real, S, true, o, slot, wpart, lane, red,
                               &S_used);
    }
  }
  pdl_launch_dependents();
}

// Launch shape of the row encoders: R blocks per lane (R * 512 values per
// warp) and WPR warps per row; 0 = rows too long (one CTA per row).
struct RowShape {
  int R, WPR;
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

}  // namespace

cudaError_t launch_nvfp4_per_token(const void* x, int64_t T, int64_t H,
                                   int64_t ldx, uint8_t* codes,
                                   uint8_t* scales, float* token_scales,
                                   int swizzled, cudaStream_t stream) {
  const int64_t T_pad = swizzled ? (T + 127) / 128 * 128 : T;
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  const RowShape sh = pick_shape(H);
  if (sh.R == 0) {
    return launch_pdl(nvfp4_token_long_kernel, dim3((unsigned)T_pad),
                      dim3(CTA_WARPS * 32), 0, stream, false, xs, T, H, ldx,
                      codes, scales, token_scales, swizzled);
  }
  const int rows_per_cta = CTA_WARPS / sh.WPR;
  const unsigned grid = (unsigned)((T_pad + rows_per_cta - 1) / rows_per_cta);
#define MXQ_TOKEN_LAUNCH(R_, W_)                                          \
  launch_pdl(nvfp4_token_kernel<R_, W_>, dim3(grid), dim3(CTA_WARPS * 32), \
             0, stream, false, xs, T, T_pad, H, ldx, codes, scales,        \
             token_scales, swizzled)
  if (sh.R == 1) return MXQ_TOKEN_LAUNCH(1, 1);
  if (sh.R == 2) return MXQ_TOKEN_LAUNCH(2, 1);
  if (sh.WPR == 1) return MXQ_TOKEN_LAUNCH(4, 1);
  if (sh.WPR == 2) return MXQ_TOKEN_LAUNCH(4, 2);
  if (sh.WPR == 4) return MXQ_TOKEN_LAUNCH(4, 4);
  return MXQ_TOKEN_LAUNCH(4, 8);
#undef MXQ_TOKEN_LAUNCH
}

size_t nvfp4_weight_ws_bytes(int64_t num_groups) {
  return (size_t)(((kWsHeaderWords + num_groups) * 4 + 255) / 256 * 256);
}

cudaError_t nvfp4_take_wait_error(unsigned int* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_nvfp4_wait_error, sizeof(*word));
  if (e != cudaSuccess || *word == 0) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_nvfp4_wait_error, &zero, sizeof(zero));
}

namespace {

template <int R, int WPR>
cudaError_t launch_weight_coop(const GroupTable& tab, const GroupParams& p,
                               int dev, cudaStream_t stream) {
  static int occ[64] = {};
  int n = (dev >= 0 && dev < 64) ? occ[dev] : 0;
  if (n == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &n, nvfp4_weight_kernel<R, WPR>, CTA_WARPS * 32, 0);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) occ[dev] = n;
  }
  const unsigned grid = (unsigned)(n * sm_count(dev));
  return launch_pdl(nvfp4_weight_kernel<R, WPR>, dim3(grid),
                    dim3(CTA_WARPS * 32), 0, stream, true, tab, p);
}

}  // namespace

cudaError_t launch_nvfp4_weight_shared(
    int64_t num_groups, int num_parts, const void* const* parts,
    const int64_t* part_rows, int64_t K, uint8_t* codes, uint8_t* scales,
    float* group_scales, const float* group_scales_in, int swizzled,
    uint32_t* ws, cudaStream_t stream) {
  const RowShape sh = pick_shape(K);
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
  p.units_per_group =
      (p.part_chunk0[num_parts] + kAmaxUnitChunks - 1) / kAmaxUnitChunks;
  p.codes = codes;
  p.scales = scales;
  p.scale_stride = scale_bytes(p.R, K / 16, swizzled);
  p.group_scales = group_scales;
  p.S_in = group_scales_in;
  p.ws = ws;
  p.swizzled = swizzled;

  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  // Groups per L2 chunk: what phase A reads should still be in L2 when
  // phase B reads it again.
  const int64_t group_bytes = p.R * K * 2;
  int64_t chunk = kMaxGroupsPerLaunch;
  if (!group_scales_in && group_bytes > 0) {
    chunk = (int64_t)(0.55 * (double)l2_bytes(dev)) / group_bytes;
    chunk = chunk < 1 ? 1 : chunk;
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
    p.chunk = (int)(chunk < ng ? chunk : ng);
    if (!group_scales_in) {
      // Zero the barrier counter and this launch's amax words.
      err = cudaMemsetAsync(ws, 0, kWsHeaderWords * 4, stream);
      if (err == cudaSuccess)
        err = cudaMemsetAsync(ws + kWsHeaderWords + g0, 0, (size_t)ng * 4,
                              stream);
      if (err != cudaSuccess) return err;
    }
    if (sh.R == 1) err = launch_weight_coop<1, 1>(tab, p, dev, stream);
    else if (sh.R == 2) err = launch_weight_coop<2, 1>(tab, p, dev, stream);
    else if (sh.WPR == 1) err = launch_weight_coop<4, 1>(tab, p, dev, stream);
    else if (sh.WPR == 2) err = launch_weight_coop<4, 2>(tab, p, dev, stream);
    else if (sh.WPR == 4) err = launch_weight_coop<4, 4>(tab, p, dev, stream);
    else err = launch_weight_coop<4, 8>(tab, p, dev, stream);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace mxq
