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
// Weight groups take two kernels: a grid-wide amax of the group (CTA
// partial maxima combined with an integer atomicMax on the float bits,
// exact for non-negative values), then the row encoder with the group's S.
// Groups are processed in chunks sized to a fraction of L2 so that the
// encoder's second read of a chunk is served from L2, not HBM.
#include <float.h>

#include "common.cuh"
#include "launch.h"

namespace mxq {

namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int ROW_WARPS = 8;                 // rows per 256-thread CTA
constexpr int kMaxGroupsPerLaunch = 64;

struct RowOut {
  uint8_t* codes_row;   // H/2 bytes of this row
  uint8_t* scales;      // base of this row's scale matrix
  int64_t row;          // row index within the scale matrix
  int64_t col_tiles;    // swizzled: ceil(nblocks / 4)
  int64_t nblocks;      // H / 16
  int swizzled;
};

__device__ __forceinline__ uint32_t chunk_absmax(const uint4& v) {
  return bf16x2_hmax(bf16x2_max(bf16x2_absmax(v.x, v.y),
                                bf16x2_absmax(v.z, v.w)));
}

// Encode ROUNDS x 32 chunks of one row (chunk c = chunk_base + r*32 + lane)
// with FP32 scale S.  Lanes holding chunks beyond the row carry zeros.
template <int ROUNDS>
__device__ __forceinline__ void encode_rounds(const uint4 (&v)[ROUNDS],
                                              int chunk_base, int nchunks,
                                              float S, int lane,
                                              bool write_codes,
                                              const RowOut& o) {
  const float six_s = __fmul_rn(6.0f, S);
  const int64_t padded_cols = o.swizzled ? ((o.nblocks + 3) & ~int64_t(3))
                                         : o.nblocks;
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    if (chunk_base + r * 32 >= nchunks) break;       // warp-uniform
    const int c = chunk_base + r * 32 + lane;
    uint32_t a = chunk_absmax(v[r]);
    a = max(a, __shfl_xor_sync(FULL, a, 1));
    const float ab = __uint_as_float(a << 16);
    uint32_t sb = 0;
    if (S != 0.0f) sb = cvt_e4m3x2(__fdiv_rn(ab, six_s), 0.0f) & 0xFFu;
    const float d = __fmul_rn(e4m3_to_f32(sb), S);
    float enc = 0.0f;
    if (d != 0.0f) enc = fminf(__frcp_rn(d), FLT_MAX);
    float q[8];
    q[0] = __fmul_rn(bf16lo_to_f32(v[r].x), enc);
    q[1] = __fmul_rn(bf16hi_to_f32(v[r].x), enc);
    q[2] = __fmul_rn(bf16lo_to_f32(v[r].y), enc);
    q[3] = __fmul_rn(bf16hi_to_f32(v[r].y), enc);
    q[4] = __fmul_rn(bf16lo_to_f32(v[r].z), enc);
    q[5] = __fmul_rn(bf16hi_to_f32(v[r].z), enc);
    q[6] = __fmul_rn(bf16lo_to_f32(v[r].w), enc);
    q[7] = __fmul_rn(bf16hi_to_f32(v[r].w), enc);
    const uint32_t packed = cvt_e2m1x8(q);
    if (write_codes && c < nchunks)
      *reinterpret_cast<uint32_t*>(o.codes_row + (int64_t)c * 4) = packed;
    // Lanes 0, 8, 16, 24 gather the scales of blocks b0..b0+3 (held by the
    // even lanes l, l+2, l+4, l+6).
    const uint32_t s1 = __shfl_down_sync(FULL, sb, 2);
    const uint32_t s2 = __shfl_down_sync(FULL, sb, 4);
    const uint32_t s3 = __shfl_down_sync(FULL, sb, 6);
    if ((lane & 7) == 0) {
      const int64_t b0 = c >> 1;
      const uint32_t word = sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
      if (o.swizzled) {
        if (b0 < padded_cols)
          *reinterpret_cast<uint32_t*>(
              o.scales + swz_offset(o.row, b0, o.col_tiles)) = word;
      } else if ((o.nblocks & 3) == 0) {
        if (b0 < o.nblocks)
          *reinterpret_cast<uint32_t*>(o.scales + o.row * o.nblocks + b0) =
              word;
      } else {
        for (int j = 0; j < 4; ++j)
          if (b0 + j < o.nblocks)
            o.scales[o.row * o.nblocks + b0 + j] = (uint8_t)(word >> (8 * j));
      }
    }
  }
}

template <int ROUNDS>
__device__ __forceinline__ void load_rounds(uint4 (&v)[ROUNDS],
                                            const uint16_t* row,
                                            int chunk_base, int nchunks,
                                            bool real, int lane) {
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int c = chunk_base + r * 32 + lane;
    v[r] = (real && c < nchunks) ? ld_stream_v4(row + (int64_t)c * 8)
                                 : make_uint4(0, 0, 0, 0);
  }
}

template <int ROUNDS>
__device__ __forceinline__ uint32_t rounds_absmax(const uint4 (&v)[ROUNDS]) {
  uint32_t a = 0;
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) a = max(a, chunk_absmax(v[r]));
  return a;
}

__device__ __forceinline__ uint32_t warp_max(uint32_t a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(FULL, a, o));
  return a;
}

// ---------------------------------------------------------------------------
// Per-token activations.
// ---------------------------------------------------------------------------
template <int ROUNDS>
__global__ void __launch_bounds__(ROW_WARPS * 32)
    nvfp4_token_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t T_pad,
                       int64_t H, int64_t ldx, uint8_t* __restrict__ codes,
                       uint8_t* __restrict__ scales, float* __restrict__ S_out,
                       int swizzled) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * ROW_WARPS + (threadIdx.x >> 5);
  if (t >= T_pad) return;
  const bool real = t < T;
  const int nchunks = (int)(H >> 3);
  const uint16_t* row = x + t * ldx;
  RowOut o{codes + t * (H >> 1), scales, t, ((H >> 4) + 3) >> 2, H >> 4,
           swizzled};
  float S;
  if ((int64_t)ROUNDS * 32 >= nchunks) {
    uint4 v[ROUNDS];
    load_rounds<ROUNDS>(v, row, 0, nchunks, real, lane);
    const uint32_t a = warp_max(rounds_absmax<ROUNDS>(v));
    S = __fdiv_rn(__uint_as_float(a << 16), kNvfp4ScaleDenom);
    encode_rounds<ROUNDS>(v, 0, nchunks, S, lane, real, o);
  } else {
    // Long rows: amax pass, then a second (cache-served) pass to encode.
    uint32_t a = 0;
    for (int base = 0; base < nchunks; base += ROUNDS * 32) {
      uint4 v[ROUNDS];
      load_rounds<ROUNDS>(v, row, base, nchunks, real, lane);
      a = max(a, rounds_absmax<ROUNDS>(v));
    }
    a = warp_max(a);
    S = __fdiv_rn(__uint_as_float(a << 16), kNvfp4ScaleDenom);
    for (int base = 0; base < nchunks; base += ROUNDS * 32) {
      uint4 v[ROUNDS];
      load_rounds<ROUNDS>(v, row, base, nchunks, real, lane);
      encode_rounds<ROUNDS>(v, base, nchunks, S, lane, real, o);
    }
  }
  if (real && lane == 0) S_out[t] = S;
}

// ---------------------------------------------------------------------------
// Weight groups.
// ---------------------------------------------------------------------------
struct GroupTable {
  const uint16_t* part[kMaxGroupsPerLaunch][kMaxParts];
};

struct GroupParams {
  int num_parts;
  int64_t part_row0[kMaxParts + 1];   // prefix sums of the parts' rows
  int64_t R, R_pad, K;
  int64_t g0;                         // global index of local group 0
  int ng;
  uint8_t* codes;                     // group g at g * R * K/2
  uint8_t* scales;                    // group g at g * scale_stride
  int64_t scale_stride;
  float* group_scales;
  const float* S_in;                  // NULL: S from amax
  const uint32_t* amax;               // f32 bit patterns, global group index
  int swizzled;
};

__global__ void __launch_bounds__(256)
    nvfp4_group_amax_kernel(const __grid_constant__ GroupTable tab,
                            const __grid_constant__ GroupParams p,
                            uint32_t* __restrict__ amax) {
  const int gl = blockIdx.y;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  uint32_t a = 0;
  for (int pi = 0; pi < p.num_parts; ++pi) {
    const uint16_t* base = tab.part[gl][pi];
    const int64_t n = (p.part_row0[pi + 1] - p.part_row0[pi]) * p.K / 8;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
      const uint4 v0 = ld_stream_v4(base + i * 8);
      const uint4 v1 = ld_stream_v4(base + (i + stride) * 8);
      const uint4 v2 = ld_stream_v4(base + (i + 2 * stride) * 8);
      const uint4 v3 = ld_stream_v4(base + (i + 3 * stride) * 8);
      a = max(a, max(max(chunk_absmax(v0), chunk_absmax(v1)),
                     max(chunk_absmax(v2), chunk_absmax(v3))));
    }
    for (; i < n; i += stride) a = max(a, chunk_absmax(ld_stream_v4(base + i * 8)));
  }
  a = warp_max(a);
  __shared__ uint32_t red[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = max(m, red[w]);
    // Non-negative float bit patterns order like their values.
    atomicMax(&amax[p.g0 + gl], m << 16);
  }
}

template <int ROUNDS>
__global__ void __launch_bounds__(ROW_WARPS * 32)
    nvfp4_group_rows_kernel(const __grid_constant__ GroupTable tab,
                            const __grid_constant__ GroupParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * ROW_WARPS + (threadIdx.x >> 5);
  if (w >= (int64_t)p.ng * p.R_pad) return;
  const int gl = (int)(w / p.R_pad);
  const int64_t r = w - (int64_t)gl * p.R_pad;
  const int64_t g = p.g0 + gl;
  const bool real = r < p.R;
  const uint16_t* row = nullptr;
  if (real) {
    int pi = 0;
    while (pi + 1 < p.num_parts && r >= p.part_row0[pi + 1]) ++pi;
    row = tab.part[gl][pi] + (r - p.part_row0[pi]) * p.K;
  }
  const float S = p.S_in ? p.S_in[g]
                         : __fdiv_rn(__uint_as_float(p.amax[g]),
                                     kNvfp4ScaleDenom);
  if (r == 0 && lane == 0) p.group_scales[g] = S;
  const int nchunks = (int)(p.K >> 3);
  RowOut o{p.codes + (g * p.R + r) * (p.K >> 1), p.scales + g * p.scale_stride,
           r, ((p.K >> 4) + 3) >> 2, p.K >> 4, p.swizzled};
  for (int base = 0; base < nchunks; base += ROUNDS * 32) {
    uint4 v[ROUNDS];
    load_rounds<ROUNDS>(v, row, base, nchunks, real, lane);
    encode_rounds<ROUNDS>(v, base, nchunks, S, lane, real, o);
  }
}

// Smallest supported ROUNDS >= the rounds a row needs (capped at 16; longer
// rows loop).
int pick_rounds(int64_t H) {
  const int64_t need = ((H >> 3) + 31) / 32;
  if (need <= 1) return 1;
  if (need <= 2) return 2;
  if (need <= 4) return 4;
  if (need <= 8) return 8;
  return 16;
}

}  // namespace

cudaError_t launch_nvfp4_per_token(const void* x, int64_t T, int64_t H,
                                   int64_t ldx, uint8_t* codes,
                                   uint8_t* scales, float* token_scales,
                                   int swizzled, cudaStream_t stream) {
  const int64_t T_pad = swizzled ? (T + 127) / 128 * 128 : T;
  const int64_t grid = (T_pad + ROW_WARPS - 1) / ROW_WARPS;
  const uint16_t* xs = static_cast<const uint16_t*>(x);
#define MXQ_TOKEN_LAUNCH(R)                                                  \
  nvfp4_token_kernel<R><<<(unsigned)grid, ROW_WARPS * 32, 0, stream>>>(      \
      xs, T, T_pad, H, ldx, codes, scales, token_scales, swizzled)
  switch (pick_rounds(H)) {
    case 1: MXQ_TOKEN_LAUNCH(1); break;
    case 2: MXQ_TOKEN_LAUNCH(2); break;
    case 4: MXQ_TOKEN_LAUNCH(4); break;
    case 8: MXQ_TOKEN_LAUNCH(8); break;
    default: MXQ_TOKEN_LAUNCH(16); break;
  }
#undef MXQ_TOKEN_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_weight_shared(
    int64_t num_groups, int num_parts, const void* const* parts,
    const int64_t* part_rows, int64_t K, uint8_t* codes, uint8_t* scales,
    float* group_scales, const float* group_scales_in, int swizzled,
    uint32_t* amax_ws, cudaStream_t stream) {
  GroupParams p;
  p.num_parts = num_parts;
  p.part_row0[0] = 0;
  for (int i = 0; i < num_parts; ++i)
    p.part_row0[i + 1] = p.part_row0[i] + part_rows[i];
  for (int i = num_parts + 1; i <= kMaxParts; ++i)
    p.part_row0[i] = p.part_row0[num_parts];
  p.R = p.part_row0[num_parts];
  p.R_pad = swizzled ? (p.R + 127) / 128 * 128 : p.R;
  p.K = K;
  p.codes = codes;
  p.scales = scales;
  p.scale_stride = scale_bytes(p.R, K / 16, swizzled);
  p.group_scales = group_scales;
  p.S_in = group_scales_in;
  p.amax = amax_ws;
  p.swizzled = swizzled;

  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  // Groups per launch: the chunk read by the amax kernel should still be in
  // L2 when the encoder reads it again.
  const int64_t group_bytes = p.R * K * 2;
  int64_t chunk = kMaxGroupsPerLaunch;
  if (!group_scales_in && group_bytes > 0) {
    chunk = (int64_t)(0.4 * (double)l2_bytes(dev)) / group_bytes;
    chunk = chunk < 1 ? 1 : (chunk > kMaxGroupsPerLaunch ? kMaxGroupsPerLaunch : chunk);
  }
  const int64_t group_chunks = group_bytes / 16;
  int64_t ctas_per_group = (group_chunks + 256 * 16 - 1) / (256 * 16);
  ctas_per_group = ctas_per_group < 1 ? 1 : (ctas_per_group > 65535 ? 65535 : ctas_per_group);

  GroupTable tab;
  for (int64_t g0 = 0; g0 < num_groups; g0 += chunk) {
    const int ng = (int)((num_groups - g0) < chunk ? (num_groups - g0) : chunk);
    for (int gl = 0; gl < kMaxGroupsPerLaunch; ++gl)
      for (int pi = 0; pi < kMaxParts; ++pi)
        tab.part[gl][pi] =
            (gl < ng && pi < num_parts)
                ? static_cast<const uint16_t*>(parts[(g0 + gl) * num_parts + pi])
                : nullptr;
    p.g0 = g0;
    p.ng = ng;
    if (!group_scales_in) {
      err = cudaMemsetAsync(amax_ws + g0, 0, (size_t)ng * 4, stream);
      if (err != cudaSuccess) return err;
      nvfp4_group_amax_kernel<<<dim3((unsigned)ctas_per_group, (unsigned)ng),
                                256, 0, stream>>>(tab, p, amax_ws);
      err = cudaGetLastError();
      if (err != cudaSuccess) return err;
    }
    const int64_t rows = (int64_t)ng * p.R_pad;
    const unsigned grid = (unsigned)((rows + ROW_WARPS - 1) / ROW_WARPS);
#define MXQ_GROUP_LAUNCH(R) \
  nvfp4_group_rows_kernel<R><<<grid, ROW_WARPS * 32, 0, stream>>>(tab, p)
    switch (pick_rounds(K)) {
      case 1: MXQ_GROUP_LAUNCH(1); break;
      case 2: MXQ_GROUP_LAUNCH(2); break;
      case 4: MXQ_GROUP_LAUNCH(4); break;
      case 8: MXQ_GROUP_LAUNCH(8); break;
      default: MXQ_GROUP_LAUNCH(16); break;
    }
#undef MXQ_GROUP_LAUNCH
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace mxq
