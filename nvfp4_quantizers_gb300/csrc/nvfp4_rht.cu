// nvfp4_rht.cu -- per-token NVFP4 with the stabilizers of the original NVFP4
// pretraining recipe: a 16-value Random Hadamard Transform before
// quantization and stochastic rounding of the E2M1 codes.
//
// "Miles: end-to-end MXFP8 and per-token NVFP4 RL", NVFP4 recipe section:
// the pretraining recipe uses stochastic rounding (applied to gradients, so
// that the quantized values are unbiased) and Random Hadamard Transforms
// (which disperse block-level outliers, especially of weight-gradient GEMM
// inputs); the RL recipe itself leaves both out.
//
// Readings (the pages give no formulas):
//   random bits  Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
//                numbers: as easy as 1, 2, 3", SC 2011): every element's bits
//                depend only on (seed, position)
//   RHT          y = (1/4) H16 (s * x) per 16-value block along the row, H16
//                the Sylvester Hadamard matrix, s the signs given by the low
//                16 bits of word 0 of Philox(counter 0, key (seed, 1)) (bit i
//                set: s_i = -1); binary32 butterflies h = 1, 2, 4, 8
//                ((a, b) -> (a + b, a - b)), then times 1/4 (exact)
//   scales       the per-token S and the E4M3 block scales of the per-token
//                quantizer, computed on the transformed binary32 values
//   SR           element (r, c): u = (w >> 8) 2^-24, w the 32-bit word c % 8
//                of Philox(counter (r, c / 8, 0, 0), key (seed, 2)); |v|
//                (saturated at 6) rounds up to the next E2M1 magnitude iff
//                u < (|v| - lo) / (hi - lo); sign kept
//
// Design (sm_103a): one warp per row (grid-stride), a lane per 16-value
// block.  Pass 1 loads (up to four blocks per lane at once), transforms and
// reduces the row's amax; pass 2 encodes.  Rows of up to 4 x 32 blocks keep
// their transformed values in registers between the passes; longer rows
// are reloaded (from L1/L2) and transformed again in pass 2.
#include <float.h>

#include "common.cuh"
#include "launch.h"

namespace mxq {

namespace {

constexpr int RS_THREADS = 256;
constexpr int kChunk = 4;           // blocks per lane loaded together
constexpr unsigned FULL = 0xffffffffu;

// Philox4x64-10: one 4-word block from a 4-word counter and a 2-word key.
__device__ __forceinline__ void philox4x64(uint64_t c0, uint64_t c1,
                                           uint64_t c2, uint64_t c3,
                                           uint64_t k0, uint64_t k1,
                                           uint64_t out[4]) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
    const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
    const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += W0;
    k1 += W1;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

// Two binary32 values in one 64-bit register pair, and packed add /
// subtract of two such pairs (two IEEE operations each, round to nearest
// even, no flush to zero).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t p, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// The 16 binary32 values of a block from its bf16 words, sign-flipped,
// butterflied and, for QUARTER, scaled by 1/4 when rht.  smask[i] holds the
// signs of values 2i (bit 15) and 2i + 1 (bit 31): they are applied to the
// packed bf16 words, as a sign flip commutes with the exact widening.
template <bool QUARTER = true>
__device__ __forceinline__ void block_values(const uint4& a, const uint4& b,
                                             bool rht,
                                             const uint32_t (&smask)[8],
                                             float (&v)[16]) {
  uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  if (rht) {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] ^= smask[i];
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16lo_to_f32(w[i]);
    v[2 * i + 1] = bf16hi_to_f32(w[i]);
  }
  if (!rht) return;
  // butterflies h = 1, 2, 4 on 64-bit pairs P[i] = (v[i], v[i + 8]): the
  // partners i ^ h of both halves sit in the same lanes of P[i ^ h], so one
  // packed add and one packed subtract do two butterflies; then h = 8
  // inside each pair.  The same IEEE operations in the same order as the
  // scalar stages.
  uint64_t P[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) P[i] = pack_f32x2(v[i], v[i + 8]);
#pragma unroll
  for (int h = 1; h < 8; h <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & h) == 0) {
        const uint64_t a = P[i], b = P[i + h];
        P[i] = add_f32x2(a, b);
        P[i + h] = sub_f32x2(a, b);
      }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float x0, x1;
    unpack_f32x2(P[i], x0, x1);
    v[i] = __fadd_rn(x0, x1);
    v[i + 8] = __fsub_rn(x0, x1);
  }
  if (QUARTER) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], 0.25f);
  }
}

__device__ __forceinline__ float block_amax(const float (&v)[16]) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
  return m;
}

// E2M1 code of v by stochastic rounding with u in [0, 1), without
// branches: the grid spacing d around a = min(|v|, 6) is 0.5 below 2, 1
// below 4 and 2 up to 6, i.e. 2^(e - 1) with e = max(floor(log2 a), 0);
// f = floor(a / d) (0 .. 3) puts lo = f d, the grid value at or below a,
// at code f + 2e (exact: d is a power of two), and the code steps up iff
// u d < a - lo, which is u < (a - lo) / (hi - lo) with both sides scaled
// by d (exact).
__device__ __forceinline__ uint32_t sr_e2m1(float v, float u) {
  const uint32_t neg = __float_as_uint(v) >> 31;
  const float a = fminf(fabsf(v), 6.0f);
  const int e = max((int)(__float_as_uint(a) >> 23) - 127, 0);
  const float d = __uint_as_float((uint32_t)(126 + e) << 23);
  const float inv_d = __uint_as_float((uint32_t)(128 - e) << 23);
  const float f = floorf(__fmul_rn(a, inv_d));
  uint32_t idx = (uint32_t)f + 2u * (uint32_t)e;
  if (__fmul_rn(u, d) < __fsub_rn(a, __fmul_rn(f, d))) ++idx;
  return idx | (neg << 3);
}

// Block scale and codes of block b of a row from its 16 transformed values
// v (1/4 applied), then the stores: 8 bytes of codes, and (lanes 0, 4, ...)
// the 32-bit word of four consecutive block scales.  All 32 lanes call it.
template <bool SR>
__device__ __forceinline__ void encode_store(
    const float (&v)[16], float S, float six_s, int64_t row, int64_t b,
    bool real, bool valid, int64_t H, int64_t nb, int64_t col_tiles,
    uint64_t seed, int swizzled, int lane, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales) {
  uint32_t sb = 0;
  if (S != 0.0f)
    sb = cvt_e4m3x2(__fdiv_rn(block_amax(v), six_s), 0.0f) & 0xFFu;
  const float d = __fmul_rn(e4m3_to_f32(sb), S);
  float enc = 0.0f;
  if (d != 0.0f) enc = fminf(__frcp_rn(d), FLT_MAX);
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; i += 2)
    fmul2(v[i], v[i + 1], enc, enc, q[i], q[i + 1]);
  uint32_t lo, hi;
  if (!SR) {
    lo = cvt_e2m1x8(*reinterpret_cast<const float(*)[8]>(&q[0]));
    hi = cvt_e2m1x8(*reinterpret_cast<const float(*)[8]>(&q[8]));
  } else {
    uint32_t c[16];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      uint64_t o[4];
      philox4x64((uint64_t)row, (uint64_t)(b * 2 + g), 0, 0, seed, 2, o);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint64_t wd = o[k >> 1];
        const uint32_t w = (uint32_t)((k & 1) ? (wd >> 32) : wd);
        const float u = __uint2float_rn(w >> 8) * 0x1p-24f;
        c[g * 8 + k] = sr_e2m1(q[g * 8 + k], u);
      }
    }
    lo = hi = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      lo |= c[k] << (4 * k);
      hi |= c[8 + k] << (4 * k);
    }
  }
  if (real && valid) st_v2(codes + row * (H >> 1) + b * 8, lo, hi);
  // lanes 4i .. 4i+3 hold four consecutive blocks: one 32-bit word
  const uint32_t pair = sb | (__shfl_down_sync(FULL, sb, 1) << 8);
  const uint32_t word = pair | (__shfl_down_sync(FULL, pair, 2) << 16);
  if ((lane & 3) == 0) {
    if (swizzled) {
      if (b < 4 * col_tiles)
        *reinterpret_cast<uint32_t*>(scales + swz_offset(row, b, col_tiles)) =
            word;
    } else if (real) {
      if ((nb & 3) == 0) {
        if (b < nb)
          *reinterpret_cast<uint32_t*>(scales + row * nb + b) = word;
      } else {
        for (int k = 0; k < 4; ++k)
          if (b + k < nb) scales[row * nb + b + k] = (uint8_t)(word >> (8 * k));
      }
    }
  }
}

// SR is a template parameter: without stochastic rounding the kernel needs
// no Philox state.  KEEP (no SR, rows of at most 4 x 32 blocks, e.g. hidden
// 2048): pass 1 keeps each lane's transformed blocks in registers (64
// values) and pass 2 encodes them, instead of reloading and transforming
// the row again (ragged 132106 x 2048 with the RHT: 211 -> 179 us); it
// runs 3 CTAs per SM at 80 registers with a few values spilled to L1
// (2 CTAs at 120 registers: 178 -> 170 us); otherwise pass 2 reloads the
// row (from L1/L2) and transforms it again.
template <bool SR, bool KEEP>
__global__ void __launch_bounds__(RS_THREADS, SR ? 2 : (KEEP ? 3 : 4))
    nvfp4_rht_sr_kernel(const uint16_t* __restrict__ x, int64_t T,
                        int64_t T_pad, int64_t H, int64_t ldx, uint64_t seed,
                        int flags, uint8_t* __restrict__ codes,
                        uint8_t* __restrict__ scales, float* __restrict__ S_out,
                        int swizzled) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = ((int64_t)blockIdx.x * RS_THREADS + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * RS_THREADS) >> 5;
  const bool rht = (flags & 1) != 0;
  const int64_t nb = H >> 4;
  const int64_t col_tiles = (nb + 3) >> 2;
  const int64_t iters = (nb + 31) >> 5;           // warp-uniform
  uint32_t signs = 0;
  if (rht) {
    uint64_t o[4];
    philox4x64(0, 0, 0, 0, seed, 1, o);
    signs = (uint32_t)(o[0] & 0xffffu);
  }
  uint32_t smask[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    smask[i] = (((signs >> (2 * i)) & 1u) << 15) |
               (((signs >> (2 * i + 1)) & 1u) << 31);
  pdl_wait();
  for (int64_t row = warp_id; row < T_pad; row += nwarps) {
    const bool real = row < T;
    const uint16_t* xr = x + (real ? row : 0) * ldx;
    // ---- pass 1: the row's amax over the (transformed) values; up to
    // four of a lane's blocks loaded before any is transformed ----
    float am = 0.0f;
    float kept[KEEP ? kChunk : 1][16];
    for (int64_t j0 = 0; j0 < (KEEP ? 1 : iters); j0 += kChunk) {
      uint4 raw[2 * kChunk];
#pragma unroll
      for (int k = 0; k < kChunk; ++k) {
        const int64_t b = (j0 + k) * 32 + lane;
        if (real && j0 + k < iters && b < nb) {
          raw[2 * k] = *reinterpret_cast<const uint4*>(xr + b * 16);
          raw[2 * k + 1] = *reinterpret_cast<const uint4*>(xr + b * 16 + 8);
        } else {
          raw[2 * k] = make_uint4(0, 0, 0, 0);
          raw[2 * k + 1] = raw[2 * k];
        }
      }
#pragma unroll
      for (int k = 0; k < kChunk; ++k) {
        float v[16];
        block_values<false>(raw[2 * k], raw[2 * k + 1], rht, smask, v);
        am = fmaxf(am, block_amax(v));
        if (KEEP) {
#pragma unroll
          for (int i = 0; i < 16; ++i) kept[KEEP ? k : 0][i] = v[i];
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(FULL, am, o));
    // pass 1 leaves out the 1/4: rounding is monotone and symmetric, so the
    // largest |fl(y / 4)| is fl(max |y| / 4), subnormals included
    if (rht) am = __fmul_rn(am, 0.25f);
    const float S = __fdiv_rn(am, kNvfp4ScaleDenom);
    const float six_s = __fmul_rn(6.0f, S);
    if (real && lane == 0) S_out[row] = S;
    // ---- pass 2: block scales and codes ----
    if (KEEP) {
#pragma unroll
      for (int k = 0; k < kChunk; ++k) {
        if (k >= iters) break;                    // warp-uniform
        const int64_t b = k * 32 + lane;
        const bool valid = b < nb;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          v[i] = (real && valid)
                     ? (rht ? __fmul_rn(kept[KEEP ? k : 0][i], 0.25f)
                            : kept[KEEP ? k : 0][i])
                     : 0.0f;
        encode_store<SR>(v, S, six_s, row, b, real, valid, H, nb, col_tiles,
                         seed, swizzled, lane, codes, scales);
      }
    } else {
      for (int64_t j = 0; j < iters; ++j) {
        const int64_t b = j * 32 + lane;
        const bool valid = b < nb;
        float v[16];
        if (real && valid) {
          const uint4 a0 = *reinterpret_cast<const uint4*>(xr + b * 16);
          const uint4 a1 = *reinterpret_cast<const uint4*>(xr + b * 16 + 8);
          block_values(a0, a1, rht, smask, v);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.0f;
        }
        encode_store<SR>(v, S, six_s, row, b, real, valid, H, nb, col_tiles,
                         seed, swizzled, lane, codes, scales);
      }
    }
  }
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_nvfp4_rht_sr(const void* x, int64_t T, int64_t H,
                                int64_t ldx, uint64_t seed, int flags,
                                uint8_t* codes, uint8_t* scales,
                                float* token_scales, int swizzled,
                                cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int64_t T_pad = swizzled ? (T + 127) / 128 * 128 : T;
  const int64_t per_cta = RS_THREADS / 32;
  // Rows kept in registers only without SR: the Philox state and the kept
  // values together spill (ragged 132106 x 2048 with SR: 786 -> 874 us).
  const bool keep = !(flags & 2) && ((H >> 4) + 31) / 32 <= kChunk;
  int64_t grid = (T_pad + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)sm_count(dev) * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
#define MXQ_RHT_LAUNCH(SR_, KEEP_)                                          \
  launch_pdl(nvfp4_rht_sr_kernel<SR_, KEEP_>, dim3((unsigned)grid),        \
             dim3(RS_THREADS), 0, stream, false,                           \
             static_cast<const uint16_t*>(x), T, T_pad, H, ldx, seed, flags, \
             codes, scales, token_scales, swizzled)
  if (flags & 2) return MXQ_RHT_LAUNCH(true, false);
  return keep ? MXQ_RHT_LAUNCH(false, true) : MXQ_RHT_LAUNCH(false, false);
#undef MXQ_RHT_LAUNCH
}

}  // namespace mxq
