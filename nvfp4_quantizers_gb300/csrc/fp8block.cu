// fp8block.cu -- FP8 E4M3 with one FP32 scale per block: 1x128 activation
// tiles, 128x128 weight blocks, their dequantization to bf16, and the
// backward-orientation conversion of 1x128-tile activations.
//
// "Miles: end-to-end MXFP8 and per-token NVFP4 RL", introduction: the
// DeepSeek-V3-style block-scaled FP8 recipe scales weights in 128x128
// blocks and activations in 1x128 tiles, one FP32 scale per tile or block
// computed online.  MXFP8 recipe section: that recipe stores forward
// activations in 1x128 tiles and, before the backward GEMM, converts them
// to the backward orientation by dequantizing and requantizing.
//
// Arithmetic (IEEE binary32, round-to-nearest-even, no FTZ, no FMA):
//   S    = amax / 448          (a decode scale: value = code * S)
//   enc  = 1 / S               (0 when S = 0, clamped to FLT_MAX)
//   code = E4M3_RNE(x * enc)   (saturating at +-448, sign kept)
//   y    = bf16_RNE(E4M3(code) * S)
// The conversion dequantizes a 128 x 128 tile of X [M x K] to bf16 exactly
// as the dequantizer does, transposes it in shared memory and quantizes
// each column (128 consecutive rows of X) as one 1x128 tile of X^T.
//
// Design (sm_103a): HBM-streaming.  Tiles: 8 lanes per 1x128 tile, 32
// bytes of bf16 per lane in one load (two tiles per lane in flight), amax
// by three shuffles, 16 codes per lane in one 16-byte store.  Blocks: one
// CTA per 128x128 block in a grid-stride loop, the block staged in shared
// memory by one TMA load (bounded wait).  Dequantizer: one 16-code unit
// per thread per step, one 32-byte store.  Conversion: all of a thread's
// code loads issued before it decodes, and eight columns quantized per
// step with one reduce-scatter for all of them.
#include <float.h>

#include "common.cuh"
#include "launch.h"

namespace mxq {

namespace {

constexpr int FB_THREADS = 256;
constexpr unsigned FULL = 0xffffffffu;

// S and enc of a block whose amax (bf16 bit pattern) is a.
__device__ __forceinline__ void fb_scales(uint32_t a, float& S, float& enc) {
  S = __fdiv_rn(__uint_as_float(a << 16), 448.0f);
  enc = 0.0f;
  if (S != 0.0f) enc = fminf(__frcp_rn(S), FLT_MAX);
}

// max |x| (bf16 bits) of 16 packed bf16 values.
__device__ __forceinline__ uint32_t absmax16(const uint4& a, const uint4& b) {
  const uint32_t m =
      bf16x2_maxabs(bf16x2_maxabs(bf16x2_maxabs(a.x, a.y),
                                  bf16x2_maxabs(a.z, a.w)),
                    bf16x2_maxabs(bf16x2_maxabs(b.x, b.y),
                                  bf16x2_maxabs(b.z, b.w)));
  return bf16x2_hmax(m & 0x7FFF7FFFu);
}

// 16 bf16 values -> 16 E4M3 codes (element 0 in the lowest byte).
__device__ __forceinline__ uint4 encode16(const uint4& a, const uint4& b,
                                          float enc) {
  return make_uint4(
      bf16x2_scale_e4m3x2(a.x, enc, enc) |
          (bf16x2_scale_e4m3x2(a.y, enc, enc) << 16),
      bf16x2_scale_e4m3x2(a.z, enc, enc) |
          (bf16x2_scale_e4m3x2(a.w, enc, enc) << 16),
      bf16x2_scale_e4m3x2(b.x, enc, enc) |
          (bf16x2_scale_e4m3x2(b.y, enc, enc) << 16),
      bf16x2_scale_e4m3x2(b.z, enc, enc) |
          (bf16x2_scale_e4m3x2(b.w, enc, enc) << 16));
}

__device__ __forceinline__ void load16(const uint16_t* p, bool wide, uint4& a,
                                       uint4& b) {
  if (wide) {
    ld_stream_v8(p, a, b);
  } else {
    a = ld_stream_v4(p);
    b = ld_stream_v4(p + 8);
  }
}

// 1x128 tiles along the rows of x [rows x cols]: lanes 8s .. 8s+7 of a warp
// take tile 4w + s, 16 values each.
__global__ void __launch_bounds__(FB_THREADS)
    fp8blk_tile_kernel(const uint16_t* __restrict__ x, int64_t rows,
                       int64_t cols, int64_t ldx, uint8_t* __restrict__ codes,
                       float* __restrict__ scales, int wide) {
  const int64_t per_row = cols >> 7;
  const int64_t ntiles = rows * per_row;
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3, part = lane & 7;
  const int64_t warp_id =
      ((int64_t)blockIdx.x * FB_THREADS + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * FB_THREADS) >> 5;
  pdl_wait();
  // two tiles per lane per step (tiles t0 + sub and t0 + 4 nwarps + sub),
  // both loads issued before either is used
  for (int64_t t0 = warp_id * 4; t0 < ntiles; t0 += nwarps * 8) {
    int64_t t[2], r[2], c[2];
    bool valid[2];
    uint4 a[2], b[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      t[h] = t0 + h * nwarps * 4 + sub;
      valid[h] = t[h] < ntiles;
      r[h] = valid[h] ? t[h] / per_row : 0;
      c[h] = valid[h] ? (t[h] - r[h] * per_row) * 128 + part * 16 : 0;
      a[h] = make_uint4(0, 0, 0, 0);
      b[h] = a[h];
      if (valid[h]) load16(x + r[h] * ldx + c[h], wide, a[h], b[h]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t m = absmax16(a[h], b[h]);
      m = max(m, __shfl_xor_sync(FULL, m, 1));
      m = max(m, __shfl_xor_sync(FULL, m, 2));
      m = max(m, __shfl_xor_sync(FULL, m, 4));
      float S, enc;
      fb_scales(m, S, enc);
      if (valid[h]) {
        st_v4(codes + r[h] * cols + c[h], encode16(a[h], b[h], enc));
        if (part == 0) scales[t[h]] = S;
      }
    }
  }
  pdl_launch_dependents();
}

// 128x128 blocks: a CTA takes one block at a time, brought into shared
// memory by one 2-D TMA load (128 x 128 bf16, 32 KiB); the next block's
// load is issued as soon as every thread has read the current one, so it
// lands while the codes are stored.  Six CTAs per SM: the block stays in
// shared memory, not registers, so that six blocks per SM (912 on the
// GPU) are in flight at once; with the block held in registers (64 values
// a thread) only four fit, and the 1024 blocks of an [8192 x 2048] weight
// took two full rounds of load latency.  A warp reads two rows per
// step, 16 bytes a lane (conflict-free), once for the amax and again to
// encode; the codes of a lane's 8 values leave in one 8-byte store (a
// warp writes two whole 128-byte rows).
constexpr int FB_BLK_CTAS = 6;

__device__ unsigned int g_fp8blk_wait_error = 0;

__device__ __forceinline__ uint32_t absmax8(const uint4& v) {
  return bf16x2_hmax(bf16x2_maxabs(bf16x2_maxabs(v.x, v.y),
                                   bf16x2_maxabs(v.z, v.w)) &
                     0x7FFF7FFFu);
}

__global__ void __launch_bounds__(FB_THREADS, FB_BLK_CTAS)
    fp8blk_block_kernel(const __grid_constant__ CUtensorMap tmap,
                        int64_t rows, int64_t cols,
                        uint8_t* __restrict__ codes,
                        float* __restrict__ scales) {
  __shared__ __align__(128) uint4 blk[128 * 16];   // row r: chunks 16 r ..
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t red[FB_THREADS / 32];
  __shared__ int abort_flag;
  const int64_t nbc = cols >> 7;
  const int64_t nblk = (rows >> 7) * nbc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ch = lane & 15;                         // 16-byte chunk of a row
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  auto issue = [&](int64_t k) {                     // thread 0
    const int64_t bi = k / nbc, bj = k - bi * nbc;
    mbar_arrive_expect_tx(b, 128 * 128 * 2);
    tma_load_2d(smem_addr(blk), &tmap, (int32_t)(bj * 128),
                (int32_t)(bi * 128), b);
  };
  bool pending = false;                             // thread 0: a load in flight
  if (threadIdx.x == 0 && (int64_t)blockIdx.x < nblk) {
    issue(blockIdx.x);
    pending = true;
  }
  uint32_t ph = 0;
  for (int64_t k = blockIdx.x; k < nblk; k += gridDim.x) {
    const bool ok = mbar_wait(b, ph, &abort_flag, &g_fp8blk_wait_error);
    if (ok) {                           // else the load may still land:
      ph ^= 1u;                         // phase ph stays the one in flight
      if (threadIdx.x == 0) pending = false;
    }
    // rows p * 16 + warp * 2 + lane / 16, p = 0 .. 7
    uint32_t m = 0;
    if (ok) {
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        const int r = pp * 16 + warp * 2 + (lane >> 4);
        m = max(m, absmax8(blk[r * 16 + ch]));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(FULL, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    uint32_t a = red[0];
#pragma unroll
    for (int w = 1; w < FB_THREADS / 32; ++w) a = max(a, red[w]);
    float S, enc;
    fb_scales(a, S, enc);
    uint2 cw[8];
#pragma unroll
    for (int pp = 0; pp < 8; ++pp) {
      const int r = pp * 16 + warp * 2 + (lane >> 4);
      const uint4 v = blk[r * 16 + ch];
      cw[pp] = make_uint2(bf16x2_scale_e4m3x2(v.x, enc, enc) |
                              (bf16x2_scale_e4m3x2(v.y, enc, enc) << 16),
                          bf16x2_scale_e4m3x2(v.z, enc, enc) |
                              (bf16x2_scale_e4m3x2(v.w, enc, enc) << 16));
    }
    __syncthreads();                    // blk and red are free again
    if (threadIdx.x == 0 && k + gridDim.x < nblk && !abort_flag) {
      issue(k + gridDim.x);
      pending = true;
    }
    if (ok) {
      const int64_t bi = k / nbc, bj = k - bi * nbc;
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        const int r = pp * 16 + warp * 2 + (lane >> 4);
        st_v2(codes + (bi * 128 + r) * cols + bj * 128 + ch * 8, cw[pp].x,
              cw[pp].y);
      }
      if (threadIdx.x == 0) scales[k] = S;
    }
  }
  if (threadIdx.x == 0 && pending) {
    // after a wait gave up: let the load in flight (phase ph) land before
    // the CTA exits (bounded)
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(b, ph) && global_timer_ns() - t0 < kWaitLimitNs) {
    }
  }
  pdl_launch_dependents();
}

// 16 E4M3 codes times S -> 16 bf16 (two 16-byte halves).
__device__ __forceinline__ void decode16(const uint4& c, float S, uint4& lo,
                                         uint4& hi) {
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
  uint32_t w[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    float a, b;
    e4m3x2_to_f32((cw[h >> 1] >> ((h & 1) * 16)) & 0xFFFFu, a, b);
    fmul2(a, b, S, S, a, b);
    w[h] = f32x2_to_bf16x2(a, b);
  }
  lo = make_uint4(w[0], w[1], w[2], w[3]);
  hi = make_uint4(w[4], w[5], w[6], w[7]);
}

// Dequantize codes [rows x cols] with scales per block of brows x 128
// (brows_log2 = 0 or 7).
__global__ void __launch_bounds__(FB_THREADS, 8)
    fp8blk_dequant_kernel(const uint8_t* __restrict__ codes,
                          const float* __restrict__ scales, int64_t rows,
                          int64_t cols, int brows_log2, int wide,
                          uint16_t* __restrict__ y) {
  const int64_t c16 = cols >> 4, nbc = cols >> 7;
  const int64_t n16 = rows * c16;
  pdl_wait();
  for (int64_t i = (int64_t)blockIdx.x * FB_THREADS + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * FB_THREADS) {
    const uint4 c = ld_stream_v4(codes + i * 16);
    const int64_t r = i / c16;
    const int64_t col = (i - r * c16) * 16;
    const float S = scales[(r >> brows_log2) * nbc + (col >> 7)];
    uint4 lo, hi;
    decode16(c, S, lo, hi);
    st_32B(y + i * 16, lo, hi, wide);
  }
  pdl_launch_dependents();
}

// Backward-orientation conversion: tile (ti, tj) of X [M x K] is dequantized
// into shared memory transposed (column-major bf16, 256 bytes a column),
// then each of its 128 columns is quantized as one 1x128 tile of X^T.
//   Dequantize: a thread takes 8 rows and 8 columns (one 8-byte code load
//   per row: a warp's loads are two whole 128-byte rows), converts them,
//   transposes the 8 x 8 bf16 block in registers (byte permutes) and
//   writes each column's 8 rows as one 16-byte store.  Chunk k (rows
//   8k .. 8k + 7) of column c sits at chunk k ^ ((c / 8) % 16) of the
//   column, so the 8 lanes of a store phase (8 column groups, one row
//   group) hit 8 different bank quads.  Its loads of the CTA's next tile
//   are issued right after, so they are in flight while this tile is
//   quantized.  (Two rows and 4-byte stores per column made the kernel
//   shared-memory-instruction bound: 512 store instructions a tile
//   against 128.)
//   Quantize: a warp takes 16 columns, 8 at a time, a lane 4 rows of each,
//   so every code store is 128 contiguous bytes per warp.  The 8 column
//   maxima are reduced together by a reduce-scatter over the lanes (lane
//   bits 4, 3, 2 select the half of the remaining columns a lane keeps: 4
//   + 2 + 1 exchanges, then two for the last lane bits), which leaves the
//   maximum of column (lane / 4) % 8 in lanes 4j .. 4j + 3; each lane then
//   derives the scales of that one column (one IEEE divide and reciprocal
//   per lane instead of per column and lane), and the encoders fetch the
//   8 reciprocals by shuffle.  (A thread per column, with no cross-lane
//   reduction, measured slower: its 16-byte stores land in 32 different
//   rows of X^T.)
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

// Byte offset of rows 8k .. 8k + 7 of column c in the transposed tile.
__device__ __forceinline__ int rt_chunk(int c, int k) {
  return c * 256 + ((k ^ ((c >> 3) & 15)) << 4);
}

__global__ void __launch_bounds__(FB_THREADS)
    fp8blk_requant_t_kernel(const uint8_t* __restrict__ codes,
                            const float* __restrict__ scales, int64_t M,
                            int64_t K, uint8_t* __restrict__ codes_t,
                            float* __restrict__ scales_t) {
  __shared__ __align__(16) uint8_t sm[128 * 256];
  const int64_t nti = M >> 7, ntj = K >> 7;
  const int64_t ntiles = nti * ntj;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cg = threadIdx.x & 15;                  // columns 8 cg .. + 7
  const int rg = threadIdx.x >> 4;                  // rows 8 rg .. + 7
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  const int mycol = (lane >> 2) & 7;                // column whose scales
  pdl_wait();                                       // this lane derives
  // the codes and scales of this thread's 8 rows of a tile; the next
  // tile's are loaded while the current one is quantized
  uint2 cv[8];
  float Sr[8];
  auto load_tile = [&](int64_t tile) {
    const int64_t ti = tile / ntj, tj = tile - ti * ntj;
    const int64_t ra = ti * 128 + 8 * rg;
    const uint8_t* src = codes + ra * K + tj * 128 + 8 * cg;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      Sr[i] = scales[(ra + i) * ntj + tj];
      cv[i] = ld_stream_v2(src + i * K);
    }
  };
  if ((int64_t)blockIdx.x < ntiles) load_tile(blockIdx.x);
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t ti = tile / ntj, tj = tile - ti * ntj;
    const int64_t r0 = ti * 128, c0 = tj * 128;
    // w[i][j]: row i, columns 2j and 2j + 1 (low half = column 2j)
    uint32_t w[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float a, b;
        e4m3x2_to_f32(((j < 2 ? cv[i].x : cv[i].y) >> ((j & 1) * 16)) & 0xFFFFu,
                      a, b);
        fmul2(a, b, Sr[i], Sr[i], a, b);
        w[i][j] = f32x2_to_bf16x2(a, b);
      }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int j = c >> 1;
      const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
      // column 8 cg + c, rows 8 rg .. 8 rg + 7 as four row pairs
      const uint4 col = make_uint4(__byte_perm(w[0][j], w[1][j], sel),
                                   __byte_perm(w[2][j], w[3][j], sel),
                                   __byte_perm(w[4][j], w[5][j], sel),
                                   __byte_perm(w[6][j], w[7][j], sel));
      *reinterpret_cast<uint4*>(&sm[rt_chunk(8 * cg + c, rg)]) = col;
    }
    if (tile + gridDim.x < ntiles) load_tile(tile + gridDim.x);
    __syncthreads();
#pragma unroll 1
    for (int q0 = 0; q0 < 16; q0 += 8) {
      const int cbase = warp * 16 + q0;
      uint2 v[8];
      uint32_t m[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        // rows 4 lane .. 4 lane + 3: half (lane & 1) of chunk lane / 2
        v[j] = *reinterpret_cast<const uint2*>(
            &sm[rt_chunk(cbase + j, lane >> 1) + (lane & 1) * 8]);
        m[j] = bf16x2_hmax(bf16x2_maxabs(v[j].x, v[j].y) & 0x7FFF7FFFu);
      }
      // reduce-scatter of the 8 column maxima (bf16 bit patterns of
      // non-negative values order like the values)
      uint32_t r4[4], r2[2], r1;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t send = b4 ? m[k] : m[k + 4];
        const uint32_t keep = b4 ? m[k + 4] : m[k];
        r4[k] = max(keep, __shfl_xor_sync(FULL, send, 16));
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t send = b3 ? r4[k] : r4[k + 2];
        const uint32_t keep = b3 ? r4[k + 2] : r4[k];
        r2[k] = max(keep, __shfl_xor_sync(FULL, send, 8));
      }
      {
        const uint32_t send = b2 ? r2[0] : r2[1];
        const uint32_t keep = b2 ? r2[1] : r2[0];
        r1 = max(keep, __shfl_xor_sync(FULL, send, 4));
      }
      r1 = max(r1, __shfl_xor_sync(FULL, r1, 2));
      r1 = max(r1, __shfl_xor_sync(FULL, r1, 1));
      float S2, enc;
      fb_scales(r1, S2, enc);
      if ((lane & 3) == 0) scales_t[(c0 + cbase + mycol) * nti + ti] = S2;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float ej = __shfl_sync(FULL, enc, 4 * j);
        const uint32_t word = bf16x2_scale_e4m3x2(v[j].x, ej, ej) |
                              (bf16x2_scale_e4m3x2(v[j].y, ej, ej) << 16);
        *reinterpret_cast<uint32_t*>(codes_t + (c0 + cbase + j) * M + r0 +
                                     4 * lane) = word;
      }
    }
    __syncthreads();                    // sm is rewritten by the next tile
  }
  pdl_launch_dependents();
}

unsigned fb_grid(int64_t work, int64_t per_cta, int dev, int ctas_per_sm) {
  int64_t g = (work + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)sm_count(dev) * ctas_per_sm;
  return (unsigned)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

cudaError_t launch_fp8blk_quantize(const void* x, int64_t rows, int64_t cols,
                                   int64_t ldx, int block_rows,
                                   uint8_t* codes, float* scales,
                                   cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  // every 16-value segment starts a multiple of 32 bytes from x
  const int wide = (reinterpret_cast<uintptr_t>(x) & 31u) == 0 && ldx % 16 == 0;
  if (block_rows == 1) {
    const int64_t ntiles = rows * (cols >> 7);
    const unsigned grid = fb_grid(ntiles, (FB_THREADS / 32) * 8, dev, 8);
    return launch_pdl(fp8blk_tile_kernel, dim3(grid), dim3(FB_THREADS), 0,
                      stream, false, xs, rows, cols, ldx, codes, scales, wide);
  }
  const int64_t nblk = (rows >> 7) * (cols >> 7);
  CUtensorMap tmap;
  err = make_tmap_2d_bf16(&tmap, x, (uint64_t)cols, (uint64_t)rows,
                          (uint64_t)ldx * 2, 128, 128, false);
  if (err != cudaSuccess) return err;
  const unsigned grid = fb_grid(nblk, 1, dev, FB_BLK_CTAS);
  return launch_pdl(fp8blk_block_kernel, dim3(grid), dim3(FB_THREADS), 0,
                    stream, false, tmap, rows, cols, codes, scales);
}

cudaError_t launch_fp8blk_dequantize(const uint8_t* codes, const float* scales,
                                     int64_t rows, int64_t cols,
                                     int block_rows, void* y,
                                     cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int64_t n16 = rows * (cols >> 4);
  // all 64 warps of an SM (8192 x 4096 tiles: 18.7 -> 18.3 us against 4 CTAs)
  const unsigned grid = fb_grid(n16, FB_THREADS, dev, 8);
  const int wide = (reinterpret_cast<uintptr_t>(y) & 31u) == 0;
  return launch_pdl(fp8blk_dequant_kernel, dim3(grid), dim3(FB_THREADS), 0,
                    stream, false, codes, scales, rows, cols,
                    block_rows == 1 ? 0 : 7, wide, static_cast<uint16_t*>(y));
}

cudaError_t fp8blk_take_wait_error(unsigned int* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_fp8blk_wait_error, sizeof(*word));
  if (e != cudaSuccess || *word == 0) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_fp8blk_wait_error, &zero, sizeof(zero));
}

cudaError_t launch_fp8blk_requant_t(const uint8_t* codes, const float* scales,
                                    int64_t M, int64_t K, uint8_t* codes_t,
                                    float* scales_t, cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int64_t ntiles = (M >> 7) * (K >> 7);
  // 4 resident CTAs per SM (63 registers x 256 threads)
  const unsigned grid = fb_grid(ntiles, 1, dev, 4);
  return launch_pdl(fp8blk_requant_t_kernel, dim3(grid), dim3(FB_THREADS), 0,
                    stream, false, codes, scales, M, K, codes_t, scales_t);
}

}  // namespace mxq
