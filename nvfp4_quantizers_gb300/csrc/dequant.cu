// dequant.cu -- MXFP8 and NVFP4 dequantization to bf16.
//
// "Miles: end-to-end MXFP8 and per-token NVFP4 RL", backward-mode section:
// in dequantized-backward mode the BF16 backward GEMMs consume BF16
// dequantizations of the exact low-precision operands of the forward pass.
// "Using Quantization in RL", section "Two Ways to Configure Training and
// Inference": a stored value is interpreted as code x scale.
//
//   MXFP8: y = bf16_RNE( E4M3(c) * 2^(s - 127) )             (f32 product)
//   NVFP4: y = bf16_RNE( (E2M1(c) * E4M3(sb)) * S )          (f32 products,
//          the inner one exact)
//
// Design (sm_103a): pure streaming.  A thread converts 8 elements per step:
// an 8-byte (MXFP8) or 4-byte (NVFP4) code load and one 16-byte bf16 store,
// so a warp's loads and stores are both contiguous.  The codes widen
// exactly through cvt.rn.f16x2.{e4m3x2,e2m1x2}; the scale multiply is one
// binary32 multiply and the bf16 rounding one cvt.rn.bf16x2.f32.  The
// (row, column) of a thread's chunk is advanced incrementally across the
// grid-stride loop, so no per-element integer division is needed.
#include "common.cuh"
#include "launch.h"

namespace mxq {

namespace {

constexpr int DQ_THREADS = 256;
constexpr int DQ_UNROLL = 4;

// Coordinates (batch entry, row, column) of a thread's current 8-element
// chunk, advanced by a fixed grid stride with carries instead of divisions.
struct Cursor {
  int64_t bi, row, col;       // batch entry, row within it, column
  int64_t dbi, drow, dcol;    // advance per grid-stride step
  int64_t rows, cols;
  __device__ __forceinline__ void advance() {
    col += dcol;
    row += drow;
    bi += dbi;
    if (col >= cols) { col -= cols; row += 1; }
    if (row >= rows) { row -= rows; bi += 1; }
  }
};

__device__ __forceinline__ Cursor make_cursor(int64_t chunk, int64_t stride,
                                              int64_t rows, int64_t cols) {
  Cursor c;
  const int64_t e = chunk * 8, de = stride * 8;
  const int64_t grow = e / cols, dgrow = de / cols;
  c.col = e - grow * cols;
  c.dcol = de - dgrow * cols;
  c.bi = grow / rows;
  c.row = grow - c.bi * rows;
  c.dbi = dgrow / rows;
  c.drow = dgrow - c.dbi * rows;
  c.rows = rows;
  c.cols = cols;
  return c;
}

__global__ void __launch_bounds__(DQ_THREADS)
    dequant_mxfp8_kernel(const uint8_t* __restrict__ codes,
                         const uint8_t* __restrict__ scales, int64_t rows,
                         int64_t cols, int swizzled,
                         uint16_t* __restrict__ y) {
  const int64_t nchunks = rows * cols / 8;
  const int64_t stride = (int64_t)gridDim.x * DQ_THREADS;
  int64_t i = (int64_t)blockIdx.x * DQ_THREADS + threadIdx.x;
  if (i >= nchunks) return;
  Cursor cur = make_cursor(i, stride, rows, cols);
  const int64_t nb = cols >> 5, col_tiles = (nb + 3) >> 2;
  for (; i < nchunks; i += stride * DQ_UNROLL) {
    uint2 c[DQ_UNROLL];
    uint32_t sbyte[DQ_UNROLL];
    int64_t out[DQ_UNROLL];
    bool ok[DQ_UNROLL];
    Cursor k = cur;
#pragma unroll
    for (int u = 0; u < DQ_UNROLL; ++u) {
      const int64_t j = i + u * stride;
      ok[u] = j < nchunks;
      if (ok[u]) {
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                     : "=r"(c[u].x), "=r"(c[u].y)
                     : "l"(codes + j * 8));
        const int64_t b = k.col >> 5;
        sbyte[u] = swizzled ? scales[swz_offset(k.row, b, col_tiles)]
                            : scales[k.row * nb + b];
        out[u] = j * 8;
      }
      k.advance();
    }
    cur = k;
#pragma unroll
    for (int u = 0; u < DQ_UNROLL; ++u) {
      if (!ok[u]) continue;
      const float sc = e8m0_scale(sbyte[u]);
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint32_t two = ((h < 2 ? c[u].x : c[u].y) >> ((h & 1) * 16)) & 0xFFFFu;
        float a, b;
        e4m3x2_to_f32(two, a, b);
        w[h] = f32x2_to_bf16x2(__fmul_rn(a, sc), __fmul_rn(b, sc));
      }
      st_v4(y + out[u], make_uint4(w[0], w[1], w[2], w[3]));
    }
  }
}

__global__ void __launch_bounds__(DQ_THREADS)
    dequant_nvfp4_kernel(const uint8_t* __restrict__ codes,
                         const uint8_t* __restrict__ scales,
                         const float* __restrict__ S, int per_batch,
                         int64_t rows_per_batch, int64_t total_rows,
                         int64_t cols, int swizzled, int64_t scale_stride,
                         uint16_t* __restrict__ y) {
  const int64_t nchunks = total_rows * cols / 8;
  const int64_t stride = (int64_t)gridDim.x * DQ_THREADS;
  int64_t i = (int64_t)blockIdx.x * DQ_THREADS + threadIdx.x;
  if (i >= nchunks) return;
  Cursor cur = make_cursor(i, stride, rows_per_batch, cols);
  const int64_t nb = cols >> 4, col_tiles = (nb + 3) >> 2;
  for (; i < nchunks; i += stride * DQ_UNROLL) {
    uint32_t c[DQ_UNROLL];
    uint32_t sbyte[DQ_UNROLL];
    float s32[DQ_UNROLL];
    bool ok[DQ_UNROLL];
    Cursor k = cur;
#pragma unroll
    for (int u = 0; u < DQ_UNROLL; ++u) {
      const int64_t j = i + u * stride;
      ok[u] = j < nchunks;
      if (ok[u]) {
        asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];"
                     : "=r"(c[u])
                     : "l"(codes + j * 4));
        const int64_t b = k.col >> 4;
        const int64_t grow = k.bi * rows_per_batch + k.row;
        sbyte[u] = swizzled ? scales[k.bi * scale_stride +
                                     swz_offset(k.row, b, col_tiles)]
                            : scales[grow * nb + b];
        s32[u] = per_batch ? S[k.bi] : S[grow];
      }
      k.advance();
    }
    cur = k;
#pragma unroll
    for (int u = 0; u < DQ_UNROLL; ++u) {
      if (!ok[u]) continue;
      const float bs = e4m3_to_f32(sbyte[u]);
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float a, b;
        e2m1x2_to_f32(c[u] >> (8 * h), a, b);
        w[h] = f32x2_to_bf16x2(__fmul_rn(__fmul_rn(a, bs), s32[u]),
                               __fmul_rn(__fmul_rn(b, bs), s32[u]));
      }
      st_v4(y + (i + u * stride) * 8, make_uint4(w[0], w[1], w[2], w[3]));
    }
  }
}

int64_t dq_grid(int64_t nchunks, int dev) {
  const int64_t per_cta = (int64_t)DQ_THREADS * DQ_UNROLL;
  int64_t g = (nchunks + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)sm_count(dev) * 8;
  return g < 1 ? 1 : (g > cap ? cap : g);
}

}  // namespace

cudaError_t launch_dequant_mxfp8(const uint8_t* codes, const uint8_t* scales,
                                 int64_t rows, int64_t cols, int swizzled,
                                 void* y, cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int64_t nchunks = rows * cols / 8;
  dequant_mxfp8_kernel<<<(unsigned)dq_grid(nchunks, dev), DQ_THREADS, 0,
                         stream>>>(codes, scales, rows, cols, swizzled,
                                   static_cast<uint16_t*>(y));
  return cudaGetLastError();
}

cudaError_t launch_dequant_nvfp4(const uint8_t* codes, const uint8_t* scales,
                                 const float* S, int per_batch, int64_t batch,
                                 int64_t rows, int64_t cols, int swizzled,
                                 void* y, cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int64_t total_rows = batch * rows;
  const int64_t nchunks = total_rows * cols / 8;
  dequant_nvfp4_kernel<<<(unsigned)dq_grid(nchunks, dev), DQ_THREADS, 0,
                         stream>>>(codes, scales, S, per_batch, rows,
                                   total_rows, cols, swizzled,
                                   scale_bytes(rows, cols / 16, swizzled),
                                   static_cast<uint16_t*>(y));
  return cudaGetLastError();
}

}  // namespace mxq
