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
// Design (sm_103a): pure streaming, grid-stride over 16-element units with
// eight 256-thread CTAs per SM.  A thread converts 16 values per unit: a
// 16-byte (MXFP8) or 8-byte (NVFP4) code load, one scale byte, and one
// 32-byte bf16 store.  The NVFP4 kernel takes two units per step, one grid
// stride apart, and issues both units' loads before the first conversion
// (one at a time left it waiting on load latency: the ragged 132106 x 2048
// batch 138 -> 108 us) while the work still splits evenly over the grid in
// single units; the MXFP8 kernel measured best one unit at a time.  The codes widen exactly through
// cvt.rn.f16x2.{e4m3x2,e2m1x2}; the scale multiply is one binary32
// multiply and the bf16 rounding one cvt.rn.bf16x2.f32.  Index math is
// 32-bit whenever every index fits.
#include "common.cuh"
#include "launch.h"

namespace mxq {

namespace {

constexpr int DQ_THREADS = 256;
// Eight CTAs per SM (all 64 warps; at most 48 registers a thread): with
// four, too few loads were in flight per SM (8192 x 4096 MXFP8 19.1 ->
// 17.5 us, 128 gate/up NVFP4 weights 187 -> 162 us with two units a step).
constexpr int DQ_CTAS_PER_SM = 8;
constexpr int DQ_UNROLL_MXFP8 = 1;         // units per thread per step
constexpr int DQ_UNROLL_NVFP4_ROW = 2;     // NVFP4, S per row
constexpr int DQ_UNROLL_NVFP4_BATCH = 2;   // NVFP4, S per weight group

// MXFP8: a thread converts 16 codes (one 16-byte load, half a 1x32 block)
// into 32 bytes of bf16 per step.  Idx is uint32_t when every index fits.
template <typename Idx, int DQ_UNROLL>
__global__ void __launch_bounds__(DQ_THREADS, DQ_CTAS_PER_SM)
    dequant_mxfp8_kernel(const uint8_t* __restrict__ codes,
                         const uint8_t* __restrict__ scales, Idx rows,
                         Idx cols, int swizzled, int wide,
                         uint16_t* __restrict__ y) {
  const Idx c16 = cols >> 4, nb = cols >> 5;
  const Idx n16 = rows * c16;
  const int64_t col_tiles = ((int64_t)nb + 3) >> 2;
  pdl_wait();
  const Idx stride = (Idx)gridDim.x * DQ_THREADS;
  for (Idx i0 = (Idx)blockIdx.x * DQ_THREADS + threadIdx.x; i0 < n16;
       i0 += stride * DQ_UNROLL) {
    uint4 c[DQ_UNROLL];
    uint32_t sbyte[DQ_UNROLL];
#pragma unroll
    for (int u = 0; u < DQ_UNROLL; ++u) {
      const Idx i = i0 + (Idx)u * stride;
      if (i < n16) {
        c[u] = ld_stream_v4(codes + (int64_t)i * 16);
        const Idx r = i / c16;
        const Idx b = (i - r * c16) >> 1;
        sbyte[u] = swizzled ? scales[swz_offset(r, b, col_tiles)]
                            : scales[(int64_t)r * nb + b];
      }
    }
#pragma unroll
    for (int u = 0; u < DQ_UNROLL; ++u) {
      const Idx i = i0 + (Idx)u * stride;
      if (i >= n16) break;
      const float sc = e8m0_scale(sbyte[u]);
      const uint32_t cw[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
      uint32_t w[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        float a, bb;
        e4m3x2_to_f32((cw[h >> 1] >> ((h & 1) * 16)) & 0xFFFFu, a, bb);
        fmul2(a, bb, sc, sc, a, bb);
        w[h] = f32x2_to_bf16x2(a, bb);
      }
      st_32B(y + (int64_t)i * 16, make_uint4(w[0], w[1], w[2], w[3]),
             make_uint4(w[4], w[5], w[6], w[7]), wide);
    }
  }
  pdl_launch_dependents();
}

// NVFP4: a thread converts one 16-value block (8 bytes of codes) into 32
// bytes of bf16 per step.  Rows are grouped in `batch` matrices of
// rows_per_batch rows, each with its own scale matrix (scale_stride bytes
// apart); S is per row (global row index) or per batch entry.
template <typename Idx, int DQ_UNROLL>
__global__ void __launch_bounds__(DQ_THREADS, DQ_CTAS_PER_SM)
    dequant_nvfp4_kernel(const uint8_t* __restrict__ codes,
                         const uint8_t* __restrict__ scales,
                         const float* __restrict__ S, int per_batch,
                         Idx rows_per_batch, Idx total_rows, Idx cols,
                         int swizzled, int64_t scale_stride, int wide,
                         uint16_t* __restrict__ y) {
  const Idx nb = cols >> 4;
  const Idx nblk = total_rows * nb;
  const int64_t col_tiles = ((int64_t)nb + 3) >> 2;
  const bool need_batch = swizzled || per_batch;
  pdl_wait();
  const Idx stride = (Idx)gridDim.x * DQ_THREADS;
  for (Idx i0 = (Idx)blockIdx.x * DQ_THREADS + threadIdx.x; i0 < nblk;
       i0 += stride * DQ_UNROLL) {
    uint2 c[DQ_UNROLL];
    uint32_t sbyte[DQ_UNROLL];
    float s32[DQ_UNROLL];
#pragma unroll
    for (int u = 0; u < DQ_UNROLL; ++u) {
      const Idx i = i0 + (Idx)u * stride;
      if (i < nblk) {
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                     : "=r"(c[u].x), "=r"(c[u].y)
                     : "l"(codes + (int64_t)i * 8));
        const Idx grow = i / nb;
        const Idx b = i - grow * nb;
        Idx bi = 0, r = grow;
        if (need_batch) {
          bi = grow / rows_per_batch;
          r = grow - bi * rows_per_batch;
        }
        sbyte[u] = swizzled ? scales[(int64_t)bi * scale_stride +
                                     swz_offset(r, b, col_tiles)]
                            : scales[(int64_t)grow * nb + b];
        s32[u] = per_batch ? S[bi] : S[grow];
      }
    }
#pragma unroll
    for (int u = 0; u < DQ_UNROLL; ++u) {
      const Idx i = i0 + (Idx)u * stride;
      if (i >= nblk) break;
      const float bs = e4m3_to_f32(sbyte[u]);
      uint32_t w[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        float a, bb;
        e2m1x2_to_f32((h < 4 ? c[u].x : c[u].y) >> (8 * (h & 3)), a, bb);
        fmul2(a, bb, bs, bs, a, bb);    // exact: at most 6 significant bits
        fmul2(a, bb, s32[u], s32[u], a, bb);
        w[h] = f32x2_to_bf16x2(a, bb);
      }
      st_32B(y + (int64_t)i * 16, make_uint4(w[0], w[1], w[2], w[3]),
             make_uint4(w[4], w[5], w[6], w[7]), wide);
    }
  }
  pdl_launch_dependents();
}

unsigned dq_grid(int64_t units, int dev) {
  int64_t g = (units + DQ_THREADS - 1) / DQ_THREADS;
  const int64_t cap = (int64_t)sm_count(dev) * DQ_CTAS_PER_SM;
  return (unsigned)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

cudaError_t launch_dequant_mxfp8(const uint8_t* codes, const uint8_t* scales,
                                 int64_t rows, int64_t cols, int swizzled,
                                 void* y, cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int64_t units = rows * (cols / 16);
  const unsigned grid = dq_grid(units, dev);
  uint16_t* out = static_cast<uint16_t*>(y);
  // a unit's 16 outputs are 32 bytes at a multiple of 32 bytes from y
  const int wide = (reinterpret_cast<uintptr_t>(y) & 31u) == 0;
  // 32-bit indices when the largest index and the grid stride fit.
  constexpr int U = DQ_UNROLL_MXFP8;
  if (units + (int64_t)grid * DQ_THREADS * U < (1ll << 32))
    return launch_pdl(dequant_mxfp8_kernel<uint32_t, U>, dim3(grid),
                      dim3(DQ_THREADS), 0, stream, false, codes, scales,
                      (uint32_t)rows, (uint32_t)cols, swizzled, wide, out);
  return launch_pdl(dequant_mxfp8_kernel<int64_t, U>, dim3(grid), dim3(DQ_THREADS),
                    0, stream, false, codes, scales, rows, cols, swizzled,
                    wide, out);
}

cudaError_t launch_dequant_nvfp4(const uint8_t* codes, const uint8_t* scales,
                                 const float* S, int per_batch, int64_t batch,
                                 int64_t rows, int64_t cols, int swizzled,
                                 void* y, cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int64_t total_rows = batch * rows;
  const int64_t units = total_rows * (cols / 16);
  const unsigned grid = dq_grid(units, dev);
  const int64_t stride = scale_bytes(rows, cols / 16, swizzled);
  uint16_t* out = static_cast<uint16_t*>(y);
  const int wide = (reinterpret_cast<uintptr_t>(y) & 31u) == 0;
  if (per_batch) {
    constexpr int U = DQ_UNROLL_NVFP4_BATCH;
    if (units + (int64_t)grid * DQ_THREADS * U < (1ll << 32))
      return launch_pdl(dequant_nvfp4_kernel<uint32_t, U>, dim3(grid),
                        dim3(DQ_THREADS), 0, stream, false, codes, scales, S,
                        per_batch, (uint32_t)rows, (uint32_t)total_rows,
                        (uint32_t)cols, swizzled, stride, wide, out);
    return launch_pdl(dequant_nvfp4_kernel<int64_t, U>, dim3(grid),
                      dim3(DQ_THREADS), 0, stream, false, codes, scales, S,
                      per_batch, rows, total_rows, cols, swizzled, stride,
                      wide, out);
  }
  constexpr int U = DQ_UNROLL_NVFP4_ROW;
  if (units + (int64_t)grid * DQ_THREADS * U < (1ll << 32))
    return launch_pdl(dequant_nvfp4_kernel<uint32_t, U>, dim3(grid),
                      dim3(DQ_THREADS), 0, stream, false, codes, scales, S,
                      per_batch, (uint32_t)rows, (uint32_t)total_rows,
                      (uint32_t)cols, swizzled, stride, wide, out);
  return launch_pdl(dequant_nvfp4_kernel<int64_t, U>, dim3(grid), dim3(DQ_THREADS),
                    0, stream, false, codes, scales, S, per_batch, rows,
                    total_rows, cols, swizzled, stride, wide, out);
}

}  // namespace mxq
