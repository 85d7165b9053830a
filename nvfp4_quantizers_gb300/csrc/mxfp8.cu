// mxfp8.cu -- MXFP8 quantize, rowwise (1x32) and columnwise (32x1) copies
// produced in one pass over the bf16 input.
//
// "Miles: end-to-end MXFP8 and per-token NVFP4 RL", formats section: 32
// consecutive E4M3 values share one E8M0 power-of-two scale, rounded up so
// the block maximum is not clipped.  MXFP8 recipe section: the rowwise and
// columnwise blocks are quantized independently from the full-precision
// data and both copies are materialized by the same quantization.
//
// Design (sm_103a):
//  * Persistent CTAs, 2 per SM.  A producer warp streams 128x128 bf16
//    tiles (32 KB) into a 3-stage shared-memory ring with 2-D TMA
//    (cp.async.bulk.tensor), completion tracked by mbarriers.
//  * 8 consumer warps read each staged tile twice from shared memory:
//    rowwise, a lane owns 8 consecutive values of a row and 4 lanes form a
//    1x32 block (amax by two xor-shuffles); columnwise, a lane owns two
//    adjacent columns over 32 rows (amax on packed bf16x2), so the 32x1
//    blocks come from the same staged tile as the 1x32 ones.
//  * Row codes go out as 8-byte stores (a warp writes two full 128-byte
//    row segments); the columnwise copy is written transposed, 32
//    contiguous bytes per 32x1 block.
//  * A 128x128 tile owns exactly one 512-byte tile of the swizzled row
//    scales and one of the swizzled column scales; both are assembled in
//    shared memory and written out as one coalesced 512-byte store each
//    (padding entries come out as 0x00 because TMA fills out-of-range
//    elements with zeros and the scale of an all-zero block is 0x00).
#include "common.cuh"
#include "launch.h"

namespace mxq {

// Error word of the bounded mbarrier waits of this translation unit.
__device__ unsigned int g_mxfp8_wait_error = 0;

namespace {

constexpr int BM = 128;
constexpr int BK = 128;
constexpr int STAGES = 3;
constexpr int CONSUMER_WARPS = 8;
constexpr int THREADS = (CONSUMER_WARPS + 1) * 32;
constexpr uint32_t TILE_BYTES = BM * BK * 2;

struct alignas(1024) Smem {
  uint16_t tile[STAGES][BM * BK];
  alignas(16) uint8_t rscale[2][512];
  alignas(16) uint8_t cscale[2][512];
  alignas(8) uint64_t full[STAGES];
  alignas(8) uint64_t empty[STAGES];
  int abort;
};

struct Params {
  int64_t M, K;
  uint8_t* row_codes;
  uint8_t* row_scales;
  uint8_t* col_codes;
  uint8_t* col_scales;
  int do_row, do_col, swizzled;
  int64_t tiles_m, tiles_k, num_tiles;
};

// Position of logical scale (r, c), r < 128, c < 4, inside the staged
// 512-byte scale tile.
__device__ __forceinline__ int stage_pos(int r, int c, int swizzled) {
  return swizzled ? (r & 31) * 16 + (r >> 5) * 4 + c : r * 4 + c;
}

__global__ void __launch_bounds__(THREADS, 2)
    mxfp8_rowcol_kernel(const __grid_constant__ CUtensorMap tmap,
                        const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_addr(&s.full[i]), 1);
      mbar_init(smem_addr(&s.empty[i]), CONSUMER_WARPS);
    }
    s.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // ------------------------------------------------------------------ //
  // Producer warp: one lane issues the TMA loads.                       //
  // ------------------------------------------------------------------ //
  if (warp == CONSUMER_WARPS) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
        if (!mbar_wait(smem_addr(&s.empty[stage]), phase ^ 1, &s.abort,
                       &g_mxfp8_wait_error))
          break;
        const int64_t tm = t / p.tiles_k, tk = t - tm * p.tiles_k;
        const uint32_t full = smem_addr(&s.full[stage]);
        mbar_arrive_expect_tx(full, TILE_BYTES);
        tma_load_2d(smem_addr(s.tile[stage]), &tmap, (int32_t)(tk * BK),
                    (int32_t)(tm * BM), full);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    return;
  }

  // ------------------------------------------------------------------ //
  // Consumer warps.                                                     //
  // ------------------------------------------------------------------ //
  int stage = 0, par = 0;
  uint32_t phase = 0;
  for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
    const int64_t tm = t / p.tiles_k, tk = t - tm * p.tiles_k;
    const int64_t m0 = tm * BM, k0 = tk * BK;
    const int rows_valid = (int)imin<int64_t>(BM, p.M - m0);
    const int cols_valid = (int)imin<int64_t>(BK, p.K - k0);
    const bool ok = mbar_wait(smem_addr(&s.full[stage]), phase, &s.abort,
                             &g_mxfp8_wait_error);
    const uint16_t* tile = s.tile[stage];

    if (ok && p.do_row) {
      // 16 rows per warp, two rows per step; lane -> (row, 16-byte chunk).
      const int ch = lane & 15;
#pragma unroll 2
      for (int i = 0; i < 8; ++i) {
        const int r = warp * 16 + i * 2 + (lane >> 4);
        const uint4 v = *reinterpret_cast<const uint4*>(tile + r * BK + ch * 8);
        uint32_t m = bf16x2_max(bf16x2_absmax(v.x, v.y), bf16x2_absmax(v.z, v.w));
        uint32_t a = bf16x2_hmax(m);
        a = max(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = max(a, __shfl_xor_sync(0xffffffffu, a, 2));
        const uint32_t sbyte = e8m0_from_amax_bits(a);
        const float inv = e8m0_inv_scale(sbyte);
        const uint32_t w0 =
            cvt_e4m3x2(__fmul_rn(bf16lo_to_f32(v.x), inv),
                       __fmul_rn(bf16hi_to_f32(v.x), inv)) |
            (cvt_e4m3x2(__fmul_rn(bf16lo_to_f32(v.y), inv),
                        __fmul_rn(bf16hi_to_f32(v.y), inv)) << 16);
        const uint32_t w1 =
            cvt_e4m3x2(__fmul_rn(bf16lo_to_f32(v.z), inv),
                       __fmul_rn(bf16hi_to_f32(v.z), inv)) |
            (cvt_e4m3x2(__fmul_rn(bf16lo_to_f32(v.w), inv),
                        __fmul_rn(bf16hi_to_f32(v.w), inv)) << 16);
        if (r < rows_valid && ch * 8 < cols_valid)
          st_v2(p.row_codes + (m0 + r) * p.K + k0 + ch * 8, w0, w1);
        if ((lane & 3) == 0)
          s.rscale[par][stage_pos(r, ch >> 2, p.swizzled)] = (uint8_t)sbyte;
      }
    }

    if (ok && p.do_col) {
      // Warp -> 32-row block mb; lane -> columns c, c+1.
      const int mb = warp >> 1;
      const int c = (warp & 1) * 64 + lane * 2;
      uint32_t col[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        col[i] = *reinterpret_cast<const uint32_t*>(tile + (mb * 32 + i) * BK + c);
      uint32_t m = col[0] & 0x7FFF7FFFu;
#pragma unroll
      for (int i = 1; i < 32; ++i) m = bf16x2_absmax(m, col[i]);
      const uint32_t s_lo = e8m0_from_amax_bits(m & 0xFFFFu);
      const uint32_t s_hi = e8m0_from_amax_bits(m >> 16);
      const float inv_lo = e8m0_inv_scale(s_lo);
      const float inv_hi = e8m0_inv_scale(s_hi);
      uint32_t q_lo[8], q_hi[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t a0 = col[4 * j], a1 = col[4 * j + 1];
        const uint32_t a2 = col[4 * j + 2], a3 = col[4 * j + 3];
        q_lo[j] = cvt_e4m3x2(__fmul_rn(bf16lo_to_f32(a0), inv_lo),
                             __fmul_rn(bf16lo_to_f32(a1), inv_lo)) |
                  (cvt_e4m3x2(__fmul_rn(bf16lo_to_f32(a2), inv_lo),
                              __fmul_rn(bf16lo_to_f32(a3), inv_lo)) << 16);
        q_hi[j] = cvt_e4m3x2(__fmul_rn(bf16hi_to_f32(a0), inv_hi),
                             __fmul_rn(bf16hi_to_f32(a1), inv_hi)) |
                  (cvt_e4m3x2(__fmul_rn(bf16hi_to_f32(a2), inv_hi),
                              __fmul_rn(bf16hi_to_f32(a3), inv_hi)) << 16);
      }
      if (mb * 32 < rows_valid && c < cols_valid) {
        uint8_t* dst = p.col_codes + (k0 + c) * p.M + m0 + mb * 32;
        st_v4(dst, make_uint4(q_lo[0], q_lo[1], q_lo[2], q_lo[3]));
        st_v4(dst + 16, make_uint4(q_lo[4], q_lo[5], q_lo[6], q_lo[7]));
        dst += p.M;
        st_v4(dst, make_uint4(q_hi[0], q_hi[1], q_hi[2], q_hi[3]));
        st_v4(dst + 16, make_uint4(q_hi[4], q_hi[5], q_hi[6], q_hi[7]));
      }
      s.cscale[par][stage_pos(c, mb, p.swizzled)] = (uint8_t)s_lo;
      s.cscale[par][stage_pos(c + 1, mb, p.swizzled)] = (uint8_t)s_hi;
    }

    // Release the stage to the producer (all lanes' smem reads are done).
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&s.empty[stage]));
    // All scale bytes of this tile are staged.
    named_barrier_sync(1, CONSUMER_WARPS * 32);

    if (ok) {
      if (p.swizzled) {
        if (warp == 0 && p.do_row) {
          uint8_t* dst = p.row_scales + (tm * p.tiles_k + tk) * 512 + lane * 16;
          st_v4(dst, *reinterpret_cast<const uint4*>(&s.rscale[par][lane * 16]));
        } else if (warp == 1 && p.do_col) {
          uint8_t* dst = p.col_scales + (tk * p.tiles_m + tm) * 512 + lane * 16;
          st_v4(dst, *reinterpret_cast<const uint4*>(&s.cscale[par][lane * 16]));
        }
      } else {
        // Linear layout: warps 0-3 write the 4 row-scale bytes of one row,
        // warps 4-7 the 4 column-scale bytes of one column.
        const int idx = (warp & 3) * 32 + lane;
        if (warp < 4 && p.do_row && idx < rows_valid) {
          const int nblk = cols_valid >> 5;
          uint8_t* dst = p.row_scales + (m0 + idx) * (p.K >> 5) + (k0 >> 5);
          for (int b = 0; b < nblk; ++b) dst[b] = s.rscale[par][idx * 4 + b];
        } else if (warp >= 4 && p.do_col && idx < cols_valid) {
          const int nblk = rows_valid >> 5;
          uint8_t* dst = p.col_scales + (k0 + idx) * (p.M >> 5) + (m0 >> 5);
          for (int b = 0; b < nblk; ++b) dst[b] = s.cscale[par][idx * 4 + b];
        }
      }
    }
    if (++stage == STAGES) { stage = 0; phase ^= 1; }
    par ^= 1;
  }
}

}  // namespace

size_t mxfp8_rowcol_smem_bytes() { return sizeof(Smem) + 1024; }

cudaError_t mxfp8_take_wait_error(unsigned int* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_mxfp8_wait_error, sizeof(*word));
  if (e != cudaSuccess || *word == 0) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_mxfp8_wait_error, &zero, sizeof(zero));
}

cudaError_t launch_mxfp8_rowcol(const void* x, int64_t M, int64_t K,
                                int64_t ldx, uint8_t* row_codes,
                                uint8_t* row_scales, uint8_t* col_codes,
                                uint8_t* col_scales, int swizzled,
                                cudaStream_t stream) {
  CUtensorMap tmap;
  cudaError_t err = make_tmap_2d_bf16(&tmap, x, (uint64_t)K, (uint64_t)M,
                                      (uint64_t)ldx * 2, BK, BM);
  if (err != cudaSuccess) return err;
  Params p;
  p.M = M;
  p.K = K;
  p.row_codes = row_codes;
  p.row_scales = row_scales;
  p.col_codes = col_codes;
  p.col_scales = col_scales;
  p.do_row = row_codes != nullptr;
  p.do_col = col_codes != nullptr;
  p.swizzled = swizzled;
  p.tiles_m = (M + BM - 1) / BM;
  p.tiles_k = (K + BK - 1) / BK;
  p.num_tiles = p.tiles_m * p.tiles_k;

  const size_t smem = mxfp8_rowcol_smem_bytes();
  static thread_local int configured_dev = -1;
  int dev = 0;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (configured_dev != dev) {
    err = cudaFuncSetAttribute(mxfp8_rowcol_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess) return err;
    configured_dev = dev;
  }
  const int64_t grid = imin<int64_t>(p.num_tiles, (int64_t)sm_count(dev) * 2);
  mxfp8_rowcol_kernel<<<(unsigned)grid, THREADS, smem, stream>>>(tmap, p);
  return cudaGetLastError();
}

}  // namespace mxq
