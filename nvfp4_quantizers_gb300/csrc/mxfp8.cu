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
//  * Persistent CTAs of 8 warps, 3 per SM.  128x128 bf16 tiles (32 KB)
//    stream into a 2-stage shared-memory ring per CTA with 2-D TMA
//    (cp.async.bulk.tensor), completion tracked by mbarriers; thread 0
//    refills a stage as soon as the tile's column codes, staged in it,
//    have left by their TMA store.
//  * Each tile arrives as two [128 x 64] halves with the 128-byte TMA
//    swizzle (16-byte chunk q of row r stored at chunk q ^ (r % 8)), which
//    makes both read patterns below free of shared-memory bank conflicts.
//  * 8 warps read each staged tile twice: rowwise, a lane owns whole 1x32
//    blocks; columnwise, a lane owns two adjacent columns over 32 rows
//    (amax on packed bf16x2), so the 32x1 blocks come from the same staged
//    tile as the 1x32 ones.  Warps read a block from the stage right before
//    converting it and hand the stage back after the tile, so a warp holds
//    one block's values at a time (78 registers): 24 warps per SM hide the
//    latency better than 16 warps that read the whole stage up front (128
//    registers, 2 CTAs of 3 stages: 27.0 -> 26.6 us per launch in the
//    step).
//  * Scaling uses packed f32x2 multiplies (exact: the scale is a power of
//    two); each 1x32 block's row codes are 32 contiguous bytes, written
//    with one 32-byte store (two 16-byte stores if the buffer is only
//    16-byte aligned): full-sector writes cut the kernel's time by a sixth
//    against 16-byte stores.  The column codes (the columnwise copy is
//    written transposed) go into the tile's own stage once every warp has
//    read it, and leave as one 128 x 128-byte TMA store: from registers
//    each lane's 32-byte runs landed in 64 different rows of X^T per warp
//    instruction.
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
constexpr int STAGES = 2;
constexpr int CONSUMER_WARPS = 8;
constexpr int THREADS = CONSUMER_WARPS * 32;
constexpr int HALF_COLS = 64;                 // one 128-byte swizzled TMA box
constexpr uint32_t TILE_BYTES = BM * BK * 2;

struct alignas(1024) Smem {
  uint16_t tile[STAGES][BM * BK];
  alignas(16) uint8_t rscale[2][512];
  alignas(16) uint8_t cscale[2][512];
  alignas(8) uint64_t full[STAGES];
  int abort;
};

struct Params {
  int64_t M, K;
  uint8_t* row_codes;
  uint8_t* row_scales;
  uint8_t* col_codes;
  uint8_t* col_scales;
  int do_row, do_col, swizzled;
  int wide;                 // code buffers 32-byte aligned: 32-byte stores
  uint32_t tiles_m, tiles_k, num_tiles;
};

// Element offset of (r, c) in a staged tile: two [128 x 64] halves of
// 128-byte rows loaded with the 128-byte TMA swizzle, which stores 16-byte
// chunk q of row r at chunk position q ^ (r % 8).
__device__ __forceinline__ int tile_off(int r, int c) {
  return (c >> 6) * (BM * HALF_COLS) + r * HALF_COLS +
         ((((c & 63) >> 3) ^ (r & 7)) << 3) + (c & 7);
}

// Position of logical scale (r, c), r < 128, c < 4, inside the staged
// 512-byte scale tile.
__device__ __forceinline__ int stage_pos(int r, int c, int swizzled) {
  return swizzled ? (r & 31) * 16 + (r >> 5) * 4 + c : r * 4 + c;
}

__global__ void __launch_bounds__(THREADS, 3)
    mxfp8_rowcol_kernel(const __grid_constant__ CUtensorMap tmap,
                        const __grid_constant__ CUtensorMap tmap_c,
                        const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) mbar_init(smem_addr(&s.full[i]), 1);
    s.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();

  // ------------------------------------------------------------------ //
  // Prologue: thread 0 fills the ring with the first STAGES tiles.      //
  // ------------------------------------------------------------------ //
  if (threadIdx.x == 0) {
    for (int st = 0; st < STAGES; ++st) {
      const uint32_t t = blockIdx.x + (uint32_t)st * gridDim.x;
      if (t >= p.num_tiles) break;
      const uint32_t tm = t / p.tiles_k, tk = t - tm * p.tiles_k;
      const uint32_t full = smem_addr(&s.full[st]);
      mbar_arrive_expect_tx(full, TILE_BYTES);
      tma_load_2d(smem_addr(s.tile[st]), &tmap, (int32_t)(tk * BK),
                  (int32_t)(tm * BM), full);
      tma_load_2d(smem_addr(s.tile[st] + BM * HALF_COLS), &tmap,
                  (int32_t)(tk * BK + HALF_COLS), (int32_t)(tm * BM), full);
    }
  }

  // ------------------------------------------------------------------ //
  // Consumer warps.                                                     //
  // ------------------------------------------------------------------ //
  int stage = 0, par = 0;
  uint32_t phase = 0;
  for (uint32_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
    const uint32_t tm = t / p.tiles_k, tk = t - tm * p.tiles_k;
    const int64_t m0 = (int64_t)tm * BM, k0 = (int64_t)tk * BK;
    const int rows_valid = (int)imin<int64_t>(BM, p.M - m0);
    const int cols_valid = (int)imin<int64_t>(BK, p.K - k0);
    const bool ok = mbar_wait_sleep(smem_addr(&s.full[stage]), phase, &s.abort,
                             &g_mxfp8_wait_error);
    const uint16_t* tile = s.tile[stage];

    // Read everything this warp needs from the staged tile first, then hand
    // the stage back so the next TMA load overlaps the conversions below.
    //   rows: warp w owns rows 16w..16w+15; lane -> rows 16w + lane%8 and
    //         16w + 8 + lane%8, 1x32 block lane/8.  The 8 lanes of a
    //         shared-memory phase read 8 consecutive rows of one block,
    //         which the 128-byte swizzle places in 8 different bank groups.
    //   cols: warp -> 32-row block mb; lane -> columns c, c+1 (packed); a
    //         warp reads one 128-byte swizzled row per step.
    const int rlane = lane & 7;
    const int rblk = lane >> 3;
    const int mb = warp >> 1;
    const int c = (warp & 1) * 64 + lane * 2;
    if (ok && p.do_row) {
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int r = warp * 16 + it * 8 + rlane;
        uint4 v[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          v[jj] = *reinterpret_cast<const uint4*>(tile + tile_off(r, rblk * 32 + jj * 8));
        const uint32_t m =
            bf16x2_maxabs(
                bf16x2_maxabs(bf16x2_maxabs(v[0].x, v[0].y),
                              bf16x2_maxabs(v[0].z, v[0].w)),
                bf16x2_maxabs(bf16x2_maxabs(v[1].x, v[1].y),
                              bf16x2_maxabs(v[1].z, v[1].w)));
        const uint32_t m2 =
            bf16x2_maxabs(
                bf16x2_maxabs(bf16x2_maxabs(v[2].x, v[2].y),
                              bf16x2_maxabs(v[2].z, v[2].w)),
                bf16x2_maxabs(bf16x2_maxabs(v[3].x, v[3].y),
                              bf16x2_maxabs(v[3].z, v[3].w)));
        const uint32_t a = bf16x2_hmax(bf16x2_maxabs(m, m2) & 0x7FFF7FFFu);
        const uint32_t sbyte = e8m0_from_amax_bits(a);
        const float inv = e8m0_inv_scale(sbyte);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          w[2 * j] = bf16x2_scale_e4m3x2(v[j].x, inv, inv) |
                     (bf16x2_scale_e4m3x2(v[j].y, inv, inv) << 16);
          w[2 * j + 1] = bf16x2_scale_e4m3x2(v[j].z, inv, inv) |
                         (bf16x2_scale_e4m3x2(v[j].w, inv, inv) << 16);
        }
        if (r < rows_valid && rblk * 32 < cols_valid) {
          uint8_t* dst = p.row_codes + (m0 + r) * p.K + k0 + rblk * 32;
          st_32B(dst, make_uint4(w[0], w[1], w[2], w[3]),
                 make_uint4(w[4], w[5], w[6], w[7]), p.wide);
        }
        s.rscale[par][stage_pos(r, rblk, p.swizzled)] = (uint8_t)sbyte;
      }
    }

    uint32_t q_lo[8], q_hi[8];            // this lane's two columns' codes
    if (ok && p.do_col) {
      uint32_t col[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        col[i] = *reinterpret_cast<const uint32_t*>(tile + tile_off(mb * 32 + i, c));
      // amax over the 32 rows as four independent chains.
      uint32_t m0r = bf16x2_maxabs(col[0], col[1]);
      uint32_t m1r = bf16x2_maxabs(col[2], col[3]);
      uint32_t m2r = bf16x2_maxabs(col[4], col[5]);
      uint32_t m3r = bf16x2_maxabs(col[6], col[7]);
#pragma unroll
      for (int i = 8; i < 32; i += 8) {
        m0r = bf16x2_maxabs(m0r, bf16x2_maxabs(col[i], col[i + 1]));
        m1r = bf16x2_maxabs(m1r, bf16x2_maxabs(col[i + 2], col[i + 3]));
        m2r = bf16x2_maxabs(m2r, bf16x2_maxabs(col[i + 4], col[i + 5]));
        m3r = bf16x2_maxabs(m3r, bf16x2_maxabs(col[i + 6], col[i + 7]));
      }
      const uint32_t m = bf16x2_maxabs(bf16x2_maxabs(m0r, m1r),
                                       bf16x2_maxabs(m2r, m3r)) & 0x7FFF7FFFu;
      const uint32_t s_lo = e8m0_from_amax_bits(m & 0xFFFFu);
      const uint32_t s_hi = e8m0_from_amax_bits(m >> 16);
      const float inv_lo = e8m0_inv_scale(s_lo);
      const float inv_hi = e8m0_inv_scale(s_hi);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float l0, l1, l2, l3, h0, h1, h2, h3;
        fmul2(bf16lo_to_f32(col[4 * j]), bf16lo_to_f32(col[4 * j + 1]), inv_lo,
              inv_lo, l0, l1);
        fmul2(bf16lo_to_f32(col[4 * j + 2]), bf16lo_to_f32(col[4 * j + 3]),
              inv_lo, inv_lo, l2, l3);
        fmul2(bf16hi_to_f32(col[4 * j]), bf16hi_to_f32(col[4 * j + 1]), inv_hi,
              inv_hi, h0, h1);
        fmul2(bf16hi_to_f32(col[4 * j + 2]), bf16hi_to_f32(col[4 * j + 3]),
              inv_hi, inv_hi, h2, h3);
        q_lo[j] = cvt_e4m3x2(l0, l1) | (cvt_e4m3x2(l2, l3) << 16);
        q_hi[j] = cvt_e4m3x2(h0, h1) | (cvt_e4m3x2(h2, h3) << 16);
      }
      s.cscale[par][stage_pos(c, mb, p.swizzled)] = (uint8_t)s_lo;
      s.cscale[par][stage_pos(c + 1, mb, p.swizzled)] = (uint8_t)s_hi;
    }
    // Every warp must be done reading the tile before its stage takes the
    // tile's column codes: [128 columns x 128 rows] bytes, column c's
    // 32-byte run of block mb at bytes 32 mb of row c, in the 128-byte
    // swizzle of the store's tensor map (16-byte chunk q of row r at
    // q ^ (r % 8)); one TMA store then writes the whole tile.
    if (p.do_col) named_barrier_sync(2, CONSUMER_WARPS * 32);  // uniform
    if (ok && p.do_col) {
      uint8_t* cst = reinterpret_cast<uint8_t*>(s.tile[stage]);
      const int q0 = 2 * mb;
      *reinterpret_cast<uint4*>(cst + c * 128 + ((q0 ^ (c & 7)) << 4)) =
          make_uint4(q_lo[0], q_lo[1], q_lo[2], q_lo[3]);
      *reinterpret_cast<uint4*>(cst + c * 128 + (((q0 + 1) ^ (c & 7)) << 4)) =
          make_uint4(q_lo[4], q_lo[5], q_lo[6], q_lo[7]);
      *reinterpret_cast<uint4*>(cst + (c + 1) * 128 + ((q0 ^ ((c + 1) & 7)) << 4)) =
          make_uint4(q_hi[0], q_hi[1], q_hi[2], q_hi[3]);
      *reinterpret_cast<uint4*>(cst + (c + 1) * 128 +
                                (((q0 + 1) ^ ((c + 1) & 7)) << 4)) =
          make_uint4(q_hi[4], q_hi[5], q_hi[6], q_hi[7]);
      fence_proxy_async_smem();
    }

    // All scale bytes (and the column codes) of this tile are staged.
    named_barrier_sync(1, CONSUMER_WARPS * 32);
    // Thread 0: the column codes leave by one TMA store (rows and columns
    // past M and K are clipped by the tensor map); once the store has read
    // the stage, the tile STAGES iterations ahead is loaded into it.
    if (threadIdx.x == 0) {
      if (ok && p.do_col) {
        tma_store_2d(&tmap_c, smem_addr(s.tile[stage]), (int32_t)m0,
                     (int32_t)k0);
        bulk_commit();
        bulk_wait_read_0();
      }
      const uint32_t next = t + (uint32_t)STAGES * gridDim.x;
      if (next < p.num_tiles && !s.abort) {
        const uint32_t nm = next / p.tiles_k, nk = next - nm * p.tiles_k;
        const uint32_t full = smem_addr(&s.full[stage]);
        mbar_arrive_expect_tx(full, TILE_BYTES);
        tma_load_2d(smem_addr(s.tile[stage]), &tmap, (int32_t)(nk * BK),
                    (int32_t)(nm * BM), full);
        tma_load_2d(smem_addr(s.tile[stage] + BM * HALF_COLS), &tmap,
                    (int32_t)(nk * BK + HALF_COLS), (int32_t)(nm * BM), full);
      }
    }

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
  if (threadIdx.x == 0) bulk_wait_all();
  pdl_launch_dependents();
}

// Failure-detection self-test: thread 0 waits on an mbarrier that nothing
// will ever complete, through the same bounded wait the kernels use, with a
// short limit; the wait gives up, records the error word and returns.
__global__ void wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait(smem_addr(&bar), 0, &abort, &g_mxfp8_wait_error, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

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
                                      (uint64_t)ldx * 2, HALF_COLS, BM, true);
  if (err != cudaSuccess) return err;
  // the columnwise codes X^T [K x M], stored by 128 x 128-byte boxes
  CUtensorMap tmap_c;
  if (col_codes) {
    err = make_tmap_2d_bytes(&tmap_c, col_codes, (uint64_t)M, (uint64_t)K,
                             (uint64_t)M, BM, BK);
    if (err != cudaSuccess) return err;
  } else {
    tmap_c = tmap;                      // unused
  }
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
  // Every 32-byte code run starts at a multiple of 32 bytes from its
  // buffer (K and M are multiples of 32).
  p.wide = ((reinterpret_cast<uintptr_t>(row_codes) |
             reinterpret_cast<uintptr_t>(col_codes)) & 31u) == 0;
  p.tiles_m = (uint32_t)((M + BM - 1) / BM);
  p.tiles_k = (uint32_t)((K + BK - 1) / BK);
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
  const int64_t grid = imin<int64_t>((int64_t)p.num_tiles, (int64_t)sm_count(dev) * 3);
  return launch_pdl(mxfp8_rowcol_kernel, dim3((unsigned)grid), dim3(THREADS),
                    smem, stream, false, tmap, tmap_c, p);
}

}  // namespace mxq
