// gemm.cu -- block-scaled GEMM consumers of the quantizer outputs, on the
// 5th-generation tensor cores (tcgen05, sm_103a).
//
// "Miles: end-to-end MXFP8 and per-token NVFP4 RL", MXFP8 recipe section:
// forward, weight-gradient and data-gradient GEMMs consume the MXFP8
// copies; experiments section: the per-token NVFP4 GEMM applies the
// per-token FP32 scale in the kernel epilogue instead of a separate op.
//
//   MXFP8:  C[m, n] = sum_k A[m, k] * B[k, n], A given rowwise (1x32 E8M0
//           blocks along K) and B given as B^T [N x K] (its columnwise
//           copy, also 1x32 blocks along K); fp32 accumulation and output.
//   NVFP4:  grouped over experts: rows off[e] .. off[e+1] of A use expert
//           e's weight W_e [N x K]; C[r, n] = S_tok[r] * S_w[e] *
//           sum_k a[r, k] w_e[n, k], where a and w are E2M1 x E4M3 block
//           values and the two FP32 scales are applied in the epilogue.
//
// Design (persistent, one CTA per SM, 128 x 256 fp32 output tiles, 11
// warps, one accumulator):
//  * warp 0 lane 0 streams K-stages of 128 bytes per row into a 4-deep
//    shared-memory ring (48 KiB of operands a stage; the MMA waits on
//    operand delivery, so the ring takes all shared memory): the A (128 rows) and B (256 rows) code tiles by
//    2-D TMA with the 128-byte swizzle, and the matching 512-byte scale
//    tiles, which the quantizers already store in the 128x4 layout the
//    tensor core reads, by one 1-D bulk copy per 128-row block; completion
//    on mbarriers.  Every CTA loads its own operands (no clusters).
//  * warp 2 polls the stage and accumulator barriers and hands each ready
//    stage to warp 1 through a named barrier, so that the MMA-issuing
//    thread never waits on shared memory between MMAs;
//  * warp 1 lane 0 copies each stage's scale tiles into tensor memory
//    (tcgen05.cp 32x128b.warpx4) and issues the block-scaled MMAs
//    (tcgen05.mma kind::mxf8f6f4 block_scale, or kind::mxf4nvf4 with
//    4 E4M3 scales per 64 values, N = 256); the 128 x 256 fp32 accumulator
//    lives in tensor memory; tcgen05.commit frees each stage when its MMAs
//    are done and hands each finished accumulator to the epilogue.
//  * warps 3-10 (4 lane quarters x 2 column halves) take the accumulator
//    into registers (128 values per thread) and release it at once, so the
//    next tile's MMAs overlap the scaling (NVFP4: S_tok x S_w) and the
//    stores; each thread writes its row's values straight from registers
//    with 32-byte stores (whole sectors).  Staging boxes for TMA stores
//    would cost the fourth stage (grouped NVFP4 124.0 -> 118.8 us with
//    four stages and direct stores, MXFP8 unchanged).
// Every wait is bounded; on timeout the kernel records the error word and
// skips the remaining work (still freeing its tensor memory).
#include "common.cuh"
#include "launch.h"

namespace mxq {

__device__ unsigned int g_gemm_wait_error = 0;

namespace {

constexpr int GM = 128;              // tile rows (A) = MMA M
constexpr int GN = 256;              // tile cols (B rows) = MMA N
constexpr int GKB = 128;             // bytes of K per stage per row
constexpr int GSTAGES = 4;
constexpr int kEpiWarps = 8;         // 4 lane quarters x 2 column halves
constexpr int kSfWarp = 3 + kEpiWarps;  // gathers A's block scales (gather mode)
// producer, MMA, waiter, epilogue, scale gatherer
constexpr int GTHREADS = 32 * (4 + kEpiWarps);
constexpr uint32_t kTmemCols = 512;  // accumulator 256 + scale columns
constexpr uint32_t kSfCol0 = 256;    // 64 scale columns per stage
constexpr uint32_t kSfColsPerStage = 64;

struct alignas(1024) GemmSmem {
  uint8_t a[GSTAGES][GM * GKB];
  uint8_t b[GSTAGES][GN * GKB];
  // scale tiles of the stage: A [tile j], B [128-row block][tile j]
  alignas(16) uint8_t sfa[GSTAGES][4][512];
  alignas(16) uint8_t sfb[GSTAGES][2][4][512];
  alignas(8) uint64_t full[GSTAGES];
  alignas(8) uint64_t empty[GSTAGES];
  alignas(8) uint64_t acc_full;
  alignas(8) uint64_t acc_empty;
  uint32_t tmem_base;
  int abort;
};

// ---------------------------------------------------------------------------
// tcgen05 / bulk-copy wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          dst_smem),
      "r"(ncols)
      : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                   taddr),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(bar)
      : "memory");
}
// 32 rows x 128 bits of shared memory (32 x 16 bytes, a 512-byte scale tile)
// into tensor memory, replicated to the four 32-lane quarters.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr),
               "l"(sdesc)
               : "memory");
}
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d, uint64_t adesc,
                                            uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d, uint64_t adesc,
                                            uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns of tensor memory -> registers
// (completion: tc_wait_ld).
__device__ __forceinline__ void tc_ld_32x32_async(uint32_t taddr,
                                                  uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, "
      "%7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, "
      "%21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Stage handoff between the waiter warp and the MMA warp: both warps
// (converged) meet at named barrier 1; the result is the OR of the abort
// flags the two warps bring.
__device__ __forceinline__ bool stage_handoff(bool abort_in) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, 64, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)abort_in)
      : "memory");
  return r != 0;
}

// 2-D tiled TMA gather of four rows (rows y0..y3, the box's columns from
// x) into four consecutive box-sized rows of shared memory, completion on
// `bar`.  The tensor map's box is one row high.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map,
                                            int32_t x, int32_t y0, int32_t y1,
                                            int32_t y2, int32_t y3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::"
      "complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2),
      "r"(y3), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor (sm_100 family): start address, leading
// and stride byte offsets (all >> 4), version 1 at bit 46, layout type at
// bits 61-63 (0 = no swizzle, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo,
                                              uint32_t sbo, uint32_t layout) {
  return (uint64_t)((addr >> 4) & 0x3FFF) |
         ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) |
         ((uint64_t)layout << 61);
}

// Instruction descriptor of a block-scaled MMA, M = 128, N = GN, both
// operands K-major: format codes a_fmt / b_fmt, scale format (1 = E8M0,
// 0 = E4M3), and the byte of each 32-bit scale cell to use (sf_id).
__device__ __forceinline__ uint32_t idesc_block_scaled(uint32_t a_fmt,
                                                       uint32_t b_fmt,
                                                       uint32_t sf_e8m0,
                                                       uint32_t sf_id) {
  return (sf_id << 4) | (a_fmt << 7) | (b_fmt << 10) |
         ((uint32_t)(GN >> 3) << 17) | (sf_e8m0 << 23) |
         ((uint32_t)(GM >> 4) << 24) | (sf_id << 29);
}

struct GemmParams {
  // tile -> operands
  int kind;                 // 0 = MXFP8, 1 = NVFP4 grouped
  int64_t M, N, K;          // K in elements
  int64_t k_stages;         // K / elements per stage
  const uint8_t* a_sf;      // swizzled scales of A
  const uint8_t* b_sf;      // swizzled scales of B (group 0)
  int64_t a_sf_ct;          // scale tiles per 128 rows of A (= K / 128 or K / 64)
  int64_t b_sf_ct;
  int64_t b_sf_group_stride;   // bytes between the scale matrices of groups
  int64_t b_rows_group_stride; // rows between the groups' weights in the B map
  // NVFP4 grouped
  // Gather mode (row_index != NULL): routed row r of A is row row_index[r]
  // of the per-token operand (codes through the A tensor map, block scales
  // in the linear layout at a_sf_lin, a_sf_ld bytes per row, S_tok per
  // source row); an index outside [0, T_src) is a padding row (zero block
  // scales and S_tok, so it contributes 0).
  const int32_t* row_index;
  int64_t T_src;
  const uint8_t* a_sf_lin;
  int64_t a_sf_ld;
  const float* s_tok;
  const float* s_w;
  int num_groups;
  int64_t tile_end[257];    // prefix sums of the M-tiles of each group
  int64_t row_off[257];     // first row of each group
  int64_t tiles_n;
  int64_t n_tiles;
  int64_t tile_cols;        // output columns per tile: 256, or 128 (SwiGLU)
  int64_t b_up_row;         // SwiGLU: row of the up half in a group's weights
  float* C;                 // fp32 C (EPI 0)
  uint16_t* H;              // bf16 h (EPI 1)
  int64_t ldc;              // row stride of C or h, elements
  int c_wide;               // rows 32-byte aligned: 32-byte stores
};

struct Tile {
  int64_t m0, n0;
  int grp;
};

// Tile index -> operand coordinates.  Each thread visits its tiles in
// increasing order, so the group is found by advancing a cursor (*grp)
// that the caller keeps across calls, instead of scanning from group 0.
__device__ __forceinline__ Tile decode_tile(const GemmParams& p, int64_t tile,
                                            int* grp) {
  const int64_t mt_all = tile / p.tiles_n;
  const int64_t nt = tile - mt_all * p.tiles_n;
  Tile t;
  if (p.kind == 1)
    while (*grp + 1 < p.num_groups && mt_all >= p.tile_end[*grp]) ++*grp;
  t.grp = *grp;
  const int64_t mt_in =
      p.kind == 1 ? mt_all - (t.grp ? p.tile_end[t.grp - 1] : 0) : mt_all;
  t.m0 = (p.kind == 1 ? p.row_off[t.grp] : 0) + mt_in * GM;
  t.n0 = nt * p.tile_cols;
  return t;
}

// Persistent: CTA b handles tiles b, b + grid, b + 2 grid, ...
//
// One 128 x 256 fp32 accumulator in tensor memory.  The eight epilogue
// warps copy it to registers (128 values per thread) and hand it back to
// the MMA warp at once, then scale and store while the next tile's MMAs
// already run.
//
// EPI = 0: C tile = the 128 x 256 accumulator (x S_tok x S_w for NVFP4),
// fp32.  EPI = 1 (SwiGLU, NVFP4 gate/up weights [gate ; up] per group): the
// B stage holds 128 gate rows and the 128 matching up rows, so one tile
// gives 128 output columns h = silu(s g) * (s u), s = S_tok x S_w, bf16
// (binary32 with a fast exponential and divide before the bf16 rounding).
template <int EPI>
__global__ void __launch_bounds__(GTHREADS, 1)
    gemm_block_scaled_kernel(const __grid_constant__ CUtensorMap tmap_a,
                             const __grid_constant__ CUtensorMap tmap_b,
                             const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t gsmem_raw[];
  GemmSmem& s = *reinterpret_cast<GemmSmem*>(
      (reinterpret_cast<uintptr_t>(gsmem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0) tmem_alloc(smem_addr(&s.tmem_base), kTmemCols);
  if (threadIdx.x == 0) {
    for (int i = 0; i < GSTAGES; ++i) {
      // the producer's arrive (+ the scale gatherer's in gather mode)
      mbar_init(smem_addr(&s.full[i]), p.row_index ? 2 : 1);
      mbar_init(smem_addr(&s.empty[i]), 1);   // freed by the MMA commit
    }
    mbar_init(smem_addr(&s.acc_full), 1);
    mbar_init(smem_addr(&s.acc_empty), kEpiWarps);
    s.abort = 0;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int64_t n_units = p.n_tiles;
  const int64_t unit0 = blockIdx.x, unit_step = gridDim.x;
  pdl_wait();

  const int n_sf = p.kind == 1 ? 4 : 1;  // scale tiles per stage and row block

  if (warp == 0) {
    // ---------------- producer ----------------
    // Lane 0 waits for free stages and issues the copies.  In gather mode
    // every lane holds four of the tile's source rows (rows 4 lane ..
    // 4 lane + 3) and issues their gather4 load itself (one lane issuing
    // all 32, with the indices passed by shuffles, took longer per stage
    // than the stage's MMAs).
    int64_t it = 0;
    int grp_cursor = 0, pf_cursor = 0;
    bool ok = true;
    // the gather rows of a tile: loaded one tile ahead, so that their
    // latency is not on the path of the tile's first stage
    int32_t nxt[4] = {0, 0, 0, 0};
    auto load_rows = [&](int64_t u, int32_t (&dst)[4]) {
      if (!p.row_index || u >= n_units) return;
      const Tile tt = decode_tile(p, u, &pf_cursor);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        dst[k] = p.row_index[tt.m0 + 4 * lane + k];
    };
    load_rows(unit0, nxt);
    for (int64_t u = unit0; u < n_units && ok; u += unit_step) {
      const Tile t = decode_tile(p, u, &grp_cursor);
      int32_t src[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)                    // padding: any real row
        src[k] = (nxt[k] >= 0 && nxt[k] < p.T_src) ? nxt[k] : 0;
      load_rows(u + unit_step, nxt);
      // B row blocks of this tile that exist (the last column tile may
      // hold only 128 columns); rows past them are never stored.
      const int nrb = (EPI == 1 || t.n0 + 128 < p.N) ? 2 : 1;
      const uint32_t stage_bytes = (uint32_t)(
          GM * GKB + GN * GKB + 512 * n_sf * ((p.row_index ? 0 : 1) + nrb));
      for (int64_t kt = 0; kt < p.k_stages; ++kt, ++it) {
        const int st = (int)(it % GSTAGES);
        const uint32_t ph = (uint32_t)((it / GSTAGES) & 1);
        if (lane == 0)
          ok = mbar_wait(smem_addr(&s.empty[st]), ph ^ 1, &s.abort,
                         &g_gemm_wait_error);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t full = smem_addr(&s.full[st]);
        if (lane == 0) {
          mbar_arrive_expect_tx(full, stage_bytes);
          if (!p.row_index)
            tma_load_2d(smem_addr(s.a[st]), &tmap_a, (int32_t)(kt * GKB),
                        (int32_t)t.m0, full);
          const int64_t brow = t.grp * p.b_rows_group_stride + t.n0;
          if (EPI == 0) {
            tma_load_2d(smem_addr(s.b[st]), &tmap_b, (int32_t)(kt * GKB),
                        (int32_t)brow, full);
          } else {
            // gate rows n0.. and up rows up_row + n0.. (128-row boxes)
            tma_load_2d(smem_addr(s.b[st]), &tmap_b, (int32_t)(kt * GKB),
                        (int32_t)brow, full);
            tma_load_2d(smem_addr(s.b[st]) + 128 * GKB, &tmap_b,
                        (int32_t)(kt * GKB), (int32_t)(brow + p.b_up_row),
                        full);
          }
          // The stage's n_sf scale tiles of one 128-row block are
          // consecutive in the swizzled layout: one copy per row block.
          const int64_t ct = kt * n_sf;
          if (!p.row_index)
            bulk_g2s(smem_addr(s.sfa[st][0]),
                     p.a_sf + ((t.m0 / 128) * p.a_sf_ct + ct) * 512,
                     512u * n_sf, full);
          for (int rb = 0; rb < nrb; ++rb) {
            const int64_t rblk =
                EPI == 0 ? t.n0 / 128 + rb : (t.n0 + rb * p.b_up_row) / 128;
            bulk_g2s(smem_addr(s.sfb[st][rb][0]),
                     p.b_sf + t.grp * p.b_sf_group_stride +
                         (rblk * p.b_sf_ct + ct) * 512,
                     512u * n_sf, full);
          }
        }
        if (p.row_index) {
          // the A stage: every lane gathers its 4 routed rows (128 bytes of
          // K each) into rows 4 lane .. 4 lane + 3 of the 128-byte-swizzled
          // tile the MMA reads, once lane 0 has set the stage's byte count
          __syncwarp();
          tma_gather4(smem_addr(s.a[st]) + lane * 4 * GKB, &tmap_a,
                      (int32_t)(kt * GKB), src[0], src[1], src[2], src[3],
                      full);
        }
      }
      if (s.abort) break;
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // The issuing thread touches no shared memory between MMAs: while the
    // tensor core streams operands out of shared memory, an mbarrier poll
    // from this thread stalls behind those reads and the MMA queue runs
    // dry.  The waiter warp polls instead and hands each ready stage over
    // through a named barrier, which carries the abort flag as well.
    int64_t it = 0;
    bool aborted = false;
    for (int64_t u = unit0; u < n_units && !aborted; u += unit_step) {
      for (int64_t kt = 0; kt < p.k_stages; ++kt, ++it) {
        __syncwarp();
        if (stage_handoff(false)) {
          aborted = true;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const int st = (int)(it % GSTAGES);
          // Scale columns of the stage: A tile j at 4j, B (row block rb,
          // tile j) at 16 + 8j + 4rb.  Scale columns of a B row block the
          // tile does not have keep stale values; they only feed output
          // columns that are never stored.
          const uint32_t sf_col =
              tmem + kSfCol0 + (uint32_t)st * kSfColsPerStage;
          for (int j = 0; j < n_sf; ++j) {
            tc_cp_sf(sf_col + j * 4,
                     smem_desc(smem_addr(s.sfa[st][j]), 16, 128, 0));
            for (int rb = 0; rb < 2; ++rb)
              tc_cp_sf(sf_col + 16 + j * 8 + rb * 4,
                       smem_desc(smem_addr(s.sfb[st][rb][j]), 16, 128, 0));
          }
          const uint32_t a_addr = smem_addr(s.a[st]);
          const uint32_t b_addr = smem_addr(s.b[st]);
          // Four MMAs per stage, each 32 bytes of K further along the
          // 128-byte swizzled rows.
          for (int j = 0; j < 4; ++j) {
            const uint64_t ad = smem_desc(a_addr + j * 32, 16, 1024, 2);
            const uint64_t bd = smem_desc(b_addr + j * 32, 16, 1024, 2);
            const uint32_t acc = (kt > 0 || j > 0) ? 1u : 0u;
            if (p.kind == 0) {
              // 8-bit operands: K = 32 per MMA, one E8M0 scale per row per
              // MMA: byte j of the stage's 32-bit scale cell.
              tc_mma_mxf8(tmem, ad, bd,
                          idesc_block_scaled(0, 0, 1, (uint32_t)j), sf_col,
                          sf_col + 16, acc);
            } else {
              // 4-bit operands: K = 64 per MMA, four E4M3 scales per row (one
              // 32-bit cell = scale tile j).
              tc_mma_nvf4(tmem, ad, bd, idesc_block_scaled(1, 1, 0, 0),
                          sf_col + j * 4, sf_col + 16 + j * 8, acc);
            }
          }
          tc_commit(smem_addr(&s.empty[st]));
          if (kt == p.k_stages - 1) tc_commit(smem_addr(&s.acc_full));
        }
      }
    }
  } else if (warp == 2) {
    // ---------------- waiter ----------------
    // Mirrors the issuer's loop: before a tile's first stage it waits until
    // the epilogue has taken the accumulator, before every stage until the
    // stage's operands have landed; then one handoff.
    int64_t it = 0;
    int local = 0;
    bool ok = true;
    for (int64_t u = unit0; u < n_units && ok; u += unit_step, ++local) {
      if (lane == 0)
        ok = mbar_wait(smem_addr(&s.acc_empty), (uint32_t)((local & 1) ^ 1),
                       &s.abort, &g_gemm_wait_error);
      for (int64_t kt = 0; kt < p.k_stages; ++kt, ++it) {
        const int st = (int)(it % GSTAGES);
        const uint32_t ph = (uint32_t)((it / GSTAGES) & 1);
        if (lane == 0 && ok)
          ok = mbar_wait(smem_addr(&s.full[st]), ph, &s.abort,
                         &g_gemm_wait_error);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        if (stage_handoff(!ok)) {
          ok = false;
          break;
        }
      }
    }
  } else if (warp == kSfWarp) {
    // ---------------- scale gatherer (gather mode) ----------------
    // Lane l holds the tile's routed rows l + 32 j: each stage it loads
    // their 16 block scales of the stage (linear layout: 16 contiguous
    // bytes of the source row, four 4-column scale tiles) before waiting
    // for the slot, then writes each 4-byte word to its place in the
    // 128x4 tile layout the tensor core reads, (r % 32) * 16 + (r / 32) * 4,
    // fences the writes to the async proxy and arrives on the stage.
    if (p.row_index) {
      // Stages in the order the producer fills them: stage it is k-stage
      // it % k_stages of this CTA's tile it / k_stages.  Scale words are
      // loaded D stages ahead into two static register buffers, and a
      // tile's source rows one tile ahead of their first use.
      const int64_t n_my = n_units > unit0 ? (n_units - unit0 + unit_step - 1) / unit_step : 0;
      const int64_t total = n_my * p.k_stages;
      const int D = p.k_stages >= 2 ? 2 : 1;
      int cursor = 0;
      int64_t cur_i = -1;                // tile of rc; rn is tile cur_i + 1
      const uint8_t* rc[4];
      const uint8_t* rn[4];
      uint32_t vc = 0, vn = 0;           // bit j: row lane + 32 j is real
      auto fetch_rows = [&](int64_t i, const uint8_t* (&src)[4], uint32_t& vb) {
        vb = 0;
        if (i >= n_my) return;
        const Tile tt = decode_tile(p, unit0 + i * unit_step, &cursor);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int32_t v = p.row_index[tt.m0 + lane + 32 * j];
          const bool ok_v = v >= 0 && v < p.T_src;
          vb |= (ok_v ? 1u : 0u) << j;
          src[j] = p.a_sf_lin + (int64_t)(ok_v ? v : 0) * p.a_sf_ld;
        }
      };
      auto load_stage = [&](int64_t j2, uint4 (&w)[4]) {
        const int64_t i = j2 / p.k_stages, kt = j2 % p.k_stages;
        if (i != cur_i) {                 // i == cur_i + 1 (or the first)
          if (cur_i < 0) {
            fetch_rows(i, rc, vc);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) rc[j] = rn[j];
            vc = vn;
          }
          cur_i = i;
          fetch_rows(i + 1, rn, vn);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          w[j] = (vc >> j) & 1 ? ld_stream_v4(rc[j] + kt * 16)
                               : make_uint4(0, 0, 0, 0);  // padding: scale 0
      };
      bool ok = true;
      // stage it: wait for its slot, write the words of buffer w, arrive,
      // then load stage it + D into w
      auto step = [&](int64_t it, uint4 (&w)[4]) {
        const int st = (int)(it % GSTAGES);
        const uint32_t ph = (uint32_t)((it / GSTAGES) & 1);
        if (lane == 0)
          ok = mbar_wait(smem_addr(&s.empty[st]), ph ^ 1, &s.abort,
                         &g_gemm_wait_error);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = lane + 32 * j;
          const int off = (r & 31) * 16 + (r >> 5) * 4;
          *reinterpret_cast<uint32_t*>(&s.sfa[st][0][off]) = w[j].x;
          *reinterpret_cast<uint32_t*>(&s.sfa[st][1][off]) = w[j].y;
          *reinterpret_cast<uint32_t*>(&s.sfa[st][2][off]) = w[j].z;
          *reinterpret_cast<uint32_t*>(&s.sfa[st][3][off]) = w[j].w;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&s.full[st]));
        if (it + D < total) load_stage(it + D, w);
      };
      uint4 wa[4], wb[4];
      if (total > 0) load_stage(0, wa);
      if (D == 2 && total > 1) load_stage(1, wb);
      for (int64_t it = 0; it < total && ok; it += D) {
        step(it, wa);
        if (D == 2 && it + 1 < total && ok) step(it + 1, wb);
      }
    }
  } else {
    // ---------------- epilogue: warps 3-10 ----------------
    // Tensor-memory lane quarter q = warp id mod 4 (lane = tile row),
    // column half h.  Each thread takes its row's 128 accumulator values
    // into registers and releases the accumulator, then stores them.
    const int e = warp - 3;
    const int q = warp & 3, h = e >> 2;
    int local = 0;
    int grp_cursor = 0;
    for (int64_t u = unit0; u < n_units; u += unit_step, ++local) {
      const bool ok = __all_sync(
          0xffffffffu,
          mbar_wait(smem_addr(&s.acc_full), (uint32_t)(local & 1), &s.abort,
                    &g_gemm_wait_error));
      if (!ok) break;
      tc_fence_after();
      uint32_t r[128];
      const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
      if (EPI == 0) {
        // columns h*128 .. h*128+127
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tc_ld_32x32_async(lane_base + (uint32_t)(h * 128 + c * 32),
                            r + c * 32);
      } else {
        // gate columns h*64.. (r[0..63]) and up columns 128 + h*64..
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tc_ld_32x32_async(lane_base + (uint32_t)(h * 64 + c * 32),
                            r + c * 32);
          tc_ld_32x32_async(lane_base + (uint32_t)(128 + h * 64 + c * 32),
                            r + 64 + c * 32);
        }
      }
      tc_wait_ld();
      // The accumulator may be overwritten once all eight warps hold it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&s.acc_empty));

      const Tile t = decode_tile(p, u, &grp_cursor);
      float rs = 1.0f;
      bool pad = false;               // gather mode: a padding row, stored as +0
      if (p.kind == 1) {
        if (p.row_index) {
          // gather mode: the routed row's source token
          const int32_t v = p.row_index[t.m0 + q * 32 + lane];
          pad = !(v >= 0 && v < p.T_src);
          rs = pad ? 0.0f : __fmul_rn(p.s_tok[v], p.s_w[t.grp]);
        } else {
          rs = __fmul_rn(p.s_tok[t.m0 + q * 32 + lane], p.s_w[t.grp]);
        }
      }
      const int64_t row_g = t.m0 + q * 32 + lane;   // M % 128 == 0
      if (EPI == 0) {
        // this thread's row: 32 consecutive fp32 per 32-column box, one
        // 32-byte store (a full sector) per 8 values
        const int64_t x0 = t.n0 + h * 128;
        float* crow = p.C + row_g * p.ldc + x0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (x0 + c * 32 >= p.N) break;  // columns past N: not stored
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            uint4 w[2];
#pragma unroll
            for (int d = 0; d < 2; ++d) {
              float4 v;
              v.x = __uint_as_float(r[c * 32 + 4 * (j + d)]);
              v.y = __uint_as_float(r[c * 32 + 4 * (j + d) + 1]);
              v.z = __uint_as_float(r[c * 32 + 4 * (j + d) + 2]);
              v.w = __uint_as_float(r[c * 32 + 4 * (j + d) + 3]);
              if (p.kind == 1) {
                v.x = __fmul_rn(v.x, rs);
                v.y = __fmul_rn(v.y, rs);
                v.z = __fmul_rn(v.z, rs);
                v.w = __fmul_rn(v.w, rs);
                if (pad) v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
              }
              w[d] = make_uint4(__float_as_uint(v.x), __float_as_uint(v.y),
                                __float_as_uint(v.z), __float_as_uint(v.w));
            }
            st_32B(crow + c * 32 + 4 * j, w[0], w[1], p.c_wide);
          }
        }
      } else {
        // h = silu(s g) * (s u) in binary32, to bf16; 64 columns of the
        // thread's row.  The fast exponential and divide (relative error below
        // 2^-20) are far inside the bf16 rounding (2^-9); for very negative
        // g, 1 + e^-g overflows and sigmoid comes out 0, the limit.
        uint16_t* hrow = p.H + row_g * p.ldc + t.n0 + h * 64;
        uint4 hw[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int col = j * 8 + k * 2;
            float g0, g1, u0, u1;
            fmul2(__uint_as_float(r[col]), __uint_as_float(r[col + 1]), rs,
                  rs, g0, g1);
            fmul2(__uint_as_float(r[64 + col]),
                  __uint_as_float(r[64 + col + 1]), rs, rs, u0, u1);
            const float s0 = __fdividef(1.0f, 1.0f + __expf(-g0));
            const float s1 = __fdividef(1.0f, 1.0f + __expf(-g1));
            float h0, h1;
            fmul2(g0, g1, s0, s1, h0, h1);
            fmul2(h0, h1, u0, u1, h0, h1);
            w[k] = pad ? 0u : f32x2_to_bf16x2(h0, h1);
          }
          hw[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        // this thread's row: 64 bf16 (128 bytes), one 32-byte store per 16
#pragma unroll
        for (int j = 0; j < 8; j += 2)
          st_32B(hrow + 8 * j, hw[j], hw[j + 1], p.c_wide);
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
  pdl_launch_dependents();
}

size_t gemm_smem_bytes() { return sizeof(GemmSmem) + 1024; }

cudaError_t make_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner,
                            uint64_t outer, uint64_t stride_bytes,
                            uint32_t box_rows) {
  return make_tmap_2d_bytes(map, base, inner, outer, stride_bytes, GKB,
                            box_rows);
}

// fp32 C [rows x cols] with row stride ldc floats, stored in 32 x 32 boxes.
cudaError_t make_tmap_c(CUtensorMap* map, float* C, int64_t rows,
                        int64_t cols, int64_t ldc) {
  return make_tmap_2d_f32(map, C, (uint64_t)cols, (uint64_t)rows,
                          (uint64_t)ldc * 4, 32, 32);
}

// A operand as a byte matrix [a_rows x a_row_bytes], loaded in boxes of
// box_rows rows (GM for tiles, 1 for the gather4 loads of gather mode).
struct AOperand {
  const uint8_t* base;
  int64_t row_bytes, rows;
  uint32_t box_rows = GM;
};

// One CTA per SM (or per tile when there are fewer tiles).
template <int EPI>
cudaError_t launch_gemm(const AOperand& a, const CUtensorMap& tb,
                        const GemmParams& p,
                        int64_t tiles, cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  GemmParams pp = p;
  pp.n_tiles = tiles;
  auto kern = gemm_block_scaled_kernel<EPI>;
  const size_t smem = gemm_smem_bytes();
  static int configured[64] = {};
  if (!configured[dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess) return err;
    configured[dev] = 1;
  }
  CUtensorMap ta;
  err = make_tmap_2d_u8(&ta, a.base, (uint64_t)a.row_bytes, (uint64_t)a.rows,
                        (uint64_t)a.row_bytes, a.box_rows);
  if (err != cudaSuccess) return err;
  const int64_t grid = imin<int64_t>(tiles, sm_count(dev));
  return launch_pdl(kern, dim3((unsigned)grid), dim3(GTHREADS), smem, stream,
                    false, ta, tb, pp);
}

// Grouped NVFP4 parameters shared by the plain and the SwiGLU GEMM.
void grouped_params(GemmParams& p, const uint8_t* a_scales, const float* a_s,
                    const int64_t* group_offsets, int64_t num_groups,
                    const uint8_t* w_scales, const float* w_s, int64_t w_rows,
                    int64_t K, int64_t* tiles_m) {
  p.kind = 1;
  p.M = group_offsets[num_groups];
  p.K = K;
  p.k_stages = K / 256;                 // 256 fp4 values (128 bytes) per stage
  p.a_sf = a_scales;
  p.b_sf = w_scales;
  p.a_sf_ct = (K / 16 + 3) / 4;
  p.b_sf_ct = p.a_sf_ct;
  p.b_sf_group_stride = scale_bytes(w_rows, K / 16, 1);
  p.b_rows_group_stride = w_rows;
  p.s_tok = a_s;
  p.s_w = w_s;
  p.num_groups = (int)num_groups;
  *tiles_m = 0;
  for (int64_t g = 0; g < num_groups; ++g) {
    p.row_off[g] = group_offsets[g];
    *tiles_m += (group_offsets[g + 1] - group_offsets[g]) / GM;
    p.tile_end[g] = *tiles_m;
  }
}

// Gather mode of the two grouped launchers: A's rows are rows row_index[r]
// of the per-token operand x (codes [T_src x K/2], linear block scales
// [T_src x K/16], S [T_src]).
void gather_params(GemmParams& p, const int32_t* row_index, int64_t T_src,
                   const uint8_t* x_scales_lin, int64_t K) {
  p.row_index = row_index;
  p.T_src = T_src;
  p.a_sf_lin = x_scales_lin;
  p.a_sf_ld = K / 16;
}

}  // namespace

cudaError_t gemm_take_wait_error(unsigned int* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_gemm_wait_error, sizeof(*word));
  if (e != cudaSuccess || *word == 0) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_gemm_wait_error, &zero, sizeof(zero));
}

cudaError_t launch_gemm_mxfp8(const uint8_t* a_codes, const uint8_t* a_scales,
                              const uint8_t* bt_codes,
                              const uint8_t* bt_scales, int64_t M, int64_t N,
                              int64_t K, float* C, int64_t ldc,
                              cudaStream_t stream) {
  CUtensorMap tb;
  cudaError_t err = make_tmap_2d_u8(&tb, bt_codes, (uint64_t)K, (uint64_t)N,
                                    (uint64_t)K, GN);
  if (err != cudaSuccess) return err;
  GemmParams p = {};
  p.kind = 0;
  p.M = M;
  p.N = N;
  p.K = K;
  p.k_stages = K / GKB;                 // 128 fp8 values per stage
  p.a_sf = a_scales;
  p.b_sf = bt_scales;
  p.a_sf_ct = (K / 32 + 3) / 4;         // 4 scale columns per tile
  p.b_sf_ct = p.a_sf_ct;
  p.b_sf_group_stride = 0;
  p.b_rows_group_stride = 0;
  p.num_groups = 1;
  p.tiles_n = (N + GN - 1) / GN;
  p.tile_cols = GN;
  p.C = C;
  p.ldc = ldc;
  p.c_wide = (reinterpret_cast<uintptr_t>(C) & 31u) == 0 && ldc % 8 == 0;
  return launch_gemm<0>(AOperand{a_codes, K, M}, tb, p,
                        (M / GM) * p.tiles_n, stream);
}

cudaError_t launch_gemm_nvfp4_grouped(
    const uint8_t* a_codes, const uint8_t* a_scales, const float* a_s,
    const int64_t* group_offsets, int64_t num_groups, const uint8_t* w_codes,
    const uint8_t* w_scales, const float* w_s, int64_t N, int64_t K, float* C,
    int64_t ldc, cudaStream_t stream, const int32_t* row_index,
    int64_t T_src) {
  // Packed E2M1: K/2 bytes per row; all groups' weights as one
  // [num_groups * N x K/2] byte matrix.
  CUtensorMap tb;
  cudaError_t err = make_tmap_2d_u8(&tb, w_codes, (uint64_t)(K / 2),
                                    (uint64_t)(num_groups * N),
                                    (uint64_t)(K / 2), GN);
  if (err != cudaSuccess) return err;
  GemmParams p = {};
  int64_t tiles_m = 0;
  grouped_params(p, a_scales, a_s, group_offsets, num_groups, w_scales, w_s,
                 N, K, &tiles_m);
  p.N = N;
  p.tiles_n = (N + GN - 1) / GN;
  p.tile_cols = GN;
  p.C = C;
  p.ldc = ldc;
  p.c_wide = (reinterpret_cast<uintptr_t>(C) & 31u) == 0 && ldc % 8 == 0;
  if (row_index) gather_params(p, row_index, T_src, a_scales, K);
  if (tiles_m == 0) return cudaSuccess;
  const AOperand a = row_index ? AOperand{a_codes, K / 2, T_src, 1}
                               : AOperand{a_codes, K / 2, p.M};
  return launch_gemm<0>(a, tb, p, tiles_m * p.tiles_n, stream);
}

cudaError_t launch_moe_gate_up_swiglu(
    const uint8_t* a_codes, const uint8_t* a_scales, const float* a_s,
    const int64_t* group_offsets, int64_t num_groups, const uint8_t* w_codes,
    const uint8_t* w_scales, const float* w_s, int64_t F, int64_t K,
    void* out, int64_t ldo, cudaStream_t stream, const int32_t* row_index,
    int64_t T_src) {
  // weights: [num_groups * 2F x K/2] bytes, gate rows then up rows per
  // group, loaded as 128-row boxes (gate block and matching up block)
  CUtensorMap tb;
  cudaError_t err = make_tmap_2d_u8(&tb, w_codes, (uint64_t)(K / 2),
                                    (uint64_t)(num_groups * 2 * F),
                                    (uint64_t)(K / 2), 128);
  if (err != cudaSuccess) return err;
  GemmParams p = {};
  int64_t tiles_m = 0;
  grouped_params(p, a_scales, a_s, group_offsets, num_groups, w_scales, w_s,
                 2 * F, K, &tiles_m);
  p.N = F;                              // output columns
  p.tiles_n = F / 128;
  p.tile_cols = 128;
  p.b_up_row = F;
  p.C = nullptr;
  p.H = static_cast<uint16_t*>(out);
  p.ldc = ldo;
  p.c_wide = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 && ldo % 16 == 0;
  if (row_index) gather_params(p, row_index, T_src, a_scales, K);
  if (tiles_m == 0) return cudaSuccess;
  const AOperand a = row_index ? AOperand{a_codes, K / 2, T_src, 1}
                               : AOperand{a_codes, K / 2, p.M};
  return launch_gemm<1>(a, tb, p, tiles_m * p.tiles_n, stream);
}

// ---------------------------------------------------------------------------
// Dequantized-backward GEMM: bf16 A times an MXFP8 operand whose bf16
// values are formed in shared memory and never written to HBM.
//
// "Miles: end-to-end MXFP8 and per-token NVFP4 RL", backward-mode section:
// in dequantized-backward mode the backward GEMMs run in BF16 on BF16
// dequantizations of the exact forward low-precision operands.  Here
//   C[m, n] = sum_k A[m, k] * Bq[k, n],   A bf16 [M x K] (e.g. dY),
// Bq given as B^T [N x K]: MXFP8 codes with 1x32 E8M0 scales along K (the
// columnwise copy of a forward operand), Bq[k, n] = E4M3(code) * 2^(s-127),
// exact in bf16.  fp32 accumulation in tensor memory, fp32 C.
//
// Design: persistent, one CTA per SM, 256 x 128 output tiles computed as
// two 128 x 128 accumulators that share one converted B tile (so each B
// value is converted once per 256 rows of A), 23 warps, a 4-deep ring of
// K-stages of 64 values.  Warp 0 lane 0 loads a stage's A tile (bf16, 256
// rows of 128 bytes, 128-byte swizzle) by 2-D TMA.  Warps 7-22, in two
// groups of 8 for the even and the odd stages (two threads per B row, 32
// values each), read the B^T codes and E8M0 scales from global memory one
// own stage ahead and, once the stage's slot is free, write the bf16
// values into its B buffer in the 128-byte-swizzled K-major layout the
// tensor core reads; then they fence the writes to the async proxy and
// count themselves on the stage's "converted" barrier.  The bf16 values
// come from integer bit moves and packed bf16 multiplies by powers of two,
// in an order free of shared-memory bank conflicts.  Warp 2 waits for the
// A tile and the conversion and hands the stage to warp 1, whose lane 0
// issues eight kind::f16 MMAs (K = 16 each, four per accumulator) and
// commits; warps 3-6 take the accumulators 32 columns at a time to
// registers, release them after the last, and store C in 32 x 32 fp32
// boxes by TMA.  Every wait is bounded.
// ---------------------------------------------------------------------------
namespace {

constexpr int DQ_M = 128, DQ_N = 128;     // one MMA / accumulator
constexpr int DQ_MT = 2 * DQ_M;           // rows of A per tile
constexpr int DQ_KE = 64;                 // K values per stage
constexpr int DQ_STAGES = 4;
constexpr int DQ_THREADS = 32 * 23;
constexpr uint32_t kDqTmemCols = 256;     // two 128 x 128 fp32 accumulators

struct alignas(1024) DqSmem {
  uint8_t a[DQ_STAGES][DQ_MT * 128];      // bf16, 128-byte swizzled rows
  uint8_t b[DQ_STAGES][DQ_N * 128];       // bf16 from the codes, same layout
  // epilogue staging boxes: 1024-byte aligned, as the 128-byte swizzle of
  // the C tensor map is laid out from 1024-byte boundaries
  alignas(1024) uint8_t cst[4][32 * 128];
  alignas(8) uint64_t full[DQ_STAGES];
  alignas(8) uint64_t conv[DQ_STAGES];
  alignas(8) uint64_t empty[DQ_STAGES];
  alignas(8) uint64_t acc_full;
  alignas(8) uint64_t acc_empty;
  uint32_t tmem_base;
  int abort;
};

struct DqParams {
  int64_t M, N, K;
  int64_t k_stages;
  int64_t tiles_n, n_tiles;
  const uint8_t* b_codes;                 // E4M3 codes of B^T [N x K]
  const uint8_t* b_sf;                    // swizzled E8M0 of B^T [N x K/32]
  int64_t b_sf_ct;                        // scale column tiles, ceil(K/128)
};

// Instruction descriptor of a dense kind::f16 MMA with bf16 A and B (both
// K-major), fp32 accumulator, M = DQ_M, N = DQ_N.
__device__ __forceinline__ uint32_t idesc_bf16() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(DQ_N >> 3) << 17) |
         ((uint32_t)(DQ_M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d, uint64_t adesc,
                                           uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Sixteen E4M3 codes with one E8M0 scale s -> sixteen bf16
// RNE_bf16(E4M3(c) * 2^(s - 127)), packed in pairs (element 0 low), without
// the conversion pipe.  A code's sign moved to bit 15 and its other seven
// bits moved up by four form the bf16 E4M3(c) * 2^-120 exactly (the E4M3
// exponent lands in the low four bits of the bf16 exponent field, the
// mantissa in the top three mantissa bits; subnormal codes land on bf16
// subnormals of the same scale).  One or two packed bf16 multiplies by
// powers of two then give the scaled value with one rounding: 2^(s - 7)
// when that is a bf16 (s <= 134), else 2^120 (exact) then 2^(s - 127).
// The product has at most four significant bits, so its binary32 value is
// exact whenever finite and rounding it once to bf16 equals the binary32
// multiply followed by the bf16 conversion; overflow gives inf on both
// routes.  The E8M0 NaN byte 0xFF multiplies by a bf16 NaN; chunks holding
// an E4M3 NaN code (S.1111.111) take the conversion instructions instead.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ void e4m3x16_scale_bf16(const uint4 v, uint32_t sb,
                                                   uint32_t (&w)[8]) {
  const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
  uint32_t nan = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    nan |= ((cw[i] & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
  if (__builtin_expect(nan != 0, 0)) {
    const float sc = e8m0_scale(sb);
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      float x0, x1;
      e4m3x2_to_f32((cw[h >> 1] >> ((h & 1) * 16)) & 0xFFFFu, x0, x1);
      fmul2(x0, x1, sc, sc, x0, x1);
      w[h] = f32x2_to_bf16x2(x0, x1);
    }
    return;
  }
  const bool one = sb <= 134u;
  const uint32_t f1 = (one ? sb + 120u : 247u) << 7;
  const uint32_t f2 = one ? (127u << 7) : sb < 255u ? sb << 7 : 0x7FC0u;
  const uint32_t f1x2 = f1 | (f1 << 16), f2x2 = f2 | (f2 << 16);
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    // codes 2h, 2h + 1 into the low bytes of the two 16-bit halves, each
    // high byte filled with copies of its code's sign bit (the permute's
    // sign-replicating selectors); shifted up by four, the mask keeps the
    // sign at bit 15 and the seven other code bits at bits 4-10
    uint32_t t;
    if ((h & 1) == 0)
      asm("prmt.b32 %0, %1, 0, %2;" : "=r"(t) : "r"(cw[h >> 1]), "n"(0x9180));
    else
      asm("prmt.b32 %0, %1, 0, %2;" : "=r"(t) : "r"(cw[h >> 1]), "n"(0xB3A2));
    w[h] = (t << 4) & 0x87F087F0u;
  }
  if (one) {
#pragma unroll
    for (int h = 0; h < 8; ++h) w[h] = bf16x2_mul(w[h], f1x2);
  } else {
#pragma unroll
    for (int h = 0; h < 8; ++h) w[h] = bf16x2_mul(bf16x2_mul(w[h], f1x2), f2x2);
  }
}

// Position in the stage ring, advanced once per K-stage: slot, phase
// parity of the slot's barriers, and the stage's parity.
struct RingPos {
  int st = 0;
  uint32_t ph = 0;
  int par = 0;
  __device__ __forceinline__ void next() {
    par ^= 1;
    if (++st == DQ_STAGES) {
      st = 0;
      ph ^= 1;
    }
  }
};

__global__ void __launch_bounds__(DQ_THREADS, 1)
    gemm_bf16_dq_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_c,
                        const __grid_constant__ DqParams p) {
  extern __shared__ uint8_t dsmem_raw[];
  DqSmem& s = *reinterpret_cast<DqSmem*>(
      (reinterpret_cast<uintptr_t>(dsmem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0) tmem_alloc(smem_addr(&s.tmem_base), kDqTmemCols);
  if (threadIdx.x == 0) {
    for (int i = 0; i < DQ_STAGES; ++i) {
      mbar_init(smem_addr(&s.full[i]), 1);
      mbar_init(smem_addr(&s.conv[i]), 8);          // converter warps
      mbar_init(smem_addr(&s.empty[i]), 1);
    }
    mbar_init(smem_addr(&s.acc_full), 1);
    mbar_init(smem_addr(&s.acc_empty), 4);          // epilogue warps
    s.abort = 0;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- producer ----------------
      RingPos rp;
      for (int64_t t = blockIdx.x; t < p.n_tiles; t += gridDim.x) {
        const int64_t m0 = (t / p.tiles_n) * DQ_MT;
        for (int64_t kt = 0; kt < p.k_stages; ++kt, rp.next()) {
          const int st = rp.st;
          const uint32_t ph = rp.ph;
          if (!mbar_wait_sleep(smem_addr(&s.empty[st]), ph ^ 1, &s.abort,
                               &g_gemm_wait_error))
            break;
          const uint32_t full = smem_addr(&s.full[st]);
          mbar_arrive_expect_tx(full, DQ_MT * 128);
          // two boxes of 128 rows; rows past M (M % 256 == 128) read as 0
          tma_load_2d(smem_addr(s.a[st]), &tmap_a, (int32_t)(kt * DQ_KE),
                      (int32_t)m0, full);
          tma_load_2d(smem_addr(s.a[st]) + DQ_M * 128, &tmap_a,
                      (int32_t)(kt * DQ_KE), (int32_t)(m0 + DQ_M), full);
        }
        if (s.abort) break;
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    RingPos rp;
    bool aborted = false;
    for (int64_t t = blockIdx.x; t < p.n_tiles && !aborted; t += gridDim.x) {
      for (int64_t kt = 0; kt < p.k_stages; ++kt, rp.next()) {
        __syncwarp();
        if (stage_handoff(false)) {
          aborted = true;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const int st = rp.st;
          const uint32_t a_addr = smem_addr(s.a[st]);
          const uint32_t b_addr = smem_addr(s.b[st]);
          // per K = 16 bf16 values (32 bytes of each row), one MMA per
          // 128-row half of A into its accumulator (columns 128 h), both on
          // the same converted B
          for (int j = 0; j < 4; ++j) {
            const uint64_t bd = smem_desc(b_addr + j * 32, 16, 1024, 2);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t ad =
                  smem_desc(a_addr + h * DQ_M * 128 + j * 32, 16, 1024, 2);
              tc_mma_f16(tmem + (uint32_t)(h * DQ_N), ad, bd, idesc_bf16(),
                         (kt > 0 || j > 0) ? 1u : 0u);
            }
          }
          tc_commit(smem_addr(&s.empty[st]));
          if (kt == p.k_stages - 1) tc_commit(smem_addr(&s.acc_full));
        }
      }
    }
  } else if (warp == 2) {
    // ---------------- waiter ----------------
    RingPos rp;
    int local = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++local) {
      if (lane == 0)
        ok = mbar_wait_sleep(smem_addr(&s.acc_empty),
                             (uint32_t)((local & 1) ^ 1), &s.abort,
                             &g_gemm_wait_error);
      for (int64_t kt = 0; kt < p.k_stages; ++kt, rp.next()) {
        const int st = rp.st;
        const uint32_t ph = rp.ph;
        if (lane == 0 && ok)
          ok = mbar_wait_sleep(smem_addr(&s.full[st]), ph, &s.abort,
                               &g_gemm_wait_error) &&
               mbar_wait_sleep(smem_addr(&s.conv[st]), ph, &s.abort,
                               &g_gemm_wait_error);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        if (stage_handoff(!ok)) {
          ok = false;
          break;
        }
      }
    }
  } else if (warp >= 7) {
    // ---------------- converters: warps 7-22 ----------------
    // Two groups of 8 warps take the even and the odd stages, so two
    // stages are converted at once.  In a group, two threads per B row:
    // thread ct: row n = ct % 128, half hc = ct / 128.  It converts the
    // code chunks 2 hh and 2 hh + 1 of its row (32 values, one E8M0 block),
    // hh = hc ^ p(n), in the order c ^ g(n): with p(n) = 1 for n % 8 in
    // {0, 1, 4, 5} and g(n) = 1 for n % 8 in {2, 3, 4, 5}, the 8 lanes of
    // every shared-memory phase write 8 different bank groups of the
    // swizzled bf16 tile (chunk j of row n at j ^ (n % 8)).  The codes and
    // the scale byte come straight from global memory (L2), loaded one own
    // stage ahead; a stage's conversion waits only for its slot to be
    // released by the MMAs, not for the A tile.
    const int grp = (warp - 7) >> 3;                  // stage parity
    const int ct = threadIdx.x - 7 * 32 - grp * 256;  // 0 .. 255
    const int n = ct & 127;
    const int hh = (ct >> 7) ^ ((0x33 >> (n & 7)) & 1);
    const int g = (0x3C >> (n & 7)) & 1;
    const int sf_in_tile = (n & 31) * 16 + (n >> 5) * 4 + hh;
    // (t, kt) advanced by d K-stages along this CTA's tile sequence
    auto advance = [&](int64_t& t_, int64_t& kt_, int d) {
      kt_ += d;
      while (kt_ >= p.k_stages) {
        kt_ -= p.k_stages;
        t_ += gridDim.x;
      }
    };
    // the row's codes and its scales' tile row, set when the tile changes
    // (loads run in tile order)
    int64_t cur_t = -1;
    const uint8_t* crow = nullptr;
    const uint8_t* srow = nullptr;
    auto load = [&](int64_t t_, int64_t kt_, uint4& c0, uint4& c1,
                    uint32_t& sbv) {
      if (t_ != cur_t) {
        cur_t = t_;
        const int64_t nrow = (t_ % p.tiles_n) * DQ_N + n;
        crow = p.b_codes + nrow * p.K + hh * 32;
        srow = p.b_sf + (nrow >> 7) * p.b_sf_ct * 512 + sf_in_tile;
      }
      const uint8_t* src = crow + kt_ * DQ_KE;
      c0 = ld_stream_v4(src + g * 16);
      c1 = ld_stream_v4(src + (g ^ 1) * 16);
      // swizzled scale tile (nrow / 128, kt / 2): block column 2 (kt % 2) + hh
      sbv = __ldg(srow + (kt_ >> 1) * 512 + 2 * (int)(kt_ & 1));
    };
    RingPos rp;
    if (grp) rp.next();
    int64_t t = blockIdx.x, kt = 0;
    advance(t, kt, grp);
    uint4 cv0 = make_uint4(0, 0, 0, 0), cv1 = cv0;
    uint32_t sb = 0;
    if (t < p.n_tiles) load(t, kt, cv0, cv1, sb);
    while (t < p.n_tiles) {
      const int st = rp.st;
      bool ok = true;
      if (lane == 0)
        ok = mbar_wait_sleep(smem_addr(&s.empty[st]), rp.ph ^ 1, &s.abort,
                             &g_gemm_wait_error);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      int64_t t2 = t, kt2 = kt;
      advance(t2, kt2, 2);
      uint4 nv0 = cv0, nv1 = cv1;
      uint32_t nsb = sb;
      if (t2 < p.n_tiles) load(t2, kt2, nv0, nv1, nsb);
      uint8_t* row = s.b[st] + n * 128;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int cc = 2 * hh + (c ^ g);                // code chunk
        uint32_t w[8];
        e4m3x16_scale_bf16(c == 0 ? cv0 : cv1, sb, w);
        // bf16 chunks 2 cc and 2 cc + 1 of the row, 128-byte swizzle
        const int q0 = (2 * cc) ^ (n & 7), q1 = (2 * cc + 1) ^ (n & 7);
        *reinterpret_cast<uint4*>(row + q0 * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(row + q1 * 16) =
            make_uint4(w[4], w[5], w[6], w[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&s.conv[st]));
      cv0 = nv0;
      cv1 = nv1;
      sb = nsb;
      t = t2;
      kt = kt2;
      rp.next();
      rp.next();
    }
  } else {
    // ---------------- epilogue: warps 3-6 ----------------
    // 32 accumulator columns at a time (32 registers): each 32 x 32 box
    // goes tensor memory -> registers -> swizzled staging -> TMA store; the
    // accumulator is released once its last columns are in registers.
    const int q = warp & 3;                           // tensor-memory quarter
    uint8_t* box = s.cst[warp - 3];
    uint8_t* rowp = box + lane * 128;
    int local = 0;
    for (int64_t t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++local) {
      // a tile's whole main loop passes here: sleep, and leave the issue
      // slots to the converter warps on the same schedulers
      const bool ok = __all_sync(
          0xffffffffu,
          mbar_wait_sleep(smem_addr(&s.acc_full), (uint32_t)(local & 1),
                          &s.abort, &g_gemm_wait_error));
      if (!ok) break;
      tc_fence_after();
      const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
      const int64_t m0 = (t / p.tiles_n) * DQ_MT;
      const int64_t n0 = (t % p.tiles_n) * DQ_N;
      // chunk c: accumulator h = c / 4 (rows m0 + 128 h + 32 q + lane),
      // columns 32 (c % 4) ..; a half past M is not stored
      const int nc = (m0 + DQ_M < p.M) ? 8 : 4;
      for (int c = 0; c < 8; ++c) {
        uint32_t r[32];
        tc_ld_32x32_async(lane_base + (uint32_t)(c * 32), r);
        tc_wait_ld();
        if (c == 7) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&s.acc_empty));
        }
        if (lane == 0) bulk_wait_read_0();              // the box's last store
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float4 v;
          v.x = __uint_as_float(r[4 * j]);
          v.y = __uint_as_float(r[4 * j + 1]);
          v.z = __uint_as_float(r[4 * j + 2]);
          v.w = __uint_as_float(r[4 * j + 3]);
          *reinterpret_cast<float4*>(rowp + ((j ^ (lane & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && c < nc) {
          tma_store_2d(&tmap_c, smem_addr(box), (int32_t)(n0 + (c & 3) * 32),
                       (int32_t)(m0 + (c >> 2) * DQ_M + q * 32));
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kDqTmemCols);
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_gemm_bf16_mxfp8(const void* a, int64_t lda,
                                   const uint8_t* bt_codes,
                                   const uint8_t* bt_scales, int64_t M,
                                   int64_t N, int64_t K, float* C, int64_t ldc,
                                   cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  CUtensorMap ta, tc;
  err = make_tmap_2d_bf16(&ta, a, (uint64_t)K, (uint64_t)M, (uint64_t)lda * 2,
                          DQ_KE, DQ_M, true);
  if (err != cudaSuccess) return err;
  err = make_tmap_c(&tc, C, M, N, ldc);
  if (err != cudaSuccess) return err;
  DqParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.k_stages = K / DQ_KE;
  p.tiles_n = N / DQ_N;
  p.n_tiles = ((M + DQ_MT - 1) / DQ_MT) * p.tiles_n;
  p.b_codes = bt_codes;
  p.b_sf = bt_scales;
  p.b_sf_ct = (K / 32 + 3) / 4;
  const size_t smem = sizeof(DqSmem) + 1024;
  static int configured[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    err = cudaFuncSetAttribute(gemm_bf16_dq_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess) return err;
    configured[dev] = 1;
  }
  const int64_t grid = imin<int64_t>(p.n_tiles, sm_count(dev));
  return launch_pdl(gemm_bf16_dq_kernel, dim3((unsigned)grid),
                    dim3(DQ_THREADS), smem, stream, false, ta, tc, p);
}

}  // namespace mxq
