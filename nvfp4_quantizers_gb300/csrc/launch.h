// launch.h -- internal interface between the C ABI (api.cu) and the kernel
// translation units.  Every launcher enqueues on `stream`, never
// synchronizes, and returns the launch status.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace mxq {

// Host utilities (api.cu).
// Host-side fault injection (mxq_set_fault_inject / MXQ_FAULT_INJECT):
// 0 = off, 1 = fail every launch with MXQ_ERR_CUDA, 2 = reject every call
// with MXQ_ERR_ARG.
int host_fault_mode();
int sm_count(int device);
int64_t l2_bytes(int device);
cudaError_t make_tmap_2d_bytes(CUtensorMap* map, const void* base,
                               uint64_t inner, uint64_t outer,
                               uint64_t outer_stride_bytes, uint32_t box_inner,
                               uint32_t box_outer);
cudaError_t make_tmap_2d_bf16(CUtensorMap* map, const void* base,
                              uint64_t inner, uint64_t outer,
                              uint64_t outer_stride_bytes, uint32_t box_inner,
                              uint32_t box_outer, bool swizzle128);
// fp32 matrix, 128-byte swizzle (box_inner * 4 <= 128).
cudaError_t make_tmap_2d_f32(CUtensorMap* map, const void* base,
                             uint64_t inner, uint64_t outer,
                             uint64_t outer_stride_bytes, uint32_t box_inner,
                             uint32_t box_outer);

// mxfp8.cu
// Reads (and clears when set) the error word of the bounded device waits.
cudaError_t mxfp8_take_wait_error(unsigned int* word);
// One CTA whose bounded mbarrier wait runs out after limit_ns.
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_mxfp8_rowcol(const void* x, int64_t M, int64_t K,
                                int64_t ldx, uint8_t* row_codes,
                                uint8_t* row_scales, uint8_t* col_codes,
                                uint8_t* col_scales, int swizzled,
                                cudaStream_t stream);

// nvfp4.cu
// row_index: NULL, or a device int32 [T]: output row t quantizes x row
// row_index[t] (indices outside [0, T_src) give a zero row).
cudaError_t launch_nvfp4_per_token(const void* x, int64_t T, int64_t H,
                                   int64_t ldx, const int32_t* row_index,
                                   int64_t T_src, uint8_t* codes,
                                   uint8_t* scales, float* token_scales,
                                   int swizzled, cudaStream_t stream);

constexpr int kMaxParts = 4;

// Workspace of the shared-scale weight quantizer: a 256-byte header (task
// counters) followed by an amax word and a progress word per group.
size_t nvfp4_weight_ws_bytes(int64_t num_groups);
// Reads (and clears when set) the error word of the weight kernel's
// bounded waits.
cudaError_t nvfp4_take_wait_error(unsigned int* word);

cudaError_t launch_nvfp4_weight_shared(
    int64_t num_groups, int num_parts, const void* const* parts,
    const int64_t* part_rows, int64_t K, uint8_t* codes, uint8_t* scales,
    float* group_scales, const float* group_scales_in, int swizzled,
    uint32_t* ws, cudaStream_t stream);

// dequant.cu
cudaError_t launch_dequant_mxfp8(const uint8_t* codes, const uint8_t* scales,
                                 int64_t rows, int64_t cols, int swizzled,
                                 void* y, cudaStream_t stream);
cudaError_t launch_dequant_nvfp4(const uint8_t* codes, const uint8_t* scales,
                                 const float* S, int per_batch, int64_t batch,
                                 int64_t rows, int64_t cols, int swizzled,
                                 void* y, cudaStream_t stream);

// Launch `kernel` on `stream` with programmatic stream serialization (and
// optionally as a cooperative grid), so its launch overlaps the tail of
// the previous kernel on the stream; the kernel itself orders its memory
// accesses after that kernel with griddepcontrol.wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                       size_t smem, cudaStream_t stream, bool cooperative,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cooperative ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// gemm.cu
cudaError_t gemm_take_wait_error(unsigned int* word);
// C [M x N] fp32 = A bf16 [M x K] (row stride lda) x dequant(B), B^T
// [N x K] given as MXFP8 codes + swizzled E8M0 scales.
cudaError_t launch_gemm_bf16_mxfp8(const void* a, int64_t lda,
                                   const uint8_t* bt_codes,
                                   const uint8_t* bt_scales, int64_t M,
                                   int64_t N, int64_t K, float* C, int64_t ldc,
                                   cudaStream_t stream);
cudaError_t launch_gemm_mxfp8(const uint8_t* a_codes, const uint8_t* a_scales,
                              const uint8_t* bt_codes,
                              const uint8_t* bt_scales, int64_t M, int64_t N,
                              int64_t K, float* C, int64_t ldc,
                              cudaStream_t stream);
// row_index != NULL (gather mode): A's routed row r is row row_index[r] of
// the per-token operand (a_codes [T_src x K/2], a_scales its LINEAR block
// scales [T_src x K/16], a_s [T_src]); indices outside [0, T_src) are
// padding rows, which contribute 0.
cudaError_t launch_gemm_nvfp4_grouped(
    const uint8_t* a_codes, const uint8_t* a_scales, const float* a_s,
    const int64_t* group_offsets, int64_t num_groups, const uint8_t* w_codes,
    const uint8_t* w_scales, const float* w_s, int64_t N, int64_t K, float* C,
    int64_t ldc, cudaStream_t stream, const int32_t* row_index = nullptr,
    int64_t T_src = 0);
// h = silu(gate) * up over the grouped gate/up GEMM, bf16 [rows x F].
cudaError_t launch_moe_gate_up_swiglu(
    const uint8_t* a_codes, const uint8_t* a_scales, const float* a_s,
    const int64_t* group_offsets, int64_t num_groups, const uint8_t* w_codes,
    const uint8_t* w_scales, const float* w_s, int64_t F, int64_t K,
    void* out, int64_t ldo, cudaStream_t stream,
    const int32_t* row_index = nullptr, int64_t T_src = 0);

// Scale-matrix size in bytes for either layout.
inline int64_t scale_bytes(int64_t rows, int64_t cols, int swizzled) {
  if (!swizzled) return rows * cols;
  return ((rows + 127) / 128) * 128 * ((cols + 3) / 4) * 4;
}

// nvfp4_rht.cu
// flags: bit 0 Random Hadamard Transform, bit 1 stochastic rounding.
cudaError_t launch_nvfp4_rht_sr(const void* x, int64_t T, int64_t H,
                                int64_t ldx, uint64_t seed, int flags,
                                uint8_t* codes, uint8_t* scales,
                                float* token_scales, int swizzled,
                                cudaStream_t stream);

// fp8block.cu
// block_rows 1 (1x128 tiles) or 128 (128x128 blocks).
// Reads (and clears when set) the error word of the bounded device waits.
cudaError_t fp8blk_take_wait_error(unsigned int* word);
cudaError_t launch_fp8blk_quantize(const void* x, int64_t rows, int64_t cols,
                                   int64_t ldx, int block_rows,
                                   uint8_t* codes, float* scales,
                                   cudaStream_t stream);
cudaError_t launch_fp8blk_dequantize(const uint8_t* codes, const float* scales,
                                     int64_t rows, int64_t cols,
                                     int block_rows, void* y,
                                     cudaStream_t stream);
cudaError_t launch_fp8blk_requant_t(const uint8_t* codes, const float* scales,
                                    int64_t M, int64_t K, uint8_t* codes_t,
                                    float* scales_t, cudaStream_t stream);

}  // namespace mxq
