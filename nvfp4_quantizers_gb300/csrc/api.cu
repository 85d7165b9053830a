// api.cu -- the extern "C" boundary of libmxq: argument validation, status
// codes and host utilities.  Kernels live in mxfp8.cu, nvfp4.cu and
// dequant.cu; nothing here allocates device memory or synchronizes (except
// mxq_get_last_error, which documents that it does).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/mxq.h"
#include "launch.h"

namespace mxq {

namespace {

std::atomic<int> g_fault_mode{-1};

int fault_mode() {
  int m = g_fault_mode.load(std::memory_order_relaxed);
  if (m < 0) {
    const char* e = getenv("MXQ_FAULT_INJECT");
    m = 0;
    if (e && strcmp(e, "launch") == 0) m = 1;
    if (e && strcmp(e, "argcheck") == 0) m = 2;
    g_fault_mode.store(m, std::memory_order_relaxed);
  }
  return m;
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool valid_layout(int layout) {
  return layout == MXQ_SCALE_LINEAR || layout == MXQ_SCALE_SWIZZLED;
}

mxq_status from_cuda(cudaError_t e) {
  return e == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
int64_t g_l2_bytes[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType,
                                  cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

int host_fault_mode() { return fault_mode(); }

int sm_count(int device) {
  if (device < 0 || device >= kMaxDevices) return 1;
  int n = g_sm_count[device];
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) !=
            cudaSuccess ||
        n <= 0)
      n = 1;
    g_sm_count[device] = n;
  }
  return n;
}

int64_t l2_bytes(int device) {
  if (device < 0 || device >= kMaxDevices) return 32ll << 20;
  int64_t b = g_l2_bytes[device];
  if (b == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, device) !=
            cudaSuccess ||
        v <= 0)
      v = 32 << 20;
    b = v;
    g_l2_bytes[device] = b;
  }
  return b;
}

cudaError_t make_tmap_2d_bf16(CUtensorMap* map, const void* base,
                              uint64_t inner, uint64_t outer,
                              uint64_t outer_stride_bytes, uint32_t box_inner,
                              uint32_t box_outer, bool swizzle128) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {outer_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B
                             : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_2d_f32(CUtensorMap* map, const void* base,
                             uint64_t inner, uint64_t outer,
                             uint64_t outer_stride_bytes, uint32_t box_inner,
                             uint32_t box_outer) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {outer_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_2d_bytes(CUtensorMap* map, const void* base,
                               uint64_t inner, uint64_t outer,
                               uint64_t outer_stride_bytes, uint32_t box_inner,
                               uint32_t box_outer) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {outer_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace mxq

using namespace mxq;

extern "C" {

const char* mxq_status_string(mxq_status s) {
  switch (s) {
    case MXQ_OK: return "MXQ_OK";
    case MXQ_ERR_NULL: return "MXQ_ERR_NULL: a required pointer is NULL";
    case MXQ_ERR_SHAPE:
      return "MXQ_ERR_SHAPE: a size is negative or not a multiple of the block";
    case MXQ_ERR_ALIGN:
      return "MXQ_ERR_ALIGN: a pointer or leading dimension is not 16-byte aligned";
    case MXQ_ERR_LAYOUT: return "MXQ_ERR_LAYOUT: unknown scale layout or mode";
    case MXQ_ERR_WORKSPACE: return "MXQ_ERR_WORKSPACE: workspace missing or too small";
    case MXQ_ERR_CUDA: return "MXQ_ERR_CUDA: a CUDA call or launch failed";
    case MXQ_ERR_TIMEOUT: return "MXQ_ERR_TIMEOUT: a bounded device wait gave up";
    case MXQ_ERR_ARG: return "MXQ_ERR_ARG: invalid argument";
    default: return "MXQ: unknown status";
  }
}

int mxq_version(void) { return 100; }

int64_t mxq_scale_bytes(int64_t rows, int64_t cols, int scale_layout) {
  if (!valid_layout(scale_layout) || rows < 0 || cols < 0) return -1;
  return scale_bytes(rows, cols, scale_layout == MXQ_SCALE_SWIZZLED);
}

mxq_status mxq_get_last_error(void) {
  cudaError_t e = cudaDeviceSynchronize();
  unsigned int word = 0, word2 = 0;
  unsigned int word3 = 0, word4 = 0;
  cudaError_t e2 = mxfp8_take_wait_error(&word);
  if (e2 == cudaSuccess) e2 = nvfp4_take_wait_error(&word2);
  if (e2 == cudaSuccess) e2 = gemm_take_wait_error(&word3);
  if (e2 == cudaSuccess) e2 = fp8blk_take_wait_error(&word4);
  if (e2 == cudaSuccess && (word | word2 | word3 | word4) != 0)
    return MXQ_ERR_TIMEOUT;
  cudaError_t last = cudaGetLastError();
  if (e != cudaSuccess || e2 != cudaSuccess || last != cudaSuccess)
    return MXQ_ERR_CUDA;
  return MXQ_OK;
}

mxq_status mxq_selftest_wait_timeout(void* stream) {
  return from_cuda(launch_wait_selftest(20ull * 1000 * 1000,
                                        static_cast<cudaStream_t>(stream)));
}

void mxq_set_fault_inject(int mode) {
  g_fault_mode.store(mode < 0 ? 0 : mode, std::memory_order_relaxed);
}

mxq_status mxfp8_quantize_rowcol(const void* x, int64_t M, int64_t K,
                                 int64_t ldx, uint8_t* row_codes,
                                 uint8_t* row_scales, uint8_t* col_codes_t,
                                 uint8_t* col_scales_t, int scale_layout,
                                 void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (!valid_layout(scale_layout)) return MXQ_ERR_LAYOUT;
  if (M < 0 || K < 0 || ldx < K) return MXQ_ERR_SHAPE;
  const bool do_row = row_codes || row_scales;
  const bool do_col = col_codes_t || col_scales_t;
  if (!do_row && !do_col) return MXQ_ERR_NULL;
  if (do_row && (!row_codes || !row_scales)) return MXQ_ERR_NULL;
  if (do_col && (!col_codes_t || !col_scales_t)) return MXQ_ERR_NULL;
  if (M == 0 || K == 0) return MXQ_OK;
  if (!x) return MXQ_ERR_NULL;
  if (K % 32 != 0 || (do_col && M % 32 != 0)) return MXQ_ERR_SHAPE;
  if (M >= (1ll << 31) || K >= (1ll << 31)) return MXQ_ERR_SHAPE;
  if (!aligned16(x) || ldx % 8 != 0) return MXQ_ERR_ALIGN;
  if ((do_row && (!aligned16(row_codes) || !aligned16(row_scales))) ||
      (do_col && (!aligned16(col_codes_t) || !aligned16(col_scales_t))))
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_mxfp8_rowcol(
      x, M, K, ldx, do_row ? row_codes : nullptr, row_scales,
      do_col ? col_codes_t : nullptr, col_scales_t,
      scale_layout == MXQ_SCALE_SWIZZLED, static_cast<cudaStream_t>(stream)));
}

mxq_status nvfp4_quantize_per_token(const void* x, int64_t T, int64_t H,
                                    int64_t ldx, uint8_t* codes,
                                    uint8_t* block_scales,
                                    float* token_scales, int scale_layout,
                                    void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (!valid_layout(scale_layout)) return MXQ_ERR_LAYOUT;
  if (T < 0 || H < 0 || ldx < H) return MXQ_ERR_SHAPE;
  if (T == 0 || H == 0) return MXQ_OK;
  if (!x || !codes || !block_scales || !token_scales) return MXQ_ERR_NULL;
  if (H % 16 != 0 || H >= (1ll << 30)) return MXQ_ERR_SHAPE;
  if (!aligned16(x) || ldx % 8 != 0 || !aligned16(codes) ||
      !aligned16(block_scales) || !aligned16(token_scales))
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_nvfp4_per_token(
      x, T, H, ldx, nullptr, T, codes, block_scales, token_scales,
      scale_layout == MXQ_SCALE_SWIZZLED, static_cast<cudaStream_t>(stream)));
}

mxq_status nvfp4_quantize_per_token_gather(
    const void* x, int64_t T_src, int64_t H, int64_t ldx,
    const int32_t* row_index, int64_t T, uint8_t* codes,
    uint8_t* block_scales, float* token_scales, int scale_layout,
    void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (!valid_layout(scale_layout)) return MXQ_ERR_LAYOUT;
  if (T < 0 || T_src < 0 || H < 0 || ldx < H) return MXQ_ERR_SHAPE;
  if (T == 0 || H == 0) return MXQ_OK;
  if (!row_index || !codes || !block_scales || !token_scales)
    return MXQ_ERR_NULL;
  if (T_src > 0 && !x) return MXQ_ERR_NULL;
  if (H % 16 != 0 || H >= (1ll << 30) || T_src >= (1ll << 31))
    return MXQ_ERR_SHAPE;
  if ((x && !aligned16(x)) || ldx % 8 != 0 || !aligned16(codes) ||
      !aligned16(block_scales) || !aligned16(token_scales) ||
      (reinterpret_cast<uintptr_t>(row_index) & 3u) != 0)
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_nvfp4_per_token(
      x, T, H, ldx, row_index, T_src, codes, block_scales, token_scales,
      scale_layout == MXQ_SCALE_SWIZZLED, static_cast<cudaStream_t>(stream)));
}

size_t nvfp4_quantize_weight_shared_workspace_size(int64_t num_groups) {
  if (num_groups <= 0) return 0;
  return nvfp4_weight_ws_bytes(num_groups);
}

mxq_status nvfp4_quantize_weight_shared(
    int64_t num_groups, int num_parts, const void* const* parts,
    const int64_t* part_rows, int64_t K, uint8_t* codes,
    uint8_t* block_scales, float* group_scales, const float* group_scales_in,
    int scale_layout, void* ws, size_t ws_bytes, void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (!valid_layout(scale_layout)) return MXQ_ERR_LAYOUT;
  if (num_groups < 0 || K < 0) return MXQ_ERR_SHAPE;
  if (num_parts < 1 || num_parts > kMaxParts) return MXQ_ERR_ARG;
  if (num_groups == 0 || K == 0) return MXQ_OK;
  if (!parts || !part_rows || !codes || !block_scales || !group_scales)
    return MXQ_ERR_NULL;
  if (K % 16 != 0 || K >= (1ll << 30)) return MXQ_ERR_SHAPE;
  int64_t R = 0;
  for (int i = 0; i < num_parts; ++i) {
    if (part_rows[i] < 0) return MXQ_ERR_SHAPE;
    R += part_rows[i];
  }
  if (R == 0) return MXQ_OK;
  for (int64_t i = 0; i < num_groups * num_parts; ++i) {
    if (part_rows[i % num_parts] > 0 && !parts[i]) return MXQ_ERR_NULL;
    if (!aligned16(parts[i])) return MXQ_ERR_ALIGN;
  }
  if (!aligned16(codes) || !aligned16(block_scales) ||
      !aligned16(group_scales) ||
      (group_scales_in && !aligned16(group_scales_in)))
    return MXQ_ERR_ALIGN;
  if (!group_scales_in) {
    if (!ws) return MXQ_ERR_WORKSPACE;
    if (ws_bytes < nvfp4_quantize_weight_shared_workspace_size(num_groups))
      return MXQ_ERR_WORKSPACE;
    if (!aligned16(ws)) return MXQ_ERR_ALIGN;
  }
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_nvfp4_weight_shared(
      num_groups, num_parts, parts, part_rows, K, codes, block_scales,
      group_scales, group_scales_in, scale_layout == MXQ_SCALE_SWIZZLED,
      static_cast<uint32_t*>(ws), static_cast<cudaStream_t>(stream)));
}

mxq_status dequantize_mxfp8(const uint8_t* codes, const uint8_t* scales,
                            int64_t rows, int64_t cols, int scale_layout,
                            void* y, void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (!valid_layout(scale_layout)) return MXQ_ERR_LAYOUT;
  if (rows < 0 || cols < 0) return MXQ_ERR_SHAPE;
  if (rows == 0 || cols == 0) return MXQ_OK;
  if (!codes || !scales || !y) return MXQ_ERR_NULL;
  if (cols % 32 != 0) return MXQ_ERR_SHAPE;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(y))
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_dequant_mxfp8(codes, scales, rows, cols,
                                        scale_layout == MXQ_SCALE_SWIZZLED, y,
                                        static_cast<cudaStream_t>(stream)));
}

mxq_status dequantize_nvfp4(const uint8_t* codes, const uint8_t* block_scales,
                            const float* S, int s_mode, int64_t batch,
                            int64_t rows, int64_t cols, int scale_layout,
                            void* y, void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (!valid_layout(scale_layout)) return MXQ_ERR_LAYOUT;
  if (s_mode != MXQ_S_PER_ROW && s_mode != MXQ_S_PER_BATCH)
    return MXQ_ERR_LAYOUT;
  if (batch < 0 || rows < 0 || cols < 0) return MXQ_ERR_SHAPE;
  if (batch == 0 || rows == 0 || cols == 0) return MXQ_OK;
  if (!codes || !block_scales || !S || !y) return MXQ_ERR_NULL;
  if (cols % 16 != 0) return MXQ_ERR_SHAPE;
  if (!aligned16(codes) || !aligned16(block_scales) || !aligned16(S) ||
      !aligned16(y))
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_dequant_nvfp4(
      codes, block_scales, S, s_mode == MXQ_S_PER_BATCH, batch, rows, cols,
      scale_layout == MXQ_SCALE_SWIZZLED, y, static_cast<cudaStream_t>(stream)));
}

mxq_status nvfp4_quantize_per_token_rht_sr(const void* x, int64_t T,
                                           int64_t H, int64_t ldx,
                                           uint64_t seed, int flags,
                                           uint8_t* codes,
                                           uint8_t* block_scales,
                                           float* token_scales,
                                           int scale_layout, void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (!valid_layout(scale_layout)) return MXQ_ERR_LAYOUT;
  if (flags < 0 || flags > (MXQ_NVFP4_RHT | MXQ_NVFP4_SR)) return MXQ_ERR_ARG;
  if (T < 0 || H < 0 || ldx < H) return MXQ_ERR_SHAPE;
  if (T == 0 || H == 0) return MXQ_OK;
  if (!x || !codes || !block_scales || !token_scales) return MXQ_ERR_NULL;
  if (H % 16 != 0) return MXQ_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(block_scales) ||
      !aligned16(token_scales) || ldx % 8 != 0)
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_nvfp4_rht_sr(
      x, T, H, ldx, seed, flags, codes, block_scales, token_scales,
      scale_layout == MXQ_SCALE_SWIZZLED, static_cast<cudaStream_t>(stream)));
}

mxq_status fp8_block_quantize(const void* x, int64_t rows, int64_t cols,
                              int64_t ldx, int block_rows, uint8_t* codes,
                              float* scales, void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (block_rows != 1 && block_rows != 128) return MXQ_ERR_ARG;
  if (rows < 0 || cols < 0 || ldx < cols) return MXQ_ERR_SHAPE;
  if (rows == 0 || cols == 0) return MXQ_OK;
  if (!x || !codes || !scales) return MXQ_ERR_NULL;
  if (cols % 128 != 0 || rows % block_rows != 0) return MXQ_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || ldx % 8 != 0)
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_fp8blk_quantize(x, rows, cols, ldx, block_rows,
                                          codes, scales,
                                          static_cast<cudaStream_t>(stream)));
}

mxq_status fp8_block_dequantize(const uint8_t* codes, const float* scales,
                                int64_t rows, int64_t cols, int block_rows,
                                void* y, void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (block_rows != 1 && block_rows != 128) return MXQ_ERR_ARG;
  if (rows < 0 || cols < 0) return MXQ_ERR_SHAPE;
  if (rows == 0 || cols == 0) return MXQ_OK;
  if (!codes || !scales || !y) return MXQ_ERR_NULL;
  if (cols % 128 != 0 || rows % block_rows != 0) return MXQ_ERR_SHAPE;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(y))
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_fp8blk_dequantize(codes, scales, rows, cols,
                                            block_rows, y,
                                            static_cast<cudaStream_t>(stream)));
}

mxq_status fp8_block_requantize_transpose(const uint8_t* codes,
                                          const float* scales, int64_t rows,
                                          int64_t cols, uint8_t* codes_t,
                                          float* scales_t, void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (rows < 0 || cols < 0) return MXQ_ERR_SHAPE;
  if (rows == 0 || cols == 0) return MXQ_OK;
  if (!codes || !scales || !codes_t || !scales_t) return MXQ_ERR_NULL;
  if (rows % 128 != 0 || cols % 128 != 0) return MXQ_ERR_SHAPE;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(codes_t) ||
      !aligned16(scales_t))
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_fp8blk_requant_t(codes, scales, rows, cols, codes_t,
                                           scales_t,
                                           static_cast<cudaStream_t>(stream)));
}

mxq_status mxq_gemm_mxfp8(const uint8_t* a_codes, const uint8_t* a_scales,
                          const uint8_t* bt_codes, const uint8_t* bt_scales,
                          int64_t M, int64_t N, int64_t K, float* C,
                          int64_t ldc, void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (M < 0 || N < 0 || K < 0 || ldc < N) return MXQ_ERR_SHAPE;
  if (M == 0 || N == 0) return MXQ_OK;
  if (!a_codes || !a_scales || !bt_codes || !bt_scales || !C)
    return MXQ_ERR_NULL;
  if (M % 128 != 0 || N % 128 != 0 || K % 128 != 0 || K == 0)
    return MXQ_ERR_SHAPE;
  if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31))
    return MXQ_ERR_SHAPE;
  if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(bt_codes) ||
      !aligned16(bt_scales) || !aligned16(C) || ldc % 4 != 0)
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_gemm_mxfp8(a_codes, a_scales, bt_codes, bt_scales, M,
                                     N, K, C, ldc,
                                     static_cast<cudaStream_t>(stream)));
}

mxq_status mxq_gemm_bf16_mxfp8(const void* a, int64_t lda,
                               const uint8_t* bt_codes,
                               const uint8_t* bt_scales, int64_t M, int64_t N,
                               int64_t K, float* C, int64_t ldc, void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (M < 0 || N < 0 || K < 0 || lda < K || ldc < N) return MXQ_ERR_SHAPE;
  if (M == 0 || N == 0) return MXQ_OK;
  if (!a || !bt_codes || !bt_scales || !C) return MXQ_ERR_NULL;
  if (M % 128 != 0 || N % 128 != 0 || K % 64 != 0 || K == 0)
    return MXQ_ERR_SHAPE;
  if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31))
    return MXQ_ERR_SHAPE;
  if (!aligned16(a) || !aligned16(bt_codes) || !aligned16(bt_scales) ||
      !aligned16(C) || lda % 8 != 0 || ldc % 4 != 0)
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_gemm_bf16_mxfp8(a, lda, bt_codes, bt_scales, M, N, K,
                                          C, ldc,
                                          static_cast<cudaStream_t>(stream)));
}

mxq_status mxq_gemm_nvfp4_grouped(
    const uint8_t* a_codes, const uint8_t* a_scales, const float* a_token_scales,
    const int64_t* group_offsets, int64_t num_groups, const uint8_t* w_codes,
    const uint8_t* w_scales, const float* w_group_scales, int64_t N, int64_t K,
    float* C, int64_t ldc, void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (num_groups < 0 || num_groups > 256 || N < 0 || K < 0 || ldc < N)
    return MXQ_ERR_SHAPE;
  if (num_groups == 0 || N == 0) return MXQ_OK;
  if (!group_offsets) return MXQ_ERR_NULL;
  if (group_offsets[0] != 0) return MXQ_ERR_SHAPE;
  for (int64_t g = 0; g < num_groups; ++g)
    if (group_offsets[g + 1] < group_offsets[g] ||
        group_offsets[g + 1] % 128 != 0)
      return MXQ_ERR_SHAPE;
  if (group_offsets[num_groups] == 0) return MXQ_OK;
  if (!a_codes || !a_scales || !a_token_scales || !w_codes || !w_scales ||
      !w_group_scales || !C)
    return MXQ_ERR_NULL;
  if (N % 128 != 0 || K % 256 != 0 || K == 0) return MXQ_ERR_SHAPE;
  if (group_offsets[num_groups] >= (1ll << 31) || num_groups * N >= (1ll << 31) ||
      K >= (1ll << 31))
    return MXQ_ERR_SHAPE;
  if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(w_codes) ||
      !aligned16(w_scales) || !aligned16(C) || ldc % 4 != 0)
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_gemm_nvfp4_grouped(
      a_codes, a_scales, a_token_scales, group_offsets, num_groups, w_codes,
      w_scales, w_group_scales, N, K, C, ldc,
      static_cast<cudaStream_t>(stream)));
}

mxq_status mxq_moe_gate_up_swiglu_nvfp4(
    const uint8_t* a_codes, const uint8_t* a_scales, const float* a_token_scales,
    const int64_t* group_offsets, int64_t num_groups, const uint8_t* w_codes,
    const uint8_t* w_scales, const float* w_group_scales, int64_t F, int64_t K,
    void* h, int64_t ldh, void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (num_groups < 0 || num_groups > 256 || F < 0 || K < 0 || ldh < F)
    return MXQ_ERR_SHAPE;
  if (num_groups == 0 || F == 0) return MXQ_OK;
  if (!group_offsets) return MXQ_ERR_NULL;
  if (group_offsets[0] != 0) return MXQ_ERR_SHAPE;
  for (int64_t g = 0; g < num_groups; ++g)
    if (group_offsets[g + 1] < group_offsets[g] ||
        group_offsets[g + 1] % 128 != 0)
      return MXQ_ERR_SHAPE;
  if (group_offsets[num_groups] == 0) return MXQ_OK;
  if (!a_codes || !a_scales || !a_token_scales || !w_codes || !w_scales ||
      !w_group_scales || !h)
    return MXQ_ERR_NULL;
  if (F % 128 != 0 || K % 256 != 0 || K == 0) return MXQ_ERR_SHAPE;
  if (group_offsets[num_groups] >= (1ll << 31) ||
      num_groups * 2 * F >= (1ll << 31) || K >= (1ll << 31))
    return MXQ_ERR_SHAPE;
  if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(w_codes) ||
      !aligned16(w_scales) || !aligned16(h) || ldh % 8 != 0)
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_moe_gate_up_swiglu(
      a_codes, a_scales, a_token_scales, group_offsets, num_groups, w_codes,
      w_scales, w_group_scales, F, K, h, ldh,
      static_cast<cudaStream_t>(stream)));
}

// Shared checks of the gathered grouped GEMMs: the per-token operand x
// [T_src rows] with linear block scales, int32 row_index [rows].
static mxq_status check_gather(const uint8_t* x_codes, const uint8_t* x_scales,
                               const float* x_s, int64_t T_src,
                               const int32_t* row_index) {
  if (T_src <= 0 || T_src >= (1ll << 31)) return MXQ_ERR_SHAPE;
  if (!x_codes || !x_scales || !x_s || !row_index) return MXQ_ERR_NULL;
  if (!aligned16(x_codes) || !aligned16(x_scales) ||
      (reinterpret_cast<uintptr_t>(row_index) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(x_s) & 3u) != 0)
    return MXQ_ERR_ALIGN;
  return MXQ_OK;
}

mxq_status mxq_gemm_nvfp4_grouped_gather(
    const uint8_t* x_codes, const uint8_t* x_scales, const float* x_token_scales,
    int64_t T_src, const int32_t* row_index, const int64_t* group_offsets,
    int64_t num_groups, const uint8_t* w_codes, const uint8_t* w_scales,
    const float* w_group_scales, int64_t N, int64_t K, float* C, int64_t ldc,
    void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (num_groups < 0 || num_groups > 256 || N < 0 || K < 0 || ldc < N)
    return MXQ_ERR_SHAPE;
  if (num_groups == 0 || N == 0) return MXQ_OK;
  if (!group_offsets) return MXQ_ERR_NULL;
  if (group_offsets[0] != 0) return MXQ_ERR_SHAPE;
  for (int64_t g = 0; g < num_groups; ++g)
    if (group_offsets[g + 1] < group_offsets[g] ||
        group_offsets[g + 1] % 128 != 0)
      return MXQ_ERR_SHAPE;
  if (group_offsets[num_groups] == 0) return MXQ_OK;
  const mxq_status st =
      check_gather(x_codes, x_scales, x_token_scales, T_src, row_index);
  if (st != MXQ_OK) return st;
  if (!w_codes || !w_scales || !w_group_scales || !C) return MXQ_ERR_NULL;
  if (N % 128 != 0 || K % 256 != 0 || K == 0) return MXQ_ERR_SHAPE;
  if (group_offsets[num_groups] >= (1ll << 31) || num_groups * N >= (1ll << 31) ||
      K >= (1ll << 31))
    return MXQ_ERR_SHAPE;
  if (!aligned16(w_codes) || !aligned16(w_scales) || !aligned16(C) ||
      ldc % 4 != 0)
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_gemm_nvfp4_grouped(
      x_codes, x_scales, x_token_scales, group_offsets, num_groups, w_codes,
      w_scales, w_group_scales, N, K, C, ldc,
      static_cast<cudaStream_t>(stream), row_index, T_src));
}

mxq_status mxq_moe_gate_up_swiglu_nvfp4_gather(
    const uint8_t* x_codes, const uint8_t* x_scales, const float* x_token_scales,
    int64_t T_src, const int32_t* row_index, const int64_t* group_offsets,
    int64_t num_groups, const uint8_t* w_codes, const uint8_t* w_scales,
    const float* w_group_scales, int64_t F, int64_t K, void* h, int64_t ldh,
    void* stream) {
  const int fm = fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (num_groups < 0 || num_groups > 256 || F < 0 || K < 0 || ldh < F)
    return MXQ_ERR_SHAPE;
  if (num_groups == 0 || F == 0) return MXQ_OK;
  if (!group_offsets) return MXQ_ERR_NULL;
  if (group_offsets[0] != 0) return MXQ_ERR_SHAPE;
  for (int64_t g = 0; g < num_groups; ++g)
    if (group_offsets[g + 1] < group_offsets[g] ||
        group_offsets[g + 1] % 128 != 0)
      return MXQ_ERR_SHAPE;
  if (group_offsets[num_groups] == 0) return MXQ_OK;
  const mxq_status st =
      check_gather(x_codes, x_scales, x_token_scales, T_src, row_index);
  if (st != MXQ_OK) return st;
  if (!w_codes || !w_scales || !w_group_scales || !h) return MXQ_ERR_NULL;
  if (F % 128 != 0 || K % 256 != 0 || K == 0) return MXQ_ERR_SHAPE;
  if (group_offsets[num_groups] >= (1ll << 31) ||
      num_groups * 2 * F >= (1ll << 31) || K >= (1ll << 31))
    return MXQ_ERR_SHAPE;
  if (!aligned16(w_codes) || !aligned16(w_scales) || !aligned16(h) ||
      ldh % 8 != 0)
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  return from_cuda(launch_moe_gate_up_swiglu(
      x_codes, x_scales, x_token_scales, group_offsets, num_groups, w_codes,
      w_scales, w_group_scales, F, K, h, ldh,
      static_cast<cudaStream_t>(stream), row_index, T_src));
}

}  // extern "C"
