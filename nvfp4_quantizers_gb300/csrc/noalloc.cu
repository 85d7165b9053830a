// noalloc.cu -- nvfp4_quantize_weight_shared_noalloc: the shared-scale
// NVFP4 weight quantizer without a caller-provided workspace.
//
// Some callers cannot allocate device memory at all: code that runs as a
// plug-in inside a host framework that owns every device allocation and
// gives its plug-ins no allocator, and latency-critical loops in which a
// cudaMalloc (which may synchronize the device) is not allowed.  Such a
// caller can still hand over its inputs and outputs, but not the small
// scratch buffer that nvfp4_quantize_weight_shared needs for the per-group
// amax words.  This entry point keeps that scratch in a fixed array in the
// library's own device memory instead.
//
//  * The scratch is a file-scope device array of 64 + 2 * kNoAllocMaxGroups
//    32-bit words (32.25 KiB: task counters, one amax word and one
//    progress counter per group).  Every GPU that loads the library holds
//    it until the process exits.
//  * Host code cannot use the array's name as a device address (on the
//    host it only stands in for the symbol).  The first call on a device
//    looks the address up with cudaGetSymbolAddress, with that device
//    current, and caches it together with the identity of the device's
//    current context; a call that finds another context (after a
//    cudaDeviceReset, say) looks the address up again.  Make the first call
//    on a device, and the first after a reset, before any stream capture.
//  * All calls share the one array and it keeps the last call's contents:
//    the words a call uses are cleared (cudaMemsetAsync on the call's
//    stream) before its kernel runs.  Calls whose kernels overlap on
//    the GPU (different streams, no ordering between them) race on the
//    array; order them on one stream.
//  * Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/mxq.h"
#include "launch.h"

namespace mxq {

namespace {

constexpr int64_t kNoAllocMaxGroups = 4096;
// 256-byte header (task counters) + an amax word and a progress counter per
// group.
constexpr int64_t kNoAllocWords = 64 + 2 * kNoAllocMaxGroups;
static __device__ __align__(256) uint32_t g_noalloc_amax[kNoAllocWords];

constexpr int kMaxDev = 64;
std::mutex g_mu;
uint32_t* g_addr[kMaxDev] = {};
unsigned long long g_ctx_id[kMaxDev] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 if it cannot be
// read), from the driver entry points cuCtxGetCurrent and cuCtxGetId.
unsigned long long current_ctx_id() {
  static std::once_flag once;
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur && get_id && get_cur(&ctx) == CUDA_SUCCESS && ctx &&
      get_id(ctx, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

// Device address of g_noalloc_amax on the current device: looked up with
// cudaGetSymbolAddress on the first call on the device, and again when the
// device's context is no longer the one the cached address belongs to.
cudaError_t noalloc_scratch(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  // 0 when no context is current yet (the lookup below creates it)
  const unsigned long long ctx = current_ctx_id();
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev] || ctx == 0 || ctx != g_ctx_id[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_amax);
    if (e != cudaSuccess) return e;
    g_addr[dev] = static_cast<uint32_t*>(p);
    g_ctx_id[dev] = current_ctx_id();   // the context the lookup used
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

bool is_aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace

}  // namespace mxq

using namespace mxq;

extern "C" {

int64_t nvfp4_quantize_weight_shared_noalloc_max_groups(void) {
  return kNoAllocMaxGroups;
}

mxq_status nvfp4_quantize_weight_shared_noalloc(
    int64_t num_groups, int num_parts, const void* const* parts,
    const int64_t* part_rows, int64_t K, uint8_t* codes,
    uint8_t* block_scales, float* group_scales, const float* group_scales_in,
    int scale_layout, void* stream) {
  const int fm = host_fault_mode();
  if (fm == 2) return MXQ_ERR_ARG;
  if (scale_layout != MXQ_SCALE_LINEAR && scale_layout != MXQ_SCALE_SWIZZLED)
    return MXQ_ERR_LAYOUT;
  if (num_groups < 0 || K < 0) return MXQ_ERR_SHAPE;
  if (num_groups > kNoAllocMaxGroups) return MXQ_ERR_SHAPE;
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
    if (!is_aligned16(parts[i])) return MXQ_ERR_ALIGN;
  }
  if (!is_aligned16(codes) || !is_aligned16(block_scales) ||
      !is_aligned16(group_scales) ||
      (group_scales_in && !is_aligned16(group_scales_in)))
    return MXQ_ERR_ALIGN;
  if (fm == 1) return MXQ_ERR_CUDA;
  uint32_t* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return MXQ_ERR_CUDA;
  cudaError_t e = launch_nvfp4_weight_shared(
      num_groups, num_parts, parts, part_rows, K, codes, block_scales,
      group_scales, group_scales_in, scale_layout == MXQ_SCALE_SWIZZLED,
      scratch, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
}

}  // extern "C"
