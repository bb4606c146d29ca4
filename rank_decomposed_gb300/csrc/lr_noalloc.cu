// lr_linear_forward_noalloc: the factorized linear with its scratch in a
// static device array, for callers that cannot allocate device memory.
//
// lr_linear_forward needs a caller-provided workspace for the rank-r
// intermediate t = x A_r.  Some callers have no way to provide one: code that
// runs where cudaMalloc is not allowed or not wanted (an allocator-free
// embedded runtime, a plugin handed only raw tensors and a stream, a serving
// loop whose memory is fixed at start-up, or code that must not risk the
// implicit device synchronisation cudaMalloc can cause).  This entry point
// takes the same inputs and outputs and keeps t in a file-scope __device__
// array instead.  Every GPU that loads the library holds that array until the
// process exits.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "lr_internal.h"

namespace lr {
namespace {

// Size of the static scratch: t = x A_r in bf16 needs 2 * M * r bytes (and,
// above 256 rows, the prefill band counters after it).
constexpr size_t kNoAllocScratchBytes = LR_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device, looked up once
// per device.  (The symbol's name in host code is only a host-side stand-in.)
lr_status scratch_address(void** out) {
  static void* addr[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "linear_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("linear_noalloc: device ordinal %d outside the supported range", dev);
    return LR_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "linear_noalloc: cudaGetSymbolAddress");
    addr[dev] = p;
  }
  *out = addr[dev];
  return LR_OK;
}

}  // namespace
}  // namespace lr

using namespace lr;

extern "C" lr_status lr_linear_forward_noalloc(const void* x, int64_t ldx, void* y, int64_t ldy,
                                               lr_dtype y_dtype, int64_t M, const lr_factor* f,
                                               int32_t* dev_status, lr_stream s) {
  // The same checks, the same kernels and the same t layout as
  // lr_linear_forward; only the home of t differs.
  lr_status st = check_factor(f, "linear_noalloc");
  if (st != LR_OK) return st;
  if (M < 0 || M > (int64_t(1) << 31) - 1) {
    set_error("linear_noalloc: bad M");
    return LR_ERR_INVALID_ARG;
  }
  if (M == 0) return LR_OK;
  st = check_linear_io("linear_noalloc", x, ldx, y, ldy, y_dtype, M, f);
  if (st != LR_OK) return st;
  const size_t need = lr_linear_workspace_bytes(M, f);
  if (need > kNoAllocScratchBytes) {
    set_error("linear_noalloc: %zu bytes of scratch needed (lr_linear_workspace_bytes), the static "
              "array holds %zu bytes (use lr_linear_forward with a workspace)",
              need, kNoAllocScratchBytes);
    return LR_ERR_UNSUPPORTED;
  }
  void* t = nullptr;
  st = scratch_address(&t);
  if (st != LR_OK) return st;
  return enqueue_linear(x, ldx, y, ldy, y_dtype, M, f, t, dev_status,
                        reinterpret_cast<cudaStream_t>(s));
}
