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

// Size of the static scratch: t = x A_r in bf16 needs 2 * M * r bytes.
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

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

lr_status bad(const char* msg) {
  set_error("linear_noalloc: %s", msg);
  return LR_ERR_INVALID_ARG;
}

}  // namespace
}  // namespace lr

using namespace lr;

extern "C" lr_status lr_linear_forward_noalloc(const void* x, int64_t ldx, void* y, int64_t ldy,
                                               lr_dtype y_dtype, int64_t M, const lr_factor* f,
                                               int32_t* dev_status, lr_stream s) {
  if (f == nullptr) return bad("null factor");
  if (f->d_in <= 0 || f->d_out <= 0 || f->r <= 0) return bad("non-positive factor dims");
  if (f->d_in % 64 || f->d_out % 64 || f->r % 64) {
    set_error("linear_noalloc: d_in=%d d_out=%d r=%d must be multiples of 64", f->d_in, f->d_out,
              f->r);
    return LR_ERR_UNSUPPORTED;
  }
  if (f->At == nullptr || f->Bt == nullptr) return bad("null factor pointer");
  if (!aligned16(f->At) || !aligned16(f->Bt)) return bad("factors not 16-byte aligned");
  if (M < 0 || M > (int64_t(1) << 31) - 1) return bad("bad M");
  if (M == 0) return LR_OK;
  if (x == nullptr || y == nullptr) return bad("null pointer");
  if (y_dtype != LR_BF16 && y_dtype != LR_F32) return bad("bad y dtype");
  if (ldx < f->d_in || ldx % 8 || !aligned16(x))
    return bad("x must be 16-byte aligned with ldx >= d_in, ldx % 8 == 0");
  if (ldy < f->d_out) return bad("ldy < d_out");
  if (M > kDecodeMaxRows && (!aligned16(y) || ldy % 8))
    return bad("y must be 16-byte aligned with ldy % 8 == 0");
  const size_t need = static_cast<size_t>(M) * static_cast<size_t>(f->r) * 2;
  if (need > kNoAllocScratchBytes) {
    set_error("linear_noalloc: M * r * 2 = %zu bytes of scratch needed, the static array holds "
              "%zu bytes (use lr_linear_forward with a workspace)",
              need, kNoAllocScratchBytes);
    return LR_ERR_UNSUPPORTED;
  }
  void* t = nullptr;
  lr_status st = scratch_address(&t);
  if (st != LR_OK) return st;
  st = ensure_configured();
  if (st != LR_OK) return st;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
  GemmOp down;
  memset(&down, 0, sizeof(down));
  down.W = f->At;
  down.N = f->r;
  down.K = f->d_in;
  down.ldw = f->d_in;
  down.act = x;
  down.ld_act = ldx;
  down.act_cols = f->d_in;
  down.epi = EPI_STORE_BF16;
  down.out = t;
  down.ldo = f->r;
  GemmOp up;
  memset(&up, 0, sizeof(up));
  up.W = f->Bt;
  up.N = f->d_out;
  up.K = f->r;
  up.ldw = f->r;
  up.act = t;
  up.ld_act = f->r;
  up.act_cols = f->r;
  up.epi = y_dtype == LR_BF16 ? EPI_STORE_BF16 : EPI_STORE_F32;
  up.out = y;
  up.ldo = ldy;
  if (M <= kDecodeMaxRows) {
    st = launch_decode(static_cast<int>(M), &down, 1, dev_status, cs);
    if (st != LR_OK) return st;
    return launch_decode(static_cast<int>(M), &up, 1, dev_status, cs);
  }
  st = launch_prefill(M, down, dev_status, cs);
  if (st != LR_OK) return st;
  return launch_prefill(M, up, dev_status, cs);
}
