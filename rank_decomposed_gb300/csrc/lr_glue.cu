// Memory-bound kernels around the GEMMs: the remap gather/scatter of the
// preparation and graph-replay stages (DeInfer, English summary page section
// 2.C), RMSNorm, SiLU-GLU and the bf16 <-> fp32 conversions of the residual
// stream.  All use 16-byte vector accesses; reductions run in a fixed order so
// every result is deterministic.
#include <cuda_bf16.h>

#include <cstring>

#include "lr_ptx.cuh"

namespace lr {
namespace {

// Launch with programmatic dependent launch when enabled.  Every kernel here
// lets its dependents launch first (they only prefetch weights before their
// own wait) and calls pdl_wait() before it touches memory written by earlier
// kernels.
template <typename... KArgs, typename... Args>
lr_status launch(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t s, const char* what,
                 Args... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl_enabled()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return LR_OK;
}

__device__ __forceinline__ int clamp_active(const int32_t* n_active, int64_t cap) {
  int n = *n_active;
  if (n < 0) n = 0;
  if (n > cap) n = static_cast<int>(cap);
  return n;
}

// Rows of the remap table one CTA copies.  Each warp copies whole rows with
// 16-byte vectors, so a run of consecutive pool rows (the contiguous blocks of
// the pages' scan) is read as one contiguous range, and rows of a few hundred
// bytes (KV latents) do not cost a CTA each.
constexpr int kCopyRows = 32;

// buf[i] = pool[remap[i]] for i < n_active, zero rows otherwise.
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ pool, int64_t pool_rows,
                                                     int64_t row_vecs, const int32_t* __restrict__ remap,
                                                     const int32_t* __restrict__ n_active,
                                                     uint4* __restrict__ buf, int64_t cap,
                                                     int32_t* status) {
  __shared__ int64_t src_row[kCopyRows];
  pdl_launch_dependents();
  pdl_wait();
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kCopyRows;
  const int n = clamp_active(n_active, cap);
  if (threadIdx.x < kCopyRows) {
    const int64_t i = i0 + threadIdx.x;
    int64_t j = -1;
    if (i < n) {
      j = remap[i];
      if (j < 0 || j >= pool_rows) {
        report_status(status, LR_ERR_REMAP_RANGE);
        j = -1;
      }
    }
    src_row[threadIdx.x] = j;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = cap - i0 < kCopyRows ? static_cast<int>(cap - i0) : kCopyRows;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int r = warp; r < rows; r += 8) {
    uint4* dst = buf + (i0 + r) * row_vecs;
    const int64_t j = src_row[r];
    if (j >= 0) {
      const uint4* src = pool + j * row_vecs;
      for (int64_t v = lane; v < row_vecs; v += 32) dst[v] = src[v];
    } else {
      for (int64_t v = lane; v < row_vecs; v += 32) dst[v] = z;
    }
  }
}

// pool[remap[i]] = buf[i] for i < n_active.
__global__ void __launch_bounds__(256) scatter_kernel(const uint4* __restrict__ buf,
                                                      const int32_t* __restrict__ remap,
                                                      const int32_t* __restrict__ n_active,
                                                      uint4* __restrict__ pool, int64_t pool_rows,
                                                      int64_t row_vecs, int64_t cap,
                                                      int32_t* status) {
  __shared__ int64_t dst_row[kCopyRows];
  pdl_launch_dependents();
  pdl_wait();
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kCopyRows;
  const int n = clamp_active(n_active, cap);
  if (threadIdx.x < kCopyRows) {
    const int64_t i = i0 + threadIdx.x;
    int64_t j = -1;
    if (i < n) {
      j = remap[i];
      if (j < 0 || j >= pool_rows) {
        report_status(status, LR_ERR_REMAP_RANGE);
        j = -1;
      }
    }
    dst_row[threadIdx.x] = j;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = cap - i0 < kCopyRows ? static_cast<int>(cap - i0) : kCopyRows;
  for (int r = warp; r < rows; r += 8) {
    const int64_t j = dst_row[r];
    if (j < 0) continue;
    const uint4* src = buf + (i0 + r) * row_vecs;
    uint4* dst = pool + j * row_vecs;
    for (int64_t v = lane; v < row_vecs; v += 32) dst[v] = src[v];
  }
}

// out[m] = bf16(h[m] / sqrt(mean(h[m]^2) + eps)); one CTA per row.  Each
// thread keeps its (up to 8) float4 of the row in registers, so the row is
// read once and all loads are in flight together.
constexpr int kNormVec = 8;

__global__ void __launch_bounds__(256) rmsnorm_kernel(const float4* __restrict__ h,
                                                      uint2* __restrict__ out, int d4, float eps) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float part[8];
  const int64_t row = blockIdx.x;
  const float4* x = h + row * d4;
  float4 v[kNormVec];
#pragma unroll
  for (int j = 0; j < kNormVec; ++j) {
    const int idx = threadIdx.x + j * 256;
    v[j] = idx < d4 ? x[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kNormVec; ++j) ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += part[w];
  const float inv = 1.0f / sqrtf(tot / static_cast<float>(4 * d4) + eps);
  uint2* y = out + row * d4;
#pragma unroll
  for (int j = 0; j < kNormVec; ++j) {
    const int idx = threadIdx.x + j * 256;
    if (idx < d4) {
      uint2 w;
      w.x = static_cast<uint32_t>(f32_to_bf16_rn(v[j].x * inv)) |
            (static_cast<uint32_t>(f32_to_bf16_rn(v[j].y * inv)) << 16);
      w.y = static_cast<uint32_t>(f32_to_bf16_rn(v[j].z * inv)) |
            (static_cast<uint32_t>(f32_to_bf16_rn(v[j].w * inv)) << 16);
      y[idx] = w;
    }
  }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// a = bf16(silu(g) * u), 8 elements per vector.
__global__ void __launch_bounds__(256) silu_mul_kernel(const uint4* __restrict__ g,
                                                       const uint4* __restrict__ u,
                                                       uint4* __restrict__ a, int64_t n8) {
  pdl_launch_dependents();
  pdl_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 gv = g[i];
    const uint4 uv = u[i];
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
    uint32_t ow[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float g0 = bf16_to_f32(static_cast<uint16_t>(gw[j] & 0xFFFFu));
      const float g1 = bf16_to_f32(static_cast<uint16_t>(gw[j] >> 16));
      const float u0 = bf16_to_f32(static_cast<uint16_t>(uw[j] & 0xFFFFu));
      const float u1 = bf16_to_f32(static_cast<uint16_t>(uw[j] >> 16));
      ow[j] = static_cast<uint32_t>(f32_to_bf16_rn(silu_f(g0) * u0)) |
              (static_cast<uint32_t>(f32_to_bf16_rn(silu_f(g1) * u1)) << 16);
    }
    a[i] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
  }
}

// out = fp32(in), 8 bf16 elements per vector.
__global__ void __launch_bounds__(256) widen_kernel(const uint4* __restrict__ in,
                                                    float4* __restrict__ out, int64_t n8) {
  pdl_launch_dependents();
  pdl_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = in[i];
    out[2 * i] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                             __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
    out[2 * i + 1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u),
                                 __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
  }
}

__global__ void __launch_bounds__(256) narrow_kernel(const float4* __restrict__ in,
                                                     uint4* __restrict__ out, int64_t n8) {
  pdl_launch_dependents();
  pdl_wait();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = in[2 * i];
    const float4 b = in[2 * i + 1];
    uint4 w;
    w.x = static_cast<uint32_t>(f32_to_bf16_rn(a.x)) | (static_cast<uint32_t>(f32_to_bf16_rn(a.y)) << 16);
    w.y = static_cast<uint32_t>(f32_to_bf16_rn(a.z)) | (static_cast<uint32_t>(f32_to_bf16_rn(a.w)) << 16);
    w.z = static_cast<uint32_t>(f32_to_bf16_rn(b.x)) | (static_cast<uint32_t>(f32_to_bf16_rn(b.y)) << 16);
    w.w = static_cast<uint32_t>(f32_to_bf16_rn(b.z)) | (static_cast<uint32_t>(f32_to_bf16_rn(b.w)) << 16);
    out[i] = w;
  }
}

// One stack row: xbuf[i] = pool[remap[i]] (zero past n_active), h[i] = widen.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ pool, int64_t pool_rows,
                                                          int d8, const int32_t* __restrict__ remap,
                                                          const int32_t* __restrict__ n_active,
                                                          uint4* __restrict__ xbuf, float4* __restrict__ h,
                                                          int64_t cap, int32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t i = blockIdx.x;
  const int n = clamp_active(n_active, cap);
  const uint4* src = nullptr;
  if (i < n) {
    const int64_t j = remap[i];
    if (j >= 0 && j < pool_rows)
      src = pool + j * d8;
    else if (threadIdx.x == 0)
      report_status(status, LR_ERR_REMAP_RANGE);
  }
  for (int v = threadIdx.x; v < d8; v += 256) {
    const uint4 w = src != nullptr ? src[v] : make_uint4(0, 0, 0, 0);
    xbuf[i * d8 + v] = w;
    h[(i * d8 + v) * 2] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                                      __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
    h[(i * d8 + v) * 2 + 1] = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u),
                                          __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
  }
}

// One stack row: ybuf[i] = bf16(h[i]); pool[remap[i]] = ybuf[i] for i < n_active.
__global__ void __launch_bounds__(256) scatter_rows_kernel(const float4* __restrict__ h, int d8,
                                                           uint4* __restrict__ ybuf,
                                                           const int32_t* __restrict__ remap,
                                                           const int32_t* __restrict__ n_active,
                                                           uint4* __restrict__ pool, int64_t pool_rows,
                                                           int64_t cap, int32_t* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t i = blockIdx.x;
  const int n = clamp_active(n_active, cap);
  uint4* dst = nullptr;
  if (i < n) {
    const int64_t j = remap[i];
    if (j >= 0 && j < pool_rows)
      dst = pool + j * d8;
    else if (threadIdx.x == 0)
      report_status(status, LR_ERR_REMAP_RANGE);
  }
  for (int v = threadIdx.x; v < d8; v += 256) {
    const float4 a = h[(i * d8 + v) * 2], b = h[(i * d8 + v) * 2 + 1];
    uint4 w;
    w.x = static_cast<uint32_t>(f32_to_bf16_rn(a.x)) | (static_cast<uint32_t>(f32_to_bf16_rn(a.y)) << 16);
    w.y = static_cast<uint32_t>(f32_to_bf16_rn(a.z)) | (static_cast<uint32_t>(f32_to_bf16_rn(a.w)) << 16);
    w.z = static_cast<uint32_t>(f32_to_bf16_rn(b.x)) | (static_cast<uint32_t>(f32_to_bf16_rn(b.y)) << 16);
    w.w = static_cast<uint32_t>(f32_to_bf16_rn(b.z)) | (static_cast<uint32_t>(f32_to_bf16_rn(b.w)) << 16);
    ybuf[i * d8 + v] = w;
    if (dst != nullptr) dst[v] = w;
  }
}

int elementwise_grid(int64_t n_vec) {
  const int64_t per = 256;
  int64_t blocks = (n_vec + per - 1) / per;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

}  // namespace

lr_status launch_gather(const void* pool, int64_t pool_rows, int64_t row_bytes,
                        const int32_t* remap, const int32_t* n_active, void* buf, int64_t cap,
                        int32_t* status, cudaStream_t s) {
  if (cap == 0) return LR_OK;
  return launch(gather_kernel, dim3(static_cast<unsigned>((cap + kCopyRows - 1) / kCopyRows)), dim3(256), s,
                "gather",
                static_cast<const uint4*>(pool), pool_rows, row_bytes / 16, remap, n_active,
                static_cast<uint4*>(buf), cap, status);
}

lr_status launch_gather_rows(const void* pool, int64_t pool_rows, int d, const int32_t* remap,
                             const int32_t* n_active, void* xbuf, float* h, int64_t cap,
                             int32_t* status, cudaStream_t s) {
  if (cap == 0) return LR_OK;
  return launch(gather_rows_kernel, dim3(static_cast<unsigned>(cap)), dim3(256), s, "gather_rows",
                static_cast<const uint4*>(pool), pool_rows, d / 8, remap, n_active,
                static_cast<uint4*>(xbuf), reinterpret_cast<float4*>(h), cap, status);
}

lr_status launch_scatter_rows(const float* h, void* ybuf, const int32_t* remap,
                              const int32_t* n_active, void* pool, int64_t pool_rows, int d,
                              int64_t cap, int32_t* status, cudaStream_t s) {
  if (cap == 0) return LR_OK;
  return launch(scatter_rows_kernel, dim3(static_cast<unsigned>(cap)), dim3(256), s, "scatter_rows",
                reinterpret_cast<const float4*>(h), d / 8, static_cast<uint4*>(ybuf), remap, n_active,
                static_cast<uint4*>(pool), pool_rows, cap, status);
}

lr_status launch_scatter(const void* buf, const int32_t* remap, const int32_t* n_active,
                         void* pool, int64_t pool_rows, int64_t row_bytes, int64_t cap,
                         int32_t* status, cudaStream_t s) {
  if (cap == 0) return LR_OK;
  return launch(scatter_kernel, dim3(static_cast<unsigned>((cap + kCopyRows - 1) / kCopyRows)), dim3(256), s,
                "scatter",
                static_cast<const uint4*>(buf), remap, n_active, static_cast<uint4*>(pool),
                pool_rows, row_bytes / 16, cap, status);
}

lr_status launch_rmsnorm(const float* h, void* out_bf16, int64_t M, int d, float eps,
                         cudaStream_t s) {
  if (M == 0) return LR_OK;
  return launch(rmsnorm_kernel, dim3(static_cast<unsigned>(M)), dim3(256), s, "rmsnorm",
                reinterpret_cast<const float4*>(h), static_cast<uint2*>(out_bf16), d / 4, eps);
}

lr_status launch_silu_mul(const void* g, const void* u, void* out, int64_t M, int d,
                          cudaStream_t s) {
  const int64_t n8 = M * d / 8;
  if (n8 == 0) return LR_OK;
  return launch(silu_mul_kernel, dim3(elementwise_grid(n8)), dim3(256), s, "silu_mul",
                static_cast<const uint4*>(g), static_cast<const uint4*>(u),
                static_cast<uint4*>(out), n8);
}

lr_status launch_widen(const void* in_bf16, float* out, int64_t n, cudaStream_t s) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return LR_OK;
  return launch(widen_kernel, dim3(elementwise_grid(n8)), dim3(256), s, "widen",
                static_cast<const uint4*>(in_bf16), reinterpret_cast<float4*>(out), n8);
}

lr_status launch_narrow(const float* in, void* out_bf16, int64_t n, cudaStream_t s) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return LR_OK;
  return launch(narrow_kernel, dim3(elementwise_grid(n8)), dim3(256), s, "narrow",
                reinterpret_cast<const float4*>(in), static_cast<uint4*>(out_bf16), n8);
}

// out[c][r] = in[r][c] for a bf16 [rows][cols] matrix (both multiples of 64):
// one 64 x 64 tile per CTA through shared memory, bit-exact.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* __restrict__ in, int rows,
                                                              int cols, uint16_t* __restrict__ out) {
  __shared__ uint16_t tile[64][66];
  pdl_wait();
  pdl_launch_dependents();
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
  for (int i = ty; i < 64; i += 4) tile[i][tx] = in[static_cast<int64_t>(r0 + i) * cols + c0 + tx];
  __syncthreads();
  for (int i = ty; i < 64; i += 4) out[static_cast<int64_t>(c0 + i) * rows + r0 + tx] = tile[tx][i];
}

lr_status launch_transpose_bf16(const void* in, int rows, int cols, void* out, cudaStream_t s) {
  return launch(transpose_bf16_kernel, dim3(cols / 64, rows / 64), dim3(256), s, "transpose",
                static_cast<const uint16_t*>(in), rows, cols, static_cast<uint16_t*>(out));
}

}  // namespace lr
