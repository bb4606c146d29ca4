// Device implementation of the seeded input generator defined in
// synth/__init__.py (SplitMix64 words, Irwin-Hall-12 variates, fp64 scaling,
// round-to-nearest-even to bf16).  It produces the same bits as the numpy
// implementation so that large inputs (whole factor stacks) can be made on the
// GPU while the oracle regenerates any slice of them on the CPU.  Input
// generation only: nothing here belongs to the computation under test.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t fmix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint16_t f64_to_bf16_rne(double v) {
  const uint64_t b = static_cast<uint64_t>(__double_as_longlong(v));
  const uint64_t sign = b >> 63;
  const uint64_t mag = b & 0x7FFFFFFFFFFFFFFFull;
  if (mag == 0) return static_cast<uint16_t>(sign << 15);
  const uint64_t lsb = (mag >> 45) & 1ull;
  const uint64_t r = (mag + ((1ull << 44) - 1) + lsb) >> 45;
  const int64_t exp8 = static_cast<int64_t>(r >> 7) - 1023 + 127;
  if (exp8 <= 0 || exp8 >= 255) return 0x7FC0;  // outside the generator's range: NaN marker
  return static_cast<uint16_t>((sign << 15) | (static_cast<uint64_t>(exp8) << 7) | (r & 0x7Full));
}

__global__ void bf16_normal_kernel(uint16_t* __restrict__ out, int64_t rows, int64_t cols,
                                   uint64_t key, double stdv, const double* __restrict__ col_scale) {
  const int64_t n = rows * cols;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint64_t base = key + static_cast<uint64_t>(i) * (6ull * kGolden);
    int64_t s = 0;
#pragma unroll
    for (int q = 0; q < 6; ++q) {
      const uint64_t w = fmix(base + static_cast<uint64_t>(q + 1) * kGolden);
      s += static_cast<int64_t>(w & 0xFFFFFFFFull) + static_cast<int64_t>(w >> 32);
    }
    const double z = static_cast<double>(s - (6ll << 32)) * (1.0 / 4294967296.0);
    double v = __dmul_rn(z, stdv);
    if (col_scale != nullptr) v = __dmul_rn(v, col_scale[i % cols]);
    out[i] = f64_to_bf16_rne(v);
  }
}

}  // namespace

extern "C" int synth_bf16_normal(void* out, int64_t rows, int64_t cols, uint64_t key, double stdv,
                                 const double* col_scale, void* stream) {
  const int64_t n = rows * cols;
  if (n <= 0) return 0;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  bf16_normal_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint16_t*>(out), rows, cols, key, stdv, col_scale);
  return static_cast<int>(cudaGetLastError());
}
