/* Host (C) implementation of the seeded input generator defined in
 * synth/__init__.py: the same SplitMix64 words, Irwin-Hall-12 variates, fp64
 * scaling and round-to-nearest-even to bf16 as the numpy definition, only
 * faster.  Input generation only.  Portable C99 with optional OpenMP. */
#include <stdint.h>
#include <string.h>

static const uint64_t kGolden = 0x9E3779B97F4A7C15ull;

static inline uint64_t fmix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint16_t f64_to_bf16_rne(double v, int* bad) {
  uint64_t b;
  memcpy(&b, &v, sizeof b);
  const uint64_t sign = b >> 63;
  const uint64_t mag = b & 0x7FFFFFFFFFFFFFFFull;
  if (mag == 0) return (uint16_t)(sign << 15);
  const uint64_t lsb = (mag >> 45) & 1ull;
  const uint64_t r = (mag + ((1ull << 44) - 1) + lsb) >> 45;
  const int64_t exp8 = (int64_t)(r >> 7) - 1023 + 127;
  if (exp8 <= 0 || exp8 >= 255) {
    *bad = 1;
    return 0x7FC0;
  }
  return (uint16_t)((sign << 15) | ((uint64_t)exp8 << 7) | (r & 0x7Full));
}

/* Returns 0, or 1 if some value fell outside the normal bf16 range. */
int synth_bf16_normal_host(uint16_t* out, int64_t rows, int64_t cols, uint64_t key, double stdv,
                           const double* col_scale) {
  const int64_t n = rows * cols;
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int64_t i = 0; i < n; ++i) {
    const uint64_t base = key + (uint64_t)i * (6ull * kGolden);
    int64_t s = 0;
    for (int q = 0; q < 6; ++q) {
      const uint64_t w = fmix(base + (uint64_t)(q + 1) * kGolden);
      s += (int64_t)(w & 0xFFFFFFFFull) + (int64_t)(w >> 32);
    }
    const double z = (double)(s - (6ll << 32)) * (1.0 / 4294967296.0);
    double v = z * stdv;
    if (col_scale) v = v * col_scale[i % cols];
    int b = 0;
    out[i] = f64_to_bf16_rne(v, &b);
    bad |= b;
  }
  return bad;
}
