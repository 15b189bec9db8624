// Division by a run-time invariant divisor with one multiply-high, an add and a shift
// (Granlund and Montgomery, "Division by invariant integers using multiplication",
// PLDI 1994): with s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1,
// floor(n / d) = (mulhi(n, m) + n) >> s for every 0 <= n < 2^31.
#pragma once

#include <cstdint>

namespace fconv {

struct FastDiv {
  uint32_t d;
  uint32_t mul;
  uint32_t shift;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  uint32_t s = 0;
  while ((1ull << s) < d) ++s;
  f.shift = s;
  f.mul = (uint32_t)((((1ull << 32) * ((1ull << s) - d)) / d) + 1);
  return f;
}

__host__ __device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
#ifdef __CUDA_ARCH__
  const uint32_t hi = __umulhi(n, f.mul);
#else
  const uint32_t hi = (uint32_t)(((uint64_t)n * f.mul) >> 32);
#endif
  return (hi + n) >> f.shift;
}

// n = q * d + r
__host__ __device__ __forceinline__ void fast_divmod(uint32_t n, const FastDiv& f, uint32_t& q,
                                                     uint32_t& r) {
  q = fast_div(n, f);
  r = n - q * f.d;
}

}  // namespace fconv
