// Division of non-negative 32-bit integers by a divisor fixed for a launch,
// as one multiply-high, an add and two shifts instead of the long integer
// division sequence: the round-up method of Granlund and Montgomery,
// "Division by invariant integers using multiplication" (PLDI 1994), which is
// exact for every 32-bit dividend.  With l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1 (which fits 32 bits),
//   t = (m n) >> 32,   n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0).
// Plain C++ on the host (the work-item walk is checked against / there), the
// multiply-high intrinsic on the device.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define FA_FASTDIV_HD __host__ __device__ __forceinline__
#else
#define FA_FASTDIV_HD inline
#endif

namespace fa {

struct FastDiv {
  uint32_t d = 1, m = 1, s1 = 0, s2 = 0;

  FastDiv() = default;
  // divisor >= 1
  explicit FastDiv(uint32_t divisor) : d(divisor) {
    uint32_t l = 0;
    while (l < 32 && (uint64_t{1} << l) < divisor) ++l;
    m = static_cast<uint32_t>((((uint64_t{1} << l) - divisor) << 32) / divisor + 1);
    s1 = l > 0 ? 1u : 0u;
    s2 = l > 0 ? l - 1 : 0u;
  }

  FA_FASTDIV_HD uint32_t div(uint32_t n) const {
#if defined(__CUDA_ARCH__)
    const uint32_t t = __umulhi(m, n);
#else
    const uint32_t t = static_cast<uint32_t>((static_cast<uint64_t>(m) * n) >> 32);
#endif
    return (t + ((n - t) >> s1)) >> s2;
  }
  FA_FASTDIV_HD int div(int n) const { return static_cast<int>(div(static_cast<uint32_t>(n))); }
  FA_FASTDIV_HD int mod(int n) const { return n - div(n) * static_cast<int>(d); }
};

}  // namespace fa
