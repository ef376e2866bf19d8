// Division of 32-bit unsigned integers by a run-time constant through one
// multiply-high, an add and a shift: the round-up method of Granlund and
// Montgomery, "Division by invariant integers using multiplication" (PLDI'94).
// For a divisor d (1 <= d < 2^31) pick l = ceil(log2 d) and
// m = floor(2^32 * (2^l - d) / d) + 1; then for n < 2^31,
// n / d = (umulhi(n, m) + n) >> l.
#pragma once

#include <cstdint>

namespace tra {

struct FastDiv {
    uint32_t d, m, l;

    FastDiv() : d(1), m(1), l(0) {}
    explicit FastDiv(uint32_t div) : d(div) {
        l = 0;
        while ((1ull << l) < div) ++l;
        m = (uint32_t)(((1ull << 32) * ((1ull << l) - div)) / div + 1);
    }
};

#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
    return (__umulhi(n, f.m) + n) >> f.l;
}
#endif

inline uint32_t fdiv_host(uint32_t n, const FastDiv& f) {
    uint32_t hi = (uint32_t)(((uint64_t)n * f.m) >> 32);
    return (hi + n) >> f.l;
}

}  // namespace tra
