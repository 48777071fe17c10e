// Division by loop-invariant divisors for the kernels' single-thread index
// arithmetic; plain C++ (host compilers build it too), see FastDiv below.
#pragma once

#include <cstdint>

#ifndef __CUDACC__
#define SGB_HD
#else
#define SGB_HD __host__ __device__
#endif

namespace sgb {

// Division by a loop-invariant divisor d >= 1 as a multiply-high, an add and a
// shift (T. Granlund and P. L. Montgomery, "Division by Invariant Integers
// using Multiplication", PLDI 1994, the round-up method): with l = ceil(log2 d)
// and mul = floor(2^32 * (2^l - d) / d) + 1, q = (umulhi(n, mul) + n) >> l
// equals floor(n / d) for every n < 2^31 (the sum then stays below 2^32).  A
// single-thread integer division by a runtime value is a chain of some thirty
// dependent instructions; the kernels' producer threads take several before
// their first load.
struct FastDiv {
    uint32_t d, mul, shift;
    SGB_HD FastDiv() : d(1), mul(1), shift(0) {}
    explicit FastDiv(uint32_t divisor) : d(divisor), mul(1), shift(0)
    {
        uint32_t l = 0;
        while (l < 32 && (uint64_t(1) << l) < divisor) ++l;
        shift = l;
        mul = static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << l) - divisor)) / divisor + 1);
    }
    SGB_HD inline uint32_t div(uint32_t n) const
    {
#ifdef __CUDA_ARCH__
        const uint32_t t = __umulhi(n, mul);
#else
        const uint32_t t = static_cast<uint32_t>((uint64_t(n) * mul) >> 32);
#endif
        return (t + n) >> shift;
    }
};

}  // namespace sgb
