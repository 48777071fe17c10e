// Checks sgb::FastDiv against plain integer division (built and run by tests/test_fastdiv.py).
#include <cstdio>
#include <cstdint>
#include <cstdlib>

#include "fastdiv.h"

int main()
{
    unsigned long long bad = 0, checks = 0;
    auto check = [&](const sgb::FastDiv& f, uint32_t d, uint32_t n) {
        ++checks;
        if (f.div(n) != n / d) {
            if (bad < 10) std::printf("d=%u n=%u got %u want %u\n", d, n, f.div(n), n / d);
            ++bad;
        }
    };
    const uint32_t ds[] = {1u, 2u, 3u, 5u, 7u, 9u, 28u, 49u, 63u, 64u, 65u, 76u, 98u, 147u, 196u, 784u, 882u,
                           1152u, 2304u, 3136u, 12544u, 65535u, 65536u, 1000003u, 0x3fffffffu, 0x40000000u, 0x7fffffffu};
    uint64_t x = 88172645463325252ull;  // xorshift64
    for (uint32_t d : ds) {
        const sgb::FastDiv f(d);
        for (uint32_t n = 0; n < 100000; ++n) check(f, d, n);
        for (int i = 0; i < 100000; ++i) {
            x ^= x << 13; x ^= x >> 7; x ^= x << 17;
            check(f, d, static_cast<uint32_t>(x) & 0x7fffffffu);
        }
        for (uint32_t n = 0x7fffffffu - 1000u; n < 0x7fffffffu; ++n) check(f, d, n);
        check(f, d, 0x7fffffffu);
        for (uint32_t k = 1; k < 64 && static_cast<uint64_t>(k) * d < 0x7fffffffull; ++k) {  // around multiples
            check(f, d, k * d - 1u);
            check(f, d, k * d);
        }
    }
    for (uint32_t d = 1; d < 4096; ++d) {
        const sgb::FastDiv f(d);
        for (uint32_t n = 0; n < 8192; n += 3) check(f, d, n);
    }
    std::printf("%llu checks, %llu wrong\n", checks, bad);
    return bad != 0;
}
