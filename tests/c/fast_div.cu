/*
 * Division by a run-time invariant (kvw_device.cuh, FastDiv) against the
 * hardware division, on the host: every divisor 1 .. 70000 with numerators
 * around its multiples and at the ends of the 32-bit range, and a sweep of
 * pseudo-random (n, d) pairs.  Exit status 0 when all agree.
 */
#include <cstdint>
#include <cstdio>

#include "kvw_device.cuh"

int main() {
    uint64_t checked = 0, bad = 0;
    auto check = [&](uint32_t n, const kvw::FastDiv& f) {
        ++checked;
        if (kvw::fast_div(n, f) != n / f.d) {
            if (bad++ < 5) printf("n=%u d=%u got %u want %u\n", n, f.d, kvw::fast_div(n, f), n / f.d);
        }
    };
    for (uint32_t d = 1; d <= 70000; ++d) {
        const kvw::FastDiv f = kvw::make_fast_div(d);
        const uint32_t ends[] = {0u, 1u, d - 1u, d, d + 1u, 2u * d - 1u, 2u * d, 0x7fffffffu,
                                 0x80000000u, 0xfffffffeu, 0xffffffffu};
        for (uint32_t n : ends) check(n, f);
        for (uint32_t k = 1; k < 64; ++k) {
            const uint64_t base = (uint64_t)d * (0xffffffffull / d / 64 * k + k);
            for (int64_t e = -1; e <= 1; ++e) {
                const uint64_t n = base + e;
                if (n <= 0xffffffffull) check((uint32_t)n, f);
            }
        }
    }
    uint64_t x = 0x9E3779B97F4A7C15ull;
    for (int i = 0; i < 20000000; ++i) {
        x ^= x << 13; x ^= x >> 7; x ^= x << 17;
        const uint32_t d = (uint32_t)(x >> 40) | 1u;
        const uint32_t n = (uint32_t)x;
        check(n, kvw::make_fast_div((i & 1) ? d : (d >> (x & 15)) + 1u));
    }
    printf("fast_div: %llu checked, %llu wrong\n", (unsigned long long)checked,
           (unsigned long long)bad);
    return bad ? 1 : 0;
}
