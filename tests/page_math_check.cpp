// Host-only check of the page division the kernels use instead of tok / P
// (csrc/page_math.h): for every page size P that is a multiple of 16 up to
// 4096, every key index below 2^20 and a sample up to 2^31 - 1 (with the
// values next to every multiple of P in range of the sample); and for every
// P from 1 to 4096 on the sample alone.
#include <cstdint>
#include <cstdio>

#include "page_math.h"

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static uint32_t next_u31() {  // splitmix64, top 31 bits
    uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return (uint32_t)(z >> 33);
}

static bool check(int P, int tok, uint32_t m, int s) {
    const int q = pkd::page_div(tok, m, s);
    return q == tok / P && tok - q * P == tok % P;
}

int main() {
    long long checked = 0;
    for (int P = 1; P <= 4096; ++P) {
        uint32_t m;
        int s;
        pkd::page_magic(P, m, s);
        if (P % 16 == 0)
            for (int tok = 0; tok < (1 << 20); ++tok, ++checked)
                if (!check(P, tok, m, s)) { std::printf("FAIL P=%d tok=%d\n", P, tok); return 1; }
        for (int i = 0; i < 20000; ++i, ++checked) {
            const int tok = (int)next_u31();
            if (!check(P, tok, m, s)) { std::printf("FAIL P=%d tok=%d\n", P, tok); return 1; }
            // the neighbours of the multiple of P just below the sample
            const int base = tok / P * P;
            for (int d = -1; d <= 1; ++d) {
                const long long t = (long long)base + d;
                if (t >= 0 && t <= 0x7fffffffLL && !check(P, (int)t, m, s)) {
                    std::printf("FAIL P=%d tok=%lld\n", P, t);
                    return 1;
                }
            }
        }
        if (!check(P, 0x7fffffff, m, s)) { std::printf("FAIL P=%d tok=2^31-1\n", P); return 1; }
    }
    std::printf("ok %lld\n", checked);
    return 0;
}
