// Host-side check of the double-float sum-of-squares helpers of
// ar_common.cuh (the same source the kernels use, compiled for the CPU):
// per-thread accumulation (the fast two-sum for non-negative terms) followed
// by a butterfly of df_add, as in a warp reduction, must give the exact sum
// of squares rounded once to fp32, with every lane ending on the same bits.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <random>

#include "ar_common.cuh"

using arf::DF;

static float bf16_trunc(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    u &= 0xffff0000u;
    memcpy(&x, &u, 4);
    return x;
}

int main()
{
    std::mt19937 rng(1234);
    std::uniform_real_distribution<float> mag(-8.0f, 8.0f);
    std::uniform_int_distribution<int> sign(0, 1);
    int bad = 0, total = 0;
    for (int trial = 0; trial < 800; ++trial) {
        const int lanes = 32, per = 8 * (1 + (trial / 2) % 32);  // up to 8192 terms per row
        DF acc[32];
        long double exact = 0.0L;
        for (int l = 0; l < lanes; ++l) {
            acc[l] = DF{0.0f, 0.0f};
            for (int i = 0; i < per; ++i) {
                float y = bf16_trunc(ldexpf(1.0f + (mag(rng) + 8.0f) / 16.0f, (int)mag(rng)));
                if (sign(rng))
                    y = -y;
                const float t = y * y;                       // exact: 8-bit significand
                exact += (long double)t;
                arf::df_add_nonneg(acc[l], t);
            }
        }
        for (int m = 16; m >= 1; m >>= 1) {                  // xor butterfly
            DF nxt[32];
            for (int l = 0; l < lanes; ++l)
                nxt[l] = arf::df_add(acc[l], acc[l ^ m]);
            memcpy(acc, nxt, sizeof acc);
        }
        for (int l = 1; l < lanes; ++l)
            if (acc[l].hi != acc[0].hi || acc[l].lo != acc[0].lo)
                ++bad;                                       // every lane must agree
        const float got = arf::df_round(acc[0]);
        const float want = (float)exact;                     // one rounding of the exact sum
        ++total;
        if (got != want) {
            ++bad;
            printf("trial %d: got %.9g want %.9g\n", trial, got, want);
        }
    }
    printf("%d/%d bad\n", bad, total);
    return bad ? 1 : 0;
}
