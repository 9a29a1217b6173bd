// Host-side check of the double-float sum-of-squares helpers of
// ar_common.cuh (the same source the kernels use, compiled for the CPU; the
// packed pair operations run per lane):
// per-thread accumulation (two lanes, even and odd terms, each by TwoSum),
// the merge of the two lanes, then a butterfly of df_add as in a warp
// reduction must give the exact sum of squares rounded once to fp32, with
// every lane of the butterfly ending on the same bits.
// The same for one lane accumulated by the fast two-sum of non-negative
// terms (df_add_nonneg, the fp32-element form).
// Built with -DAR_DF_CHECK_PLANT=1 the accumulation drops the rounding errors
// (a plain fp32 sum of the terms): that build must fail the check.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <random>

#include "ar_common.cuh"

#ifndef AR_DF_CHECK_PLANT
#define AR_DF_CHECK_PLANT 0
#endif

using arf::DF;
using arf::DF2;
using arf::F2;

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
    const auto draw = [&]() {
        float y = bf16_trunc(ldexpf(1.0f + (mag(rng) + 8.0f) / 16.0f, (int)mag(rng)));
        return sign(rng) ? -y : y;
    };
    for (int trial = 0; trial < 1600; ++trial) {
        const bool one_lane = trial >= 800;
        const int lanes = 32, per = 8 * (1 + (trial / 2) % 32);  // up to 8192 terms per row
        DF acc[32];
        long double exact = 0.0L;
        for (int l = 0; l < lanes; ++l) {
            DF2 a2 = {};
            DF a1 = {0.0f, 0.0f};
            for (int i = 0; i < per; i += 2) {
                const float y0 = draw(), y1 = draw();
                const F2 t = {y0 * y0, y1 * y1};             // exact: 8-bit significands
                exact += (long double)t.x + (long double)t.y;
                if (AR_DF_CHECK_PLANT) {
                    a2.hi = arf::f2_add(a2.hi, t);
                    a1.hi = a1.hi + t.x + t.y;
                } else if (one_lane) {
                    arf::df_add_nonneg(a1, t.x);
                    arf::df_add_nonneg(a1, t.y);
                } else {
                    arf::df2_add_terms(a2, t);
                }
            }
            acc[l] = one_lane ? a1 : arf::df2_merge(a2);
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
            if (!AR_DF_CHECK_PLANT)
                printf("trial %d: got %.9g want %.9g\n", trial, got, want);
        }
    }
    printf("%d/%d bad\n", bad, total);
    return bad ? 1 : 0;
}
