/*
 * CPU oracle for the allreduce-fusion epilogue (R-way sum + residual add +
 * RMSNorm + optional FP8 E4M3 / NVFP4 quantisation) and for the plain
 * R-way sum.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant generator
 * with the CUDA path.
 *
 * Build: plain C, strict IEEE single/double arithmetic, no FMA contraction
 *   gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 *
 * Every function is written straight from the definition it cites, in the
 * order the pages state, with no blocking, fusion or reordering:
 *
 *   [TRT]  TensorRT-LLM, cpp/tensorrt_llm/kernels/allReduceFusionKernels.cu
 *          (functions add128, rms_norm, fused_op, allreduce_sum,
 *           allreduce_fusion_kernel_oneshot_lamport, lamport_initialize,
 *           LamportComm, Workspace)
 *   [FI]   FlashInfer docs, flashinfer.comm.
 *          trtllm_create_ipc_workspace_for_all_reduce_fusion (workspace note)
 *   [MSC]  mscclpp, python/mscclpp_benchmark/allreduce.cu (vectorSum)
 *
 * Element formats (definitions, not taken from any library):
 *   bf16  : 1 sign, 8 exponent (bias 127), 7 mantissa bits
 *   fp16  : 1 sign, 5 exponent (bias 15), 10 mantissa bits
 *   e4m3  : OCP FP8 "fn" variant: 1/4/3, bias 7, no infinities,
 *           NaN = S.1111.111, largest finite 448, subnormal step 2^-9
 *   e2m1  : OCP FP4: 1/2/1, bias 1, values {0,.5,1,1.5,2,3,4,6}, no inf/NaN
 *
 * Element types: bf16 / fp16 arrays are handled as uint16 bit patterns; the
 * *_f32 functions take float arrays (FlashInfer's use_fp32_lamport exchange
 * type), where every rounding to the element type is the identity.
 *
 * Parity pins for every function live in tests/test_oracle_*.py.  The NVFP4
 * global-scale convention (gs = 2688 / amax, enc = gs / f(sf)) is a stated
 * reading (the quantiser's helper header is not on the pages): parity
 * unpinned for that convention only -- a property pin holds the oracle to the
 * reading (the amax block gets the largest block scale, 448, and its largest
 * element the code +-6), but nothing outside it fixes the reading itself.
 * The block-scale tile layout is pinned outside the oracle, by a
 * block-scaled matmul library reading it.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { OR_BF16 = 0, OR_FP16 = 1 };

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* ---------------------------------------------------------------- bf16 --- */

float oracle_bf16_to_f32(uint16_t b) { return u2f((uint32_t)b << 16); }

/* fp32 -> bf16, round to nearest, ties to even.  bf16 is the upper half of an
 * fp32 word: keep the top 16 bits and decide on the 16 dropped ones. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u = f2u(f);
    if ((u & 0x7fffffffu) > 0x7f800000u)             /* NaN: keep it a NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;                                   /* carry may reach inf: correct */
    return (uint16_t)kept;
}

/* ---------------------------------------------------------------- fp16 --- */

float oracle_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1fu;
    uint32_t m = h & 0x3ffu;
    float mag;
    if (e == 0x1fu)
        return u2f(sign | 0x7f800000u | (m << 13));   /* inf / NaN */
    if (e == 0)
        mag = (float)m * 0x1p-24f;                    /* subnormal: m * 2^-24, exact */
    else
        mag = ldexpf(1.0f + (float)m / 1024.0f, (int)e - 15);
    return sign ? -mag : mag;
}

/* fp32 -> fp16, round to nearest, ties to even, overflow to infinity. */
uint16_t oracle_f32_to_f16(float f)
{
    uint32_t u = f2u(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u)
        return sign | 0x7e00u;                        /* NaN */
    if (a >= 0x38800000u) {                           /* |f| >= 2^-14: normal range */
        int e = (int)(a >> 23) - 127 + 15;            /* fp16 biased exponent */
        if (e >= 31)
            return sign | 0x7c00u;                    /* |f| >= 65536 */
        uint32_t m = a & 0x7fffffu;
        uint32_t kept = ((uint32_t)e << 10) | (m >> 13);
        uint32_t dropped = m & 0x1fffu;
        if (dropped > 0x1000u || (dropped == 0x1000u && (kept & 1u)))
            kept += 1u;                               /* carry into exponent is correct */
        return sign | (uint16_t)kept;
    }
    /* below 2^-14: value = q * 2^-24 with integer q rounded half to even */
    float scaled = fabsf(f) * 16777216.0f;            /* exact: power-of-two scale */
    uint32_t q = (uint32_t)scaled;
    float frac = scaled - (float)q;                   /* exact */
    if (frac > 0.5f || (frac == 0.5f && (q & 1u)))
        q += 1u;
    return sign | (uint16_t)q;                        /* q == 1024 is 2^-14: correct */
}

static float dec_d(int dtype, uint16_t v)
{
    return dtype == OR_BF16 ? oracle_bf16_to_f32(v) : oracle_f16_to_f32(v);
}

static uint16_t rnd_d(int dtype, float v)
{
    return dtype == OR_BF16 ? oracle_f32_to_bf16(v) : oracle_f32_to_f16(v);
}

/* ---------------------------------------------------------------- e4m3 --- */

float oracle_e4m3_to_f32(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xf, m = c & 7;
    float mag;
    if (e == 0xf && m == 7)
        return NAN;
    if (e == 0)
        mag = (float)m * 0x1p-9f;
    else
        mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return s ? -mag : mag;
}

/* fp32 -> e4m3, round to nearest (ties to even), finite values beyond the
 * largest code saturate to +-448, infinities too ("satfinite"), NaN -> NaN,
 * sign of zero kept. */
uint8_t oracle_f32_to_e4m3(float x)
{
    uint8_t s = (uint8_t)((f2u(x) >> 24) & 0x80u);
    if (isnan(x))
        return s | 0x7f;
    float ax = fabsf(x);
    if (ax >= 448.0f)
        return s | 0x7e;
    int e;                                            /* ax in [2^e, 2^(e+1)) */
    if (ax < 0x1p-6f) {
        e = -6;                                       /* subnormal band: step 2^-9 */
    } else {
        frexpf(ax, &e);
        e -= 1;
    }
    float scaled = ldexpf(ax, 3 - e);                 /* ax / 2^(e-3), exact */
    uint32_t n = (uint32_t)scaled;
    float frac = scaled - (float)n;
    if (frac > 0.5f || (frac == 0.5f && (n & 1u)))
        n += 1u;
    if (e == -6 && n < 8u)
        return s | (uint8_t)n;                        /* subnormal code */
    if (n == 16u) { n = 8u; e += 1; }                 /* rounded up to next binade */
    uint32_t code = ((uint32_t)(e + 7) << 3) | (n - 8u);
    if (code > 0x7eu)
        code = 0x7eu;                                 /* cannot happen below 448 */
    return s | (uint8_t)code;
}

/* ---------------------------------------------------------------- e2m1 --- */

float oracle_e2m1_to_f32(uint8_t c)
{
    static const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    float v = mag[c & 7];
    return (c & 8) ? -v : v;
}

/* fp32 -> e2m1 (4-bit code in the low nibble), round to nearest with ties to
 * the even mantissa, saturate to +-6, sign of zero kept.  NaN has no code in
 * this format; it maps to the signed maximum (inputs here are finite). */
uint8_t oracle_f32_to_e2m1(float x)
{
    uint8_t s = (uint8_t)((f2u(x) >> 28) & 0x8u);
    float ax = fabsf(x);
    if (isnan(x) || ax >= 6.0f)
        return s | 0x7;
    int e;                                            /* ax in [2^e, 2^(e+1)) */
    if (ax < 1.0f) {
        e = 0;                                        /* subnormal band: step 0.5 */
    } else {
        frexpf(ax, &e);
        e -= 1;
    }
    float scaled = ldexpf(ax, 1 - e);                 /* ax / 2^(e-1), exact */
    uint32_t n = (uint32_t)scaled;
    float frac = scaled - (float)n;
    if (frac > 0.5f || (frac == 0.5f && (n & 1u)))
        n += 1u;
    if (ax < 1.0f && n < 2u)
        return s | (uint8_t)n;                        /* 0 or 0.5 */
    if (ax < 1.0f)
        return s | 0x2;                               /* rounded up to 1.0 */
    if (n == 4u) { n = 2u; e += 1; }
    uint32_t code = ((uint32_t)(e + 1) << 1) | (n - 2u);
    if (code > 7u)
        code = 7u;                                    /* cannot happen below 6 */
    return s | (uint8_t)code;
}

/* ----------------------------------------------------- Lamport sentinel --- */

/* The one-shot push step of [TRT] allreduce_fusion_kernel_oneshot_lamport
 * rewrites every 32-bit word that equals the -0.0f sentinel (0x80000000) to
 * +0.0f before it lands in the peers' slot, so that the reader can tell
 * "not yet written" from data.  For 16-bit elements one word holds a pair:
 * the pair (low=+0, high=-0) becomes (+0, +0).  Operates in place on
 * `n_words` 32-bit words. */
void oracle_lamport_flip(uint32_t* words, int64_t n_words)
{
    for (int64_t i = 0; i < n_words; ++i)
        if (words[i] == 0x80000000u)
            words[i] = 0u;
}

/* ------------------------------------------------------ fused epilogue --- */

/* Sum over ranks of one element, p[r * stride] for r < R ([TRT] allreduce_sum):
 *   acc = 0: fp32, rank order, rounded to D once by the caller (Fp32Acc, the
 *            default of [TRT] use_fp32_acc);
 *   acc = 1: every partial sum rounded to D (the other branch: chained add128
 *            in the element type; [MSC] vectorSum's half-precision adds).
 * An fp32 addition of two 16-bit values followed by one rounding to D is the
 * correctly rounded D addition.  Returns the fp32 value before the caller's
 * final rounding to D. */
static float rank_sum(int dtype, int acc, const uint16_t* p, int64_t stride, int R)
{
    float s = dec_d(dtype, p[0]);
    for (int r = 1; r < R; ++r) {
        s = s + dec_d(dtype, p[(int64_t)r * stride]);
        if (acc)
            s = dec_d(dtype, rnd_d(dtype, s));
    }
    return s;
}

/*
 * For rows t in [row_begin, row_end) of a [T][H] problem:
 *
 *   s_h   = f(P[0][t][h]) + f(P[1][t][h]) + ... + f(P[R-1][t][h])
 *           fp32, rank order                        ([TRT] allreduce_sum, Fp32Acc;
 *           acc = 1: rounded to D after every addition, see rank_sum)
 *   a_h   = rnd_D(s_h)                              (same, final cast)
 *   y_h   = rnd_D(f(a_h) + f(X[t][h]))  -> residual_out     ([TRT] add128, fused_op)
 *   ss    = sum_h f(y_h)^2   accumulated in fp64, rounded once to fp32
 *   rstd  = 1 / sqrt(ss / H + eps)   each step an IEEE-rounded fp32 op
 *                                                   ([TRT] rms_norm)
 *   n_h   = rnd_D((f(y_h) * rstd) * f(gamma_h))  -> norm_out  ([TRT] rms_norm)
 *
 * partials: element (r, t, h) at partials[r * rank_stride + t * H + h]
 * residual_in, residual_out, norm_out: [T][H]; gamma: [H].
 * residual_out / norm_out may be NULL (not written).  rstd_out (may be NULL)
 * receives the per-row fp32 rstd.
 */
void oracle_fused_rows(int dtype, int acc, int R, int64_t T, int64_t H, int64_t rank_stride,
                       const uint16_t* partials, const uint16_t* residual_in,
                       const uint16_t* gamma, float eps, int64_t row_begin, int64_t row_end,
                       uint16_t* residual_out, uint16_t* norm_out, float* rstd_out)
{
    (void)T;
    for (int64_t t = row_begin; t < row_end; ++t) {
        double ss = 0.0;
        /* pass 1: sum over ranks, round, residual add, round, square-sum */
        for (int64_t h = 0; h < H; ++h) {
            float s = rank_sum(dtype, acc, partials + t * H + h, rank_stride, R);
            uint16_t a = rnd_d(dtype, s);
            uint16_t y = rnd_d(dtype, dec_d(dtype, a) + dec_d(dtype, residual_in[t * H + h]));
            if (residual_out)
                residual_out[t * H + h] = y;
            double yd = (double)dec_d(dtype, y);
            ss += yd * yd;
        }
        float ss32 = (float)ss;
        float ms = ss32 / (float)H;
        float v = ms + eps;
        float rstd = 1.0f / sqrtf(v);
        if (rstd_out)
            rstd_out[t] = rstd;
        if (!norm_out)
            continue;
        /* pass 2: normalise (recomputes y; identical arithmetic) */
        for (int64_t h = 0; h < H; ++h) {
            float s = rank_sum(dtype, acc, partials + t * H + h, rank_stride, R);
            uint16_t a = rnd_d(dtype, s);
            uint16_t y = rnd_d(dtype, dec_d(dtype, a) + dec_d(dtype, residual_in[t * H + h]));
            float ny = dec_d(dtype, y) * rstd;
            float n = ny * dec_d(dtype, gamma[h]);
            norm_out[t * H + h] = rnd_d(dtype, n);
        }
    }
}

/* amax = max |f(x_i)| over n elements of D, with fmaxf semantics (a NaN
 * element is ignored unless all are NaN). */
float oracle_amax(int dtype, const uint16_t* x, int64_t n)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i)
        m = fmaxf(m, fabsf(dec_d(dtype, x[i])));
    return m;
}

/* Per-tensor FP8 scale convention of the target configuration: the scale is
 * amax / 448 and the kernel multiplies by its inverse, computed once.  An
 * all-zero tensor has no amax to map; it gets the multiplier 1.0 (every code
 * is then 0) instead of an infinite one. */
float oracle_fp8_inv_scale(float amax)
{
    if (!(amax > 0.0f))
        return 1.0f;
    float scale = amax / 448.0f;
    return 1.0f / scale;
}

/* q_i = e4m3(f(n_i) * inv_scale), n elements. */
void oracle_quant_fp8(int dtype, const uint16_t* n_in, int64_t n, float inv_scale, uint8_t* q)
{
    for (int64_t i = 0; i < n; ++i)
        q[i] = oracle_f32_to_e4m3(dec_d(dtype, n_in[i]) * inv_scale);
}

/* NVFP4 global encode scale: maps the tensor amax onto the largest product of
 * an E4M3 block scale (448) and an E2M1 value (6).  An all-zero tensor has no
 * amax to map; it gets 1.0 (every block scale and code is then 0). */
float oracle_nvfp4_global_scale(float amax)
{
    if (!(amax > 0.0f))
        return 1.0f;
    return 2688.0f / amax;
}

/*
 * NVFP4 of a [T][H] tensor of D (H a multiple of 16), per 16-element block b
 * of row t:
 *   bmax  = max_i |f(n_i)|
 *   sf    = e4m3(gs * (bmax / 6))            -> scale_out[t][b]   (one byte)
 *   dec   = f(sf);  enc = dec == 0 ? 0 : gs / dec
 *   q_i   = e2m1(f(n_i) * enc)               -> element 2k in the low nibble
 *                                               of quant_out[t][k]
 * Dequantised value: val(q_i) * dec / gs.
 */
void oracle_quant_nvfp4(int dtype, const uint16_t* n_in, int64_t T, int64_t H, float gs,
                        uint8_t* quant_out, uint8_t* scale_out)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t b = 0; b < H / 16; ++b) {
            const uint16_t* blk = n_in + t * H + b * 16;
            float bmax = 0.0f;
            for (int i = 0; i < 16; ++i)
                bmax = fmaxf(bmax, fabsf(dec_d(dtype, blk[i])));
            float per_block = bmax / 6.0f;
            uint8_t sf = oracle_f32_to_e4m3(gs * per_block);
            scale_out[t * (H / 16) + b] = sf;
            float dec = oracle_e4m3_to_f32(sf);
            float enc = (dec == 0.0f) ? 0.0f : gs / dec;
            for (int k = 0; k < 8; ++k) {
                uint8_t lo = oracle_f32_to_e2m1(dec_d(dtype, blk[2 * k]) * enc);
                uint8_t hi = oracle_f32_to_e2m1(dec_d(dtype, blk[2 * k + 1]) * enc);
                quant_out[t * (H / 2) + b * 8 + k] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/* NVFP4 block scales of a [T][KB] matrix rearranged into tiles of 128 rows x
 * 4 blocks, as tensor-core NVFP4 matrix multiplies read them (a layout of
 * ours to match that consumer; the pages' helper header is absent): tiles are
 * ordered row-major over (row / 128, block / 4), 512 bytes each, and inside a
 * tile row m, block k sits at (m % 32) * 16 + ((m / 32) % 4) * 4 + k % 4.
 * `out` has ceil(T / 128) * 128 * ceil(KB / 4) * 4 bytes; bytes that belong to
 * no (m < T, k < KB) are left as they are. */
void oracle_swizzle_scales(const uint8_t* linear, int64_t T, int64_t KB, uint8_t* out)
{
    int64_t ktiles = (KB + 3) / 4;
    for (int64_t m = 0; m < T; ++m) {
        for (int64_t k = 0; k < KB; ++k) {
            int64_t tile = (m / 128) * ktiles + k / 4;
            int64_t within = (m % 32) * 16 + ((m / 32) % 4) * 4 + k % 4;
            out[tile * 512 + within] = linear[m * KB + k];
        }
    }
}

/* ------------------------------------------------------- plain R-way sum --- */

/* out_i = rnd_D(f(in_0[i]) + f(in_1[i]) + ... + f(in_{R-1}[i])), fp32, rank
 * order ([MSC] vectorSum applied R-1 times, accumulating in fp32 as the fused
 * path does); acc = 1: every addition rounded to D, as vectorSum's
 * element-type adds.  Element (r, i) at in[r * rank_stride + i]. */
void oracle_sum(int dtype, int acc, int R, int64_t n, int64_t rank_stride, const uint16_t* in,
                uint16_t* out, int64_t i_begin, int64_t i_end)
{
    (void)n;
    for (int64_t i = i_begin; i < i_end; ++i)
        out[i] = rnd_d(dtype, rank_sum(dtype, acc, in + i, rank_stride, R));
}

/* ------------------------------------------- fp32 element type (f32) --- */

/* The same operation with 32-bit float elements (FlashInfer workspace
 * creation's use_fp32_lamport: the exchanged buffers hold fp32).  Every
 * rounding to the element type of the 16-bit path is the identity here:
 *   s = P_0 + ... + P_{R-1} (fp32, rank order);  y = s + X   -> residual_out
 *   ss = sum_h y_h^2 in fp64 (each square exact: 24-bit significands square
 *        into 48 bits), rounded once to fp32;  rstd = 1 / sqrt(ss / H + eps)
 *   n = (y * rstd) * gamma                                    -> norm_out
 * Arrays as in oracle_fused_rows, of float. */
void oracle_fused_rows_f32(int R, int64_t T, int64_t H, int64_t rank_stride,
                           const float* partials, const float* residual_in, const float* gamma,
                           float eps, int64_t row_begin, int64_t row_end, float* residual_out,
                           float* norm_out, float* rstd_out)
{
    (void)T;
    for (int64_t t = row_begin; t < row_end; ++t) {
        double ss = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            float s = partials[t * H + h];
            for (int r = 1; r < R; ++r)
                s = s + partials[(int64_t)r * rank_stride + t * H + h];
            float y = s + residual_in[t * H + h];
            if (residual_out)
                residual_out[t * H + h] = y;
            ss += (double)y * (double)y;
        }
        float ss32 = (float)ss;
        float ms = ss32 / (float)H;
        float v = ms + eps;
        float rstd = 1.0f / sqrtf(v);
        if (rstd_out)
            rstd_out[t] = rstd;
        if (!norm_out)
            continue;
        for (int64_t h = 0; h < H; ++h) {
            float s = partials[t * H + h];
            for (int r = 1; r < R; ++r)
                s = s + partials[(int64_t)r * rank_stride + t * H + h];
            float y = s + residual_in[t * H + h];
            float ny = y * rstd;
            norm_out[t * H + h] = ny * gamma[h];
        }
    }
}

float oracle_amax_f32(const float* x, int64_t n)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i)
        m = fmaxf(m, fabsf(x[i]));
    return m;
}

void oracle_quant_fp8_f32(const float* n_in, int64_t n, float inv_scale, uint8_t* q)
{
    for (int64_t i = 0; i < n; ++i)
        q[i] = oracle_f32_to_e4m3(n_in[i] * inv_scale);
}

/* NVFP4 of fp32 values, same block rule as oracle_quant_nvfp4. */
void oracle_quant_nvfp4_f32(const float* n_in, int64_t T, int64_t H, float gs, uint8_t* quant_out,
                            uint8_t* scale_out)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t b = 0; b < H / 16; ++b) {
            const float* blk = n_in + t * H + b * 16;
            float bmax = 0.0f;
            for (int i = 0; i < 16; ++i)
                bmax = fmaxf(bmax, fabsf(blk[i]));
            float per_block = bmax / 6.0f;
            uint8_t sf = oracle_f32_to_e4m3(gs * per_block);
            scale_out[t * (H / 16) + b] = sf;
            float dec = oracle_e4m3_to_f32(sf);
            float enc = (dec == 0.0f) ? 0.0f : gs / dec;
            for (int k = 0; k < 8; ++k) {
                uint8_t lo = oracle_f32_to_e2m1(blk[2 * k] * enc);
                uint8_t hi = oracle_f32_to_e2m1(blk[2 * k + 1] * enc);
                quant_out[t * (H / 2) + b * 8 + k] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/* out_i = in_0[i] + ... + in_{R-1}[i] in fp32, rank order. */
void oracle_sum_f32(int R, int64_t rank_stride, const float* in, float* out, int64_t i_begin,
                    int64_t i_end)
{
    for (int64_t i = i_begin; i < i_end; ++i) {
        float s = in[i];
        for (int r = 1; r < R; ++r)
            s = s + in[(int64_t)r * rank_stride + i];
        out[i] = s;
    }
}

/* ------------------------------------------------ workspace arithmetic --- */

/*
 * Byte sizes of the workspace regions, [TRT] Workspace constructor with the
 * element size taken from the data type as [FI] allows:
 *   buffer      = R * maxT * H * elem
 *   flags       = R * flag_count * 4
 *   lamport     = 3 slots of R * max(oneshot_max, maxT) * H * elem
 * out[0..3] = buffer, flags, one Lamport slot, all three Lamport slots.
 */
void oracle_workspace_sizes(int R, int64_t max_tokens, int64_t H, int elem_bytes,
                            int64_t oneshot_max, int64_t flag_count, int64_t* out)
{
    int64_t tok = max_tokens > oneshot_max ? max_tokens : oneshot_max;
    out[0] = (int64_t)R * max_tokens * H * elem_bytes;
    out[1] = (int64_t)R * flag_count * 4;
    out[2] = (int64_t)R * tok * H * elem_bytes;
    out[3] = 3 * out[2];
}

/* Lamport triple-buffer state after one call ([TRT] LamportComm): the call
 * reads slot flag % 3, clears slot (flag + 2) % 3 over `clear_size` elements,
 * then sets flag = (flag + 1) % 3 and clear_size = R * T * H.
 * io[0] = flag, io[1] = clear_size; io[2] <- slot read, io[3] <- slot cleared. */
void oracle_lamport_step(int64_t* io, int R, int64_t T, int64_t H)
{
    int64_t flag = io[0];
    io[2] = flag % 3;
    io[3] = (flag + 2) % 3;
    io[0] = (flag + 1) % 3;
    io[1] = (int64_t)R * T * H;
}
