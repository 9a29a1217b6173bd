// Per-vector steps of the fused epilogue shared by every kernel variant
// (TensorRT-LLM allReduceFusionKernels.cu: add128 / fused_op for the residual,
// rms_norm for the normalisation, fused_op's quantised output).
//
// A "vector" is 8 consecutive elements of a row (16 bytes of bf16 / fp16, 32
// bytes of fp32).
#pragma once

#include "ar_common.cuh"
#include "ar_internal.h"

namespace arf {

// From the fp32 rank sum s of one vector and the residual x:
//   a = rnd(s);  y = rnd(f(a) + f(x));  ss += y^2 (exact squares, TwoSum).
// Returns y (packed).  The squares enter two double-float lanes (even and odd
// elements) by TwoSums, packed in pairs for 16-bit elements.  fp32 elements:
// the square of a 24-bit significand needs 48 bits, so it enters as its
// rounded product plus the exact remainder (TwoProduct by fma).
template <class D>
__device__ __forceinline__ typename D::Vec residual_vec(const float (&s)[8],
                                                        const typename D::Vec& x, DF2& ss)
{
    if constexpr (D::bytes == 4) {
        float a[8];
        unpack8<D>(pack8<D>(s), a);
        add8<D>(a, x);
        const typename D::Vec y = pack8<D>(a);
        // one scalar lane (the other stays zero) by the fast two-sum of
        // non-negative terms: packed pairs measured slower here (fp32, R = 4,
        // T = 8192, H = 4096: 161.2 vs 132.7 us), and a second lane or TwoSum's
        // extra additions cost 2-4% in the wide fp32 bulk-copy pipe
        DF acc = {ss.hi.x, ss.lo.x};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float p = __fmul_rn(a[i], a[i]);
            const float e = __fmaf_rn(a[i], a[i], -p);
            df_add_nonneg(acc, p);
            acc.lo = __fadd_rn(acc.lo, e);
        }
        ss.hi.x = acc.hi;
        ss.lo.x = acc.lo;
        return y;
    } else {
        // a = rnd(s); y = rnd(f(a) + f(x)) by packed 16-bit adds
        const typename D::Vec y = add_packed<D>(pack8<D>(s), x);
        F2 t[4];
        sq2<D>(t[0].x, t[0].y, y.x);
        sq2<D>(t[1].x, t[1].y, y.y);
        sq2<D>(t[2].x, t[2].y, y.z);
        sq2<D>(t[3].x, t[3].y, y.w);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            df2_add_terms(ss, t[i]);
        return y;
    }
}

// rstd = 1 / sqrt(ss / H + eps), each step IEEE round-to-nearest.
__device__ __forceinline__ float inv_rms(DF ss, int H, float eps)
{
    const float ms = __fdiv_rn(df_round(ss), (float)H);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

// Row rstd from one DF partial per warp.  Each warp sums its lanes; warp 0
// combines the nw warp sums (lane l takes slot l, then an xor butterfly),
// computes rstd once and publishes it; `sync` is the barrier of the threads
// that share the row (a __syncthreads or a named barrier).  Two slot sets
// alternate by row parity, so one row's slots are never overwritten before
// every thread has read them.
struct BlockSync {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// barrier 1 over the first n threads of the block (the consumer warps)
struct NamedSync {
    int n;
    __device__ __forceinline__ void operator()() const
    {
        asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory");
    }
};

template <class Sync>
__device__ __forceinline__ float row_rstd(DF ss, DF* slots, float* rstd_slot, int warp, int lane,
                                          int nw, int H, float eps, Sync sync)
{
    ss = df_warp_sum(ss);
    if (lane == 0)
        slots[warp] = ss;
    sync();
    if (warp == 0) {
        DF v = lane < nw ? slots[lane] : DF{0.0f, 0.0f};
        v = df_warp_sum(v);
        if (lane == 0)
            *rstd_slot = inv_rms(v, H, eps);
    }
    sync();
    return *rstd_slot;
}

// gamma of one vector as fp32 (loaded once per kernel)
template <class D>
__device__ __forceinline__ void load_gamma(const uint8_t* gamma, int v, bool ok, float (&g)[8])
{
    if (ok) {
        unpack8<D>(ld_keep_v<D>(gamma + (size_t)v * 8 * D::bytes), g);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            g[i] = 0.0f;
    }
}

// Byte offset of NVFP4 block scale (row m, block k) of a [T][H/16] scale
// matrix: linear row-major, or tiles of 128 rows x 4 blocks (512 bytes each,
// tiles row-major over (m / 128, k / 4)) holding row m at
// (m % 32) * 16 + ((m / 32) % 4) * 4 + k % 4 -- the block-scale layout that
// tensor-core NVFP4 matrix multiplies read.
__device__ __forceinline__ size_t sf_offset(int layout, int m, int k, int kblocks)
{
    if (layout == AR_SF_LINEAR)
        return (size_t)m * kblocks + k;
    const size_t ktiles = (size_t)(kblocks + 3) / 4;
    const size_t tile = (size_t)(m >> 7) * ktiles + (size_t)(k >> 2);
    return tile * 512 + (size_t)(m & 31) * 16 + (size_t)((m >> 5) & 3) * 4 + (size_t)(k & 3);
}

// t = x * k per element (rounded to fp32), in packed pairs for 16-bit elements
template <class D>
__device__ __forceinline__ void scale8(const float (&x)[8], float k, float (&t)[8])
{
    if constexpr (D::bytes == 2) {
        const F2 k2 = {k, k};
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const F2 v = f2_mul(F2{x[i], x[i + 1]}, k2);
            t[i] = v.x;
            t[i + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            t[i] = __fmul_rn(x[i], k);
    }
}

// n = rnd((f(y) * rstd) * gamma); stores norm_out and the quantised outputs
// of vector v of `row`.  Every lane of the warp must call this (the NVFP4
// block maximum is exchanged with the xor-1 neighbour); `ok` masks the stores
// of lanes past the end of the row.
template <class D>
__device__ __forceinline__ void normalize_vec(const FusedArgs& a, int pat, int row, int v, bool ok,
                                              const typename D::Vec& y, const float (&g)[8],
                                              float rstd,
                                              float qscale, float& amax_local)
{
    const int H = a.H;
    float yf[8], nf[8];
    unpack8<D>(y, yf);
    if constexpr (D::bytes == 2) {
        // packed pairs (fp32 elements keep scalar products: the packed form
        // measured 3-4% slower in the wide fp32 bulk-copy pipe)
        const F2 r2 = {rstd, rstd};
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const F2 n = f2_mul(f2_mul(F2{yf[i], yf[i + 1]}, r2), F2{g[i], g[i + 1]});
            nf[i] = n.x;
            nf[i + 1] = n.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            nf[i] = __fmul_rn(__fmul_rn(yf[i], rstd), g[i]);
    }
    const typename D::Vec nv = pack8<D>(nf);
    if (ok && (pat & AR_NORM_OUT))
        st_vec(a.norm_out + ((size_t)row * H + (size_t)v * 8) * D::bytes, nv);
    if (!(pat & (AR_QUANT_FP8 | AR_QUANT_NVFP4)) && !a.amax_out)
        return;
    float nq[8];
    unpack8<D>(nv, nq);
    if (a.amax_out && ok) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            amax_local = fmaxf(amax_local, fabsf(nq[i]));
    }
    if (pat & AR_QUANT_FP8) {
        float t[8];
        scale8<D>(nq, qscale, t);
        const uint2 c = e4m3x8(t);
        if (ok)
            st_u2(a.quant_out + (size_t)row * H + (size_t)v * 8, c.x, c.y);
    } else if (pat & AR_QUANT_NVFP4) {
        float bm = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            bm = fmaxf(bm, fabsf(nq[i]));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
        const uint32_t sf = e4m3_byte(__fmul_rn(qscale, __fdiv_rn(bm, 6.0f)));
        const float dec = e4m3_to_f32(sf);
        const float enc = dec == 0.0f ? 0.0f : __fdiv_rn(qscale, dec);
        float t[8];
        scale8<D>(nq, enc, t);
        const uint32_t codes = e2m1x8(t);
        if (ok) {
            *reinterpret_cast<uint32_t*>(a.quant_out + (size_t)row * (H / 2) + (size_t)v * 4) = codes;
            if ((v & 1) == 0)
                a.scale_out[sf_offset(a.sf_layout, row, v >> 1, H / 16)] = (uint8_t)sf;
        }
    }
}

}  // namespace arf
