// Device helpers shared by the sm_103a kernels of libarfusion.
//
// Element conversions use the hardware cvt instructions (round to nearest
// even); no approximate math is used anywhere on the path: the RMSNorm
// division and square root are the IEEE-rounded __fdiv_rn / __fsqrt_rn.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ar_fusion.h"

namespace arf {

// A "vector" is 8 consecutive elements of a row: 16 bytes of bf16 / fp16
// (one uint4) or 32 bytes of fp32 (one V32, moved by a single 256-bit access).
struct V32 {
    uint4 lo, hi;
};

struct Bf16 {
    static constexpr int id = AR_DT_BF16;
    static constexpr int bytes = 2;
    using Vec = uint4;
};
struct Fp16 {
    static constexpr int id = AR_DT_FP16;
    static constexpr int bytes = 2;
    using Vec = uint4;
};
struct F32 {
    static constexpr int id = AR_DT_FP32;
    static constexpr int bytes = 4;
    using Vec = V32;
};

// ------------------------------------------------------ 16-bit element pairs

// Two elements packed in a 32-bit word (element 2i in the low half) -> fp32.
// Both conversions are exact.
template <class D>
__device__ __forceinline__ float2 unpack2(uint32_t w);

template <>
__device__ __forceinline__ float2 unpack2<Bf16>(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <>
__device__ __forceinline__ float2 unpack2<Fp16>(uint32_t w)
{
    __half2 h;
    memcpy(&h, &w, 4);
    return __half22float2(h);
}

// fp32 pair -> packed pair, each rounded to nearest even.
template <class D>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);

template <>
__device__ __forceinline__ uint32_t pack2<Bf16>(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    uint32_t w;
    memcpy(&w, &v, 4);
    return w;
}

template <>
__device__ __forceinline__ uint32_t pack2<Fp16>(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    uint32_t w;
    memcpy(&w, &v, 4);
    return w;
}

// 8 elements of a vector -> fp32 (exact)
template <class D>
__device__ __forceinline__ void unpack8(const typename D::Vec& v, float (&f)[8])
{
    if constexpr (D::bytes == 4) {
        f[0] = __uint_as_float(v.lo.x); f[1] = __uint_as_float(v.lo.y);
        f[2] = __uint_as_float(v.lo.z); f[3] = __uint_as_float(v.lo.w);
        f[4] = __uint_as_float(v.hi.x); f[5] = __uint_as_float(v.hi.y);
        f[6] = __uint_as_float(v.hi.z); f[7] = __uint_as_float(v.hi.w);
    } else {
        float2 p;
        p = unpack2<D>(v.x); f[0] = p.x; f[1] = p.y;
        p = unpack2<D>(v.y); f[2] = p.x; f[3] = p.y;
        p = unpack2<D>(v.z); f[4] = p.x; f[5] = p.y;
        p = unpack2<D>(v.w); f[6] = p.x; f[7] = p.y;
    }
}

// 8 fp32 -> a vector, each rounded to the element type (nearest even; the
// identity for fp32)
template <class D>
__device__ __forceinline__ typename D::Vec pack8(const float (&f)[8])
{
    typename D::Vec v;
    if constexpr (D::bytes == 4) {
        v.lo = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
        v.hi = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                          __float_as_uint(f[7]));
    } else {
        v.x = pack2<D>(f[0], f[1]);
        v.y = pack2<D>(f[2], f[3]);
        v.z = pack2<D>(f[4], f[5]);
        v.w = pack2<D>(f[6], f[7]);
    }
    return v;
}

// ------------------------------------------- mixed-precision accumulation
//
// add.rn.f32.{bf16,f16}: d = f(a) + c rounded once to fp32 -- the same value as
// unpacking a and adding, in one instruction.  Addition commutes exactly, so
// s + f(P_r) keeps the rank order of the fp32 sum.

template <class D>
__device__ __forceinline__ void add2(float& lo, float& hi, uint32_t w);

template <>
__device__ __forceinline__ void add2<Bf16>(float& lo, float& hi, uint32_t w)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(w));
}

template <>
__device__ __forceinline__ void add2<Fp16>(float& lo, float& hi, uint32_t w)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.f16 %0, l, %0;\n\tadd.rn.f32.f16 %1, h, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(w));
}

// s[i] = s[i] + f(v_i), i < 8
template <class D>
__device__ __forceinline__ void add8(float (&s)[8], const typename D::Vec& v)
{
    if constexpr (D::bytes == 4) {
        float t[8];
        unpack8<D>(v, t);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            s[i] = __fadd_rn(s[i], t[i]);
    } else {
        add2<D>(s[0], s[1], v.x);
        add2<D>(s[2], s[3], v.y);
        add2<D>(s[4], s[5], v.z);
        add2<D>(s[6], s[7], v.w);
    }
}

// rnd(f(a) + f(b)) for two packed 16-bit vectors, one packed add per pair:
// the fp32 sum of two bf16 (fp16) values rounded once more to bf16 (fp16)
// equals the correctly rounded sum (when the exact sum is not an fp32 value
// the smaller addend lies at least 16 (13) bits below the larger one's last
// bit, so the fp32 rounding cannot land on a 16-bit tie).
template <class D>
__device__ __forceinline__ uint4 add_packed(const uint4& a, const uint4& b);

template <>
__device__ __forceinline__ uint4 add_packed<Bf16>(const uint4& a, const uint4& b)
{
    uint4 r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r.x) : "r"(a.x), "r"(b.x));
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r.y) : "r"(a.y), "r"(b.y));
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r.z) : "r"(a.z), "r"(b.z));
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r.w) : "r"(a.w), "r"(b.w));
    return r;
}

template <>
__device__ __forceinline__ uint4 add_packed<Fp16>(const uint4& a, const uint4& b)
{
    uint4 r;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r.x) : "r"(a.x), "r"(b.x));
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r.y) : "r"(a.y), "r"(b.y));
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r.z) : "r"(a.z), "r"(b.z));
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r.w) : "r"(a.w), "r"(b.w));
    return r;
}

// Element-type accumulation (every partial sum rounded to the element type).
// For 16-bit elements the running sum stays packed: its four words ride, as
// bit copies, in the first four slots of the fp32 array, each rank is one
// packed add per pair (equal to the fp32 add rounded to the element type, as
// above), and elem_finish8 unpacks the final sum.  For fp32 elements it is the
// fp32 sum.
template <class D>
__device__ __forceinline__ void elem_start8(float (&s)[8], const typename D::Vec& v)
{
    if constexpr (D::bytes == 4) {
        unpack8<D>(v, s);
    } else {
        s[0] = __uint_as_float(v.x); s[1] = __uint_as_float(v.y);
        s[2] = __uint_as_float(v.z); s[3] = __uint_as_float(v.w);
    }
}

template <class D>
__device__ __forceinline__ void elem_add8(float (&s)[8], const typename D::Vec& v)
{
    if constexpr (D::bytes == 4) {
        add8<D>(s, v);
    } else {
        const uint4 w = add_packed<D>(make_uint4(__float_as_uint(s[0]), __float_as_uint(s[1]),
                                                 __float_as_uint(s[2]), __float_as_uint(s[3])),
                                      v);
        s[0] = __uint_as_float(w.x); s[1] = __uint_as_float(w.y);
        s[2] = __uint_as_float(w.z); s[3] = __uint_as_float(w.w);
    }
}

template <class D>
__device__ __forceinline__ void elem_finish8(float (&s)[8])
{
    if constexpr (D::bytes != 4) {
        const uint4 w = make_uint4(__float_as_uint(s[0]), __float_as_uint(s[1]),
                                   __float_as_uint(s[2]), __float_as_uint(s[3]));
        unpack8<D>(w, s);
    }
}

// Squares of a packed pair, exact (8- or 11-bit significands): fma with a
// -0.0 addend, so a zero element gives +0.
template <class D>
__device__ __forceinline__ void sq2(float& lo, float& hi, uint32_t w);

template <>
__device__ __forceinline__ void sq2<Bf16>(float& lo, float& hi, uint32_t w)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "fma.rn.f32.bf16 %0, l, l, 0f80000000;\n\tfma.rn.f32.bf16 %1, h, h, 0f80000000;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
}

template <>
__device__ __forceinline__ void sq2<Fp16>(float& lo, float& hi, uint32_t w)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "fma.rn.f32.f16 %0, l, l, 0f80000000;\n\tfma.rn.f32.f16 %1, h, h, 0f80000000;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
}

// ------------------------------------------------------------ memory ops

// Streaming 128-bit load of data read exactly once (no L1 allocation).
__device__ __forceinline__ uint4 ld_stream(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 128-bit load that re-reads memory on every call (Lamport slot polling).
__device__ __forceinline__ uint4 ld_poll(const void* p)
{
    uint4 v;
    asm volatile("ld.volatile.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Ask the copy engine to bring `bytes` (multiple of 16, 16-byte aligned) of
// global memory into L2 without waiting or using registers.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Cached 128-bit load (gamma: read by every row).
__device__ __forceinline__ uint4 ld_keep(const void* p)
{
    return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ void st_vec(void* p, const uint4& v)
{
    *reinterpret_cast<uint4*>(p) = v;
}

// 256-bit forms for 8 fp32 elements (32-byte aligned addresses)
__device__ __forceinline__ V32 ld_stream32(const void* p)
{
    V32 v;
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.lo.x), "=r"(v.lo.y), "=r"(v.lo.z), "=r"(v.lo.w), "=r"(v.hi.x),
                   "=r"(v.hi.y), "=r"(v.hi.z), "=r"(v.hi.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ V32 ld_poll32(const void* p)
{
    V32 v;
    asm volatile("ld.volatile.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.lo.x), "=r"(v.lo.y), "=r"(v.lo.z), "=r"(v.lo.w), "=r"(v.hi.x),
                   "=r"(v.hi.y), "=r"(v.hi.z), "=r"(v.hi.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ V32 ld_keep32(const void* p)
{
    V32 v;
    asm("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(v.lo.x), "=r"(v.lo.y), "=r"(v.lo.z), "=r"(v.lo.w), "=r"(v.hi.x), "=r"(v.hi.y),
          "=r"(v.hi.z), "=r"(v.hi.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ void st_vec(void* p, const V32& v)
{
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.lo.x),
                 "r"(v.lo.y), "r"(v.lo.z), "r"(v.lo.w), "r"(v.hi.x), "r"(v.hi.y), "r"(v.hi.z),
                 "r"(v.hi.w)
                 : "memory");
}

// Vector loads by element type: streaming (read once), polling (volatile),
// cached (gamma)
template <class D>
__device__ __forceinline__ typename D::Vec ld_stream_v(const void* p)
{
    if constexpr (D::bytes == 4)
        return ld_stream32(p);
    else
        return ld_stream(p);
}

template <class D>
__device__ __forceinline__ typename D::Vec ld_poll_v(const void* p)
{
    if constexpr (D::bytes == 4)
        return ld_poll32(p);
    else
        return ld_poll(p);
}

template <class D>
__device__ __forceinline__ typename D::Vec ld_keep_v(const void* p)
{
    if constexpr (D::bytes == 4)
        return ld_keep32(p);
    else
        return ld_keep(p);
}

template <class V>
__device__ __forceinline__ V zero_vec()
{
    V v;
    memset(&v, 0, sizeof v);
    return v;
}

__device__ __forceinline__ void st_u2(void* p, uint32_t a, uint32_t b)
{
    *reinterpret_cast<uint2*>(p) = make_uint2(a, b);
}

// Lamport sentinel (page "TensorRT-LLMs/cpp/tensorrt_llm/kernels/
// allReduceFusionKernels.cu", the one-shot Lamport kernel): a slot word whose
// 32 bits are those of -0.0f has not been written by its producer yet; true
// if any word of the vector is such a word.
__device__ __forceinline__ bool has_sentinel(const uint4& v)
{
    return (v.x == 0x80000000u) | (v.y == 0x80000000u) | (v.z == 0x80000000u) |
           (v.w == 0x80000000u);
}

__device__ __forceinline__ bool has_sentinel(const V32& v)
{
    return has_sentinel(v.lo) | has_sentinel(v.hi);
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_error(ar_fusion_state* st, int code, int detail)
{
    if (atomicCAS(&st->status, 0, code) == 0)
        atomicExch(&st->detail, detail);
}

// ------------------------------------------------------- clusters and PDL

// Thread-block cluster of this block: number of CTAs (1 when the kernel was
// launched without clusters), this CTA's rank, the cluster index and count.
__device__ __forceinline__ unsigned cluster_size()
{
    unsigned r;
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_rank()
{
    unsigned r;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_id()
{
    unsigned r;
    asm("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_count()
{
    unsigned r;
    asm("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster; release/acquire orders shared
// memory writes before the barrier with reads by other CTAs after it.
__device__ __forceinline__ void cluster_barrier()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A float pair at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ float2 ld_dsmem_f2(const void* local, unsigned rank)
{
    const uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(ra) : "memory");
    return v;
}

// Programmatic dependent launch: wait until the preceding grid in the stream
// has completed and its memory is visible (a no-op without the launch
// attribute), and allow the next grid to be scheduled early.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------- double-float accumulation
//
// Sum of squares as an unevaluated pair (hi, lo): every square of a 16-bit
// element is exact in fp32, and TwoSum keeps the rounding error of each
// addition, so hi + lo carries ~48 significant bits.  The pair is rounded to
// fp32 once at the end, which reproduces the correctly rounded sum except when
// the exact sum sits within ~2^-44 (relative) of an fp32 rounding boundary.

struct DF {
    float hi, lo;
};

// IEEE round-to-nearest fp32 addition on either side (no contraction: there
// is no multiply to fuse with).
__host__ __device__ __forceinline__ float rn_add(float a, float b)
{
#ifdef __CUDA_ARCH__
    return __fadd_rn(a, b);
#else
    return a + b;
#endif
}

// a += t for a non-negative running sum and term (sums of squares): ordering
// the two by max / min makes Dekker's fast two-sum exact (three additions
// instead of TwoSum's six); the new high part is hi + t itself, so a NaN term
// propagates.
__host__ __device__ __forceinline__ void df_add_nonneg(DF& a, float t)
{
    const float s = rn_add(a.hi, t);
    const float big = fmaxf(a.hi, t);
    const float small = fminf(a.hi, t);
    const float err = rn_add(rn_add(big, -s), small);
    a.hi = s;
    a.lo = rn_add(a.lo, err);
}

// Pair addition of two non-negative pairs (every pair summed here is a sum
// of squares): the high parts are added exactly by the fast two-sum with
// max / min ordering and every rounding error lands in lo; lo is not
// renormalised into hi between steps (its own rounding errors are ~2^-24 of
// an already tiny value).  The operation is symmetric in a and b, so every
// lane of an xor butterfly ends with the same bits.  (TwoSum's six-addition
// form measured 0.2-1% slower in the row kernels.)
__host__ __device__ __forceinline__ DF df_add(DF a, DF b)
{
    const float s = rn_add(a.hi, b.hi);
    const float err = rn_add(rn_add(fmaxf(a.hi, b.hi), -s), fminf(a.hi, b.hi));
    return DF{s, rn_add(rn_add(a.lo, b.lo), err)};
}

__host__ __device__ __forceinline__ float df_round(DF a)
{
    return rn_add(a.hi, a.lo);
}

// ------------------------------------------------------- packed fp32 pairs
//
// Two fp32 values handled by one packed instruction on the device
// (add / sub / mul .rn.f32x2: each lane rounded to nearest exactly as the
// scalar instruction, subnormals kept); the host form does the same per lane.

struct F2 {
    float x, y;
};

#ifdef __CUDA_ARCH__
#define AR_F2_OP(name, op)                                                              \
    __host__ __device__ __forceinline__ F2 name(F2 a, F2 b)                             \
    {                                                                                   \
        F2 r;                                                                           \
        asm("{\n\t.reg .b64 pa, pb, pr;\n\tmov.b64 pa, {%2, %3};\n\t"                     \
            "mov.b64 pb, {%4, %5};\n\t" op " pr, pa, pb;\n\tmov.b64 {%0, %1}, pr;\n\t}"    \
            : "=f"(r.x), "=f"(r.y)                                                      \
            : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));                                  \
        return r;                                                                       \
    }
#else
#define AR_F2_OP(name, op)                                                              \
    __host__ __device__ __forceinline__ F2 name(F2 a, F2 b)                             \
    {                                                                                   \
        return F2{name##_1(a.x, b.x), name##_1(a.y, b.y)};                              \
    }
__host__ __device__ __forceinline__ float f2_add_1(float a, float b) { return a + b; }
__host__ __device__ __forceinline__ float f2_sub_1(float a, float b) { return a - b; }
__host__ __device__ __forceinline__ float f2_mul_1(float a, float b) { return a * b; }
#endif
AR_F2_OP(f2_add, "add.rn.f32x2")
AR_F2_OP(f2_sub, "sub.rn.f32x2")
AR_F2_OP(f2_mul, "mul.rn.f32x2")
#undef AR_F2_OP

// Two double-float accumulators side by side (lane 0: even elements, lane 1:
// odd elements), updated by one TwoSum per lane in packed instructions:
// hi + lo keeps the exact sum of the terms up to the rounding of lo, as DF.
struct DF2 {
    F2 hi, lo;
};

// a += t per lane (TwoSum on the high parts, its error into lo; exact for
// any two finite terms, no ordering needed)
__host__ __device__ __forceinline__ void df2_add_terms(DF2& a, F2 t)
{
    const F2 s = f2_add(a.hi, t);
    const F2 bb = f2_sub(s, a.hi);
    const F2 err = f2_add(f2_sub(a.hi, f2_sub(s, bb)), f2_sub(t, bb));
    a.hi = s;
    a.lo = f2_add(a.lo, err);
}

// the two lanes as one pair (a TwoSum of the high parts, as df_add)
__host__ __device__ __forceinline__ DF df2_merge(const DF2& a)
{
    return df_add(DF{a.hi.x, a.lo.x}, DF{a.hi.y, a.lo.y});
}

__device__ __forceinline__ DF df_shfl_xor(DF a, int m)
{
    return DF{__shfl_xor_sync(0xffffffffu, a.hi, m), __shfl_xor_sync(0xffffffffu, a.lo, m)};
}

__device__ __forceinline__ DF df_warp_sum(DF a)
{
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        a = df_add(a, df_shfl_xor(a, m));
    return a;
}

// ----------------------------------------------------- FP8 / FP4 encoders
//
// PTX cvt with .satfinite: round to nearest even, finite overflow and
// infinities saturate to the largest finite code, sign of zero kept.
// Operand order: the first source lands in the upper part of the result.

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// 8 fp32 -> 8 E4M3 bytes (element 0 in the lowest byte)
__device__ __forceinline__ uint2 e4m3x8(const float (&f)[8])
{
    uint2 o;
    o.x = e4m3x2(f[0], f[1]) | (e4m3x2(f[2], f[3]) << 16);
    o.y = e4m3x2(f[4], f[5]) | (e4m3x2(f[6], f[7]) << 16);
    return o;
}

__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 q;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q, %1, %2;\n\t"
        "cvt.u32.u8 %0, q;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// 8 fp32 -> 8 E2M1 codes in 4 bytes (element 2k in the low nibble of byte k)
__device__ __forceinline__ uint32_t e2m1x8(const float (&f)[8])
{
    return e2m1x2(f[0], f[1]) | (e2m1x2(f[2], f[3]) << 8) | (e2m1x2(f[4], f[5]) << 16) |
           (e2m1x2(f[6], f[7]) << 24);
}

// E4M3 byte -> fp32 (exact: E4M3 values are a subset of fp16)
__device__ __forceinline__ float e4m3_to_f32(uint32_t code)
{
    uint32_t h2;
    uint16_t in = (uint16_t)code;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    __half2 h;
    memcpy(&h, &h2, 4);
    return __low2float(h);
}

__device__ __forceinline__ uint32_t e4m3_byte(float v)
{
    return e4m3x2(v, 0.0f) & 0xffu;
}

}  // namespace arf
