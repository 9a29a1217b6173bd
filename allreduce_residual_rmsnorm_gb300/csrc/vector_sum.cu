// Plain R-way sum, out[i] = rnd(sum_r f(in_r[i])) in fp32, rank order
// (mscclpp allreduce.cu: vectorSum, here out of place over R inputs and with
// fp32 accumulation).
//
// Vector-aligned inputs (16 bytes; 32 for fp32): grid-stride over vectors of
// 8 elements, two vectors per thread per step so 2R loads are in flight, and
// the n % 8 tail elements done one by one (the page's vectorSum drops nothing
// either: its 32-bit tail loop covers the rest).  16-bit elements at any
// element offset: aligned 16-byte loads realigned in registers.  Large
// 16-bit sums with 32-byte aligned pointers: 256-bit loads.  Misaligned fp32
// pointers: element-wise kernel.
#include <atomic>

#include "ar_common.cuh"
#include "ar_internal.h"

namespace arf {

template <class D>
__device__ __forceinline__ float ld_elem(const uint8_t* p, uint64_t i)
{
    if constexpr (D::bytes == 4)
        return reinterpret_cast<const float*>(p)[i];
    const uint16_t b = reinterpret_cast<const uint16_t*>(p)[i];
    if constexpr (D::id == AR_DT_BF16) {
        return __uint_as_float((uint32_t)b << 16);
    } else {
        __half h;
        memcpy(&h, &b, 2);
        return __half2float(h);
    }
}

template <class D>
__device__ __forceinline__ void st_elem(uint8_t* p, uint64_t i, float v)
{
    if constexpr (D::bytes == 4) {
        reinterpret_cast<float*>(p)[i] = v;
        return;
    }
    uint16_t b;
    if constexpr (D::id == AR_DT_BF16) {
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        memcpy(&b, &h, 2);
    } else {
        __half h = __float2half_rn(v);
        memcpy(&b, &h, 2);
    }
    reinterpret_cast<uint16_t*>(p)[i] = b;
}

// f(rnd(v)) in the element type
template <class D>
__device__ __forceinline__ float round1(float v)
{
    if constexpr (D::bytes == 4)
        return v;
    else if constexpr (D::id == AR_DT_BF16)
        return __bfloat162float(__float2bfloat16_rn(v));
    else
        return __half2float(__float2half_rn(v));
}

template <class D, int RMAX>
__device__ __forceinline__ typename D::Vec sum_vec(const SumArgs& a,
                                                   const typename D::Vec (&raw)[RMAX])
{
    if constexpr (D::bytes == 2) {
        // element-type adds: one packed add per pair and rank
        if (a.acc) {
            typename D::Vec s = raw[0];
#pragma unroll
            for (int r = 1; r < RMAX; ++r)
                if (r < a.R)
                    s = add_packed<D>(s, raw[r]);
            return s;
        }
    }
    float s[8];
    unpack8<D>(raw[0], s);
#pragma unroll
    for (int r = 1; r < RMAX; ++r) {
        if (r < a.R) {
            float t[8];
            unpack8<D>(raw[r], t);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                s[i] = __fadd_rn(s[i], t[i]);
        }
    }
    return pack8<D>(s);
}

// One element of the rank-order sum (same adds and roundings as sum_vec),
// in two halves: every rank's load is issued first (load_elem), before the
// thread's vector work, and added after it (fold_elem), so the element costs
// no memory round trip of its own on the kernel's critical path (a loop of
// load + add over the run-time rank count cost one per rank).
template <class D, int RMAX>
__device__ __forceinline__ void load_elem(const SumArgs& a, uint64_t e, float (&v)[RMAX])
{
#pragma unroll
    for (int r = 0; r < RMAX; ++r)
        v[r] = r < a.R ? ld_elem<D>(a.in[r], e) : 0.0f;
}

template <class D, int RMAX>
__device__ __forceinline__ float fold_elem(const SumArgs& a, const float (&v)[RMAX])
{
    float s = v[0];
#pragma unroll
    for (int r = 1; r < RMAX; ++r) {
        if (r < a.R) {
            s = __fadd_rn(s, v[r]);
            if (a.acc)
                s = round1<D>(s);
        }
    }
    return s;
}

template <class D, int RMAX>
__global__ void __launch_bounds__(256) vector_sum_kernel(const SumArgs a)
{
    using V = typename D::Vec;
    constexpr uint64_t VB = 8 * D::bytes;
    const uint64_t nvec = a.n / 8;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint64_t i = tid;
    for (; i + stride < nvec; i += 2 * stride) {
        V r0[RMAX], r1[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            if (r < a.R) {
                r0[r] = ld_stream_v<D>(a.in[r] + i * VB);
                r1[r] = ld_stream_v<D>(a.in[r] + (i + stride) * VB);
            }
        }
        st_vec(a.out + i * VB, sum_vec<D, RMAX>(a, r0));
        st_vec(a.out + (i + stride) * VB, sum_vec<D, RMAX>(a, r1));
    }
    if (i < nvec) {
        V r0[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
            if (r < a.R)
                r0[r] = ld_stream_v<D>(a.in[r] + i * VB);
        st_vec(a.out + i * VB, sum_vec<D, RMAX>(a, r0));
    }
    const uint64_t tail = a.n - nvec * 8;
    if (tid < tail) {
        const uint64_t e = nvec * 8 + tid;
        float v[RMAX];
        load_elem<D, RMAX>(a, e, v);
        st_elem<D>(a.out, e, fold_elem<D, RMAX>(a, v));
    }
}

// 16-bit elements, every pointer 32-byte aligned, large n: items of 16
// elements (one 256-bit load per rank), STEPS items per thread per step (2R
// loads of 32 bytes in flight), each summed as two 8-element halves; the
// n % 16 tail element by element.  Measured at R=8 fp16 against two 16-byte
// vectors per step: N=268,435,456 740.7 -> 677.2 us, N=67,108,864 185.4 ->
// 171.8 us; slower at N=16,777,216 (42.9 -> 46.3 us: one 256-thread block
// per SM hides less latency over few steps), hence the size threshold.
template <class D, int RMAX, int STEPS>
__global__ void __launch_bounds__(256) vector_sum_wide_kernel(const SumArgs a)
{
    using V = typename D::Vec;
    static_assert(D::bytes == 2, "16-bit elements");
    const uint64_t n16 = a.n / 16;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint64_t i = tid;
    for (; i + (STEPS - 1) * stride < n16; i += STEPS * stride) {
        V lo[STEPS][RMAX], hi[STEPS][RMAX];
#pragma unroll
        for (int k = 0; k < STEPS; ++k)
#pragma unroll
            for (int r = 0; r < RMAX; ++r)
                if (r < a.R) {
                    const V32 w = ld_stream32(a.in[r] + (i + k * stride) * 32);
                    lo[k][r] = w.lo;
                    hi[k][r] = w.hi;
                }
#pragma unroll
        for (int k = 0; k < STEPS; ++k) {
            V32 o;
            o.lo = sum_vec<D, RMAX>(a, lo[k]);
            o.hi = sum_vec<D, RMAX>(a, hi[k]);
            st_vec(a.out + (i + k * stride) * 32, o);
        }
    }
    for (; i < n16; i += stride) {
        V lo[RMAX], hi[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
            if (r < a.R) {
                const V32 w = ld_stream32(a.in[r] + i * 32);
                lo[r] = w.lo;
                hi[r] = w.hi;
            }
        V32 o;
        o.lo = sum_vec<D, RMAX>(a, lo);
        o.hi = sum_vec<D, RMAX>(a, hi);
        st_vec(a.out + i * 32, o);
    }
    const uint64_t tail = a.n - n16 * 16;
    if (tid < tail) {
        const uint64_t e = n16 * 16 + tid;
        float v[RMAX];
        load_elem<D, RMAX>(a, e, v);
        st_elem<D>(a.out, e, fold_elem<D, RMAX>(a, v));
    }
}

// Bytes [m, m + 16) of the 32 bytes a:b (m even, 0..14): the 16-byte vector
// that starts m bytes into the aligned block a.  m is the same for every
// thread (one input's misalignment), so the selection does not diverge.
__device__ __forceinline__ uint4 realign16(const uint4& a, const uint4& b, uint32_t m)
{
    uint32_t w0, w1, w2, w3, w4;
    switch (m >> 2) {
    case 0: w0 = a.x; w1 = a.y; w2 = a.z; w3 = a.w; w4 = b.x; break;
    case 1: w0 = a.y; w1 = a.z; w2 = a.w; w3 = b.x; w4 = b.y; break;
    case 2: w0 = a.z; w1 = a.w; w2 = b.x; w3 = b.y; w4 = b.z; break;
    default: w0 = a.w; w1 = b.x; w2 = b.y; w3 = b.z; w4 = b.w; break;
    }
    const uint32_t sh = (m & 2u) * 8u;   // 0 or 16 bits: odd element offset
    return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                      __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh));
}

// 16-bit elements, inputs or output not 16-byte aligned.  The output's
// 16-byte grid, from its first aligned element h, defines vectors j of 8
// elements; input r holds vector j at an address m_r bytes past a 16-byte
// boundary (m_r the same for every j), read as the two aligned 16-byte
// blocks that cover it and realigned in registers.  Vectors 1 .. nv-2 take
// this path; their blocks lie inside the inputs (the block after vector j's
// is inside vector j+1, the block before it inside vector j-1).  Elements
// before vector 1 and from vector nv-1 on are summed one by one.
template <class D, int RMAX>
__global__ void __launch_bounds__(256) vector_sum_shift_kernel(const SumArgs a, const uint64_t h,
                                                                const uint64_t nv)
{
    using V = typename D::Vec;
    static_assert(D::bytes == 2, "16-bit elements");
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // element by element: [0, h + 8) and [h + 8 * (nv - 1), n), element k by
    // the grid's thread stride - 1 - k, which the launch leaves without
    // vectors when the grid is not capped (so these elements add no memory
    // round trip after a thread's vectors)
    const uint64_t n_head = h + 8, tail0 = h + 8 * (nv - 1);
    const uint64_t n_elem = n_head + (a.n - tail0);
    if (tid + n_elem >= stride) {
        const uint64_t k = stride - 1 - tid;
        const uint64_t e = k < n_head ? k : tail0 + (k - n_head);
        float ev[RMAX];
        load_elem<D, RMAX>(a, e, ev);
        st_elem<D>(a.out, e, fold_elem<D, RMAX>(a, ev));
    }
    for (uint64_t j = 1 + tid; j + 1 < nv; j += stride) {
        const uint64_t off = 2 * (h + 8 * j);
        V raw[RMAX];
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
            if (r < a.R) {
                const uintptr_t p = (uintptr_t)a.in[r] + off;
                const uint32_t m = (uint32_t)(p & 15u);
                const uint4* blk = reinterpret_cast<const uint4*>(p - m);
                const uint4 lo = __ldg(blk);
                raw[r] = m ? realign16(lo, __ldg(blk + 1), m) : lo;
            }
        }
        st_vec(a.out + off, sum_vec<D, RMAX>(a, raw));
    }
}

template <class D>
__global__ void __launch_bounds__(256) vector_sum_scalar_kernel(const SumArgs a)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t e = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; e < a.n; e += stride) {
        float s = ld_elem<D>(a.in[0], e);
        for (int r = 1; r < a.R; ++r) {
            s = __fadd_rn(s, ld_elem<D>(a.in[r], e));
            if (a.acc)
                s = round1<D>(s);
        }
        st_elem<D>(a.out, e, s);
    }
}

template <class D>
static const void* sum_fn(int rmax)
{
    switch (rmax) {
    case 2: return (const void*)vector_sum_kernel<D, 2>;
    case 4: return (const void*)vector_sum_kernel<D, 4>;
    case 8: return (const void*)vector_sum_kernel<D, 8>;
    case 16: return (const void*)vector_sum_kernel<D, 16>;
    default: return nullptr;
    }
}

template <class D>
static const void* shift_fn(int rmax)
{
    if constexpr (D::bytes == 2) {
        switch (rmax) {
        case 2: return (const void*)vector_sum_shift_kernel<D, 2>;
        case 4: return (const void*)vector_sum_shift_kernel<D, 4>;
        case 8: return (const void*)vector_sum_shift_kernel<D, 8>;
        case 16: return (const void*)vector_sum_shift_kernel<D, 16>;
        default: return nullptr;
        }
    }
    return nullptr;
}

constexpr int kWideSteps = 2;
// elements from which 16-bit sums take the 256-bit-load kernel
constexpr uint64_t kWideMinN = 1ull << 25;

template <class D>
static const void* wide_fn(int rmax)
{
    if constexpr (D::bytes == 2) {
        switch (rmax) {
        case 2: return (const void*)vector_sum_wide_kernel<D, 2, kWideSteps>;
        case 4: return (const void*)vector_sum_wide_kernel<D, 4, kWideSteps>;
        case 8: return (const void*)vector_sum_wide_kernel<D, 8, kWideSteps>;
        default: return nullptr;   // 16 ranks: registers for one step only
        }
    }
    return nullptr;
}

template <class D>
static cudaError_t launch_t(const SumArgs& a, const LaunchCfg& c)
{
    constexpr uintptr_t vmask = 8 * D::bytes - 1;
    bool aligned = ((uintptr_t)a.out & vmask) == 0;
    for (int r = 0; r < a.R; ++r)
        aligned = aligned && ((uintptr_t)a.in[r] & vmask) == 0;
    const int threads = 256;
    void* args[] = {const_cast<SumArgs*>(&a)};
    const int rmax = a.R <= 2 ? 2 : a.R <= 4 ? 4 : a.R <= 8 ? 8 : 16;
    if (!aligned && D::bytes == 2) {
        // elements before the output's first 16-byte boundary, then whole vectors
        const uint64_t h = ((16u - ((uintptr_t)a.out & 15u)) & 15u) / 2u;
        const uint64_t nv = a.n > h ? (a.n - h) / 8 : 0;
        if (nv >= 3) {
            const void* fn = shift_fn<D>(rmax);
            // vectors 1 .. nv-2, then the element-by-element head and tail
            // (at most 8 + 15 elements) on threads of their own
            const uint64_t n_elem = h + 8 + (a.n - (h + 8 * (nv - 1)));
            uint64_t blocks = (nv - 2 + n_elem + threads - 1) / threads;
            const uint64_t cap = (uint64_t)c.sms * 8;
            if (blocks > cap)
                blocks = cap;
            uint64_t hh = h, nvv = nv;
            void* sargs[] = {const_cast<SumArgs*>(&a), &hh, &nvv};
            return cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3(threads), sargs, 0, c.stream);
        }
    }
    if (!aligned) {
        uint64_t blocks = (a.n + threads - 1) / threads;
        const uint64_t cap = (uint64_t)c.sms * 8;
        if (blocks > cap)
            blocks = cap;
        if (blocks < 1)
            blocks = 1;
        return cudaLaunchKernel((const void*)vector_sum_scalar_kernel<D>, dim3((unsigned)blocks),
                                dim3(threads), args, 0, c.stream);
    }
    bool aligned32 = ((uintptr_t)a.out & 31u) == 0;
    for (int r = 0; r < a.R; ++r)
        aligned32 = aligned32 && ((uintptr_t)a.in[r] & 31u) == 0;
    if (D::bytes == 2 && aligned32 && a.n >= kWideMinN && rmax <= 8) {
        const void* fn = wide_fn<D>(rmax);
        static std::atomic<int> wcached[3][17] = {};
        int per_sm = wcached[D::id][rmax].load(std::memory_order_relaxed);
        if (per_sm == 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, 0) !=
                    cudaSuccess ||
                per_sm < 1)
                per_sm = 1;
            wcached[D::id][rmax].store(per_sm, std::memory_order_relaxed);
        }
        uint64_t blocks = (a.n / 16 + kWideSteps * threads - 1) / (kWideSteps * threads);
        const uint64_t cap = (uint64_t)c.sms * per_sm;
        if (blocks > cap)
            blocks = cap;
        if (blocks < 1)
            blocks = 1;
        return cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3(threads), args, 0, c.stream);
    }
    const void* fn = sum_fn<D>(rmax);
    // blocks per SM, per type and RMAX (atomic: calls may come from several
    // host threads; every writer stores the same value)
    static std::atomic<int> cached[3][17] = {};
    int per_sm = cached[D::id][rmax].load(std::memory_order_relaxed);
    if (per_sm == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, 0) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        cached[D::id][rmax].store(per_sm, std::memory_order_relaxed);
    }
    const uint64_t nvec = a.n / 8;
    // two vectors per thread per step; at least one block (the tail needs it)
    uint64_t blocks = (nvec + 2 * threads - 1) / (2 * threads);
    const uint64_t cap = (uint64_t)c.sms * per_sm;
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    return cudaLaunchKernel(fn, dim3((unsigned)blocks), dim3(threads), args, 0, c.stream);
}

cudaError_t launch_vector_sum(int dtype, const SumArgs& a, const LaunchCfg& c)
{
    switch (dtype) {
    case AR_DT_BF16: return launch_t<Bf16>(a, c);
    case AR_DT_FP16: return launch_t<Fp16>(a, c);
    case AR_DT_FP32: return launch_t<F32>(a, c);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace arf
