// One row per thread block with the block's next row copied into shared
// memory while the current one is reduced and normalised
// (AR_VARIANT_CTA_ROW_ASYNC).
//
// Same operation and arithmetic as the one-vector-per-thread row kernel
// (TensorRT-LLM allReduceFusionKernels.cu: allreduce_sum, fused_op, add128,
// rms_norm): thread g owns vector g (8 elements, 16 bytes) of every row of its
// block, sums the R partials in rank order, adds the residual, takes part in
// the row's sum of squares and writes the normalised and quantised outputs.
//
// What differs is where a row's inputs come from.  Each thread has R + 1
// private 16-byte slots in shared memory.  It copies its vector of the
// block's next row from each rank (and the residual) into them with cp.async
// right after the current row's first block barrier, so those copies are in
// flight during the row's warp-0 combine, its second barrier and the
// normalisation, and the next row starts from shared memory instead of
// waiting on global loads.  The first barrier also orders every thread's
// reads of its slots before the copies that overwrite them.
//
// Scope: 16-bit elements, staged buffer or caller partials (no Lamport
// polling), at most 8 ranks, one vector per thread of a row block.
#include <cuda_runtime.h>

#include <mutex>
#include <set>
#include <utility>

#include "fused_core.cuh"

namespace arf {
namespace {

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16 bytes global -> shared, cached in L2 only
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_slot(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}

template <class D>
constexpr int async_max_threads(int rmax)
{
    return one_vec_threads_for(D::bytes, rmax);
}

// shared memory of a block: R + 1 slots of 16 bytes per thread
constexpr size_t async_smem_bytes(int nranks, int threads)
{
    return (size_t)(nranks + 1) * (size_t)threads * 16;
}

template <class D, int RMAX>
__global__ void __launch_bounds__(async_max_threads<D>(RMAX), 1)
fused_rows_async_kernel(const FusedArgs a)
{
    using V = typename D::Vec;
    static_assert(D::bytes == 2, "16-bit elements");
    extern __shared__ uint4 slots[];   // [R + 1][blockDim.x]

    const int H = a.H;
    const int Hv = H >> 3;
    const int R = a.R;
    const int pat = a.pattern;
    const int g = threadIdx.x;
    const int lane = g & 31;
    const int warp = g >> 5;
    const int nwarps = blockDim.x >> 5;
    const bool own = g < Hv;
    const size_t rowb = (size_t)H * 2;
    // this thread's slot of rank r: base + r * rstride (rank R: the residual)
    const uint32_t base = smem_addr(slots + g);
    const uint32_t rstride = blockDim.x * 16u;

    // inputs may be written by the preceding grid
    pdl_wait();

    float qscale = 0.0f;
    if (pat & (AR_QUANT_FP8 | AR_QUANT_NVFP4))
        qscale = *a.scale_factor;
    float gf[8];
    load_gamma<D>(a.gamma, g, own, gf);

    __shared__ DF red[2][32];
    __shared__ float rstd_sh[2];
    int parity = 0;
    float amax_local = 0.0f;

    // copies of `row` into this thread's slots (none past the last row); one
    // commit group per call, so that wait_all covers exactly what was issued
    auto issue = [&](int row) {
        if (own && row < a.T) {
            const size_t off = (size_t)row * rowb + (size_t)g * 16;
#pragma unroll
            for (int r = 0; r < RMAX; ++r)
                if (r < R)
                    cp_async16(base + (uint32_t)r * rstride, a.partial[r] + off);
            cp_async16(base + (uint32_t)R * rstride, a.residual_in + off);
        }
        cp_async_commit();
    };

    int row = blockIdx.x;
    issue(row);
    for (; row < a.T; row += gridDim.x) {
        // this thread's copies of the row have landed
        cp_async_wait_all();
        DF ss = {0.0f, 0.0f};
        V y = zero_vec<V>();
        if (own) {
            float s[8];
            if (!a.acc) {
                unpack8<D>(ld_slot(base), s);
#pragma unroll
                for (int r = 1; r < RMAX; ++r)
                    if (r < R)
                        add8<D>(s, ld_slot(base + (uint32_t)r * rstride));
            } else {
                elem_start8<D>(s, ld_slot(base));
#pragma unroll
                for (int r = 1; r < RMAX; ++r)
                    if (r < R)
                        elem_add8<D>(s, ld_slot(base + (uint32_t)r * rstride));
                elem_finish8<D>(s);
            }
            y = residual_vec<D>(s, ld_slot(base + (uint32_t)R * rstride), ss);
            if (pat & AR_RESIDUAL_OUT)
                st_vec(a.residual_out + (size_t)row * rowb + (size_t)g * 16, y);
        }

        // row sum of squares: warp partials, barrier, warp 0 combines
        ss = df_warp_sum(ss);
        if (lane == 0)
            red[parity][warp] = ss;
        __syncthreads();
        // every slot of this row has been read: copy the next row in
        issue(row + gridDim.x);
        if (warp == 0) {
            DF v = lane < nwarps ? red[parity][lane] : DF{0.0f, 0.0f};
            v = df_warp_sum(v);
            if (lane == 0)
                rstd_sh[parity] = inv_rms(v, H, a.eps);
        }
        __syncthreads();
        const float rstd = rstd_sh[parity];
        parity ^= 1;

        normalize_vec<D>(a, pat, row, g, own, y, gf, rstd, qscale, amax_local);
    }
    // the last issue copied nothing; leave with no copy in flight all the same
    cp_async_wait_all();
    pdl_trigger();

    if (a.amax_out) {
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1)
            amax_local = fmaxf(amax_local, __shfl_xor_sync(0xffffffffu, amax_local, m));
        if (lane == 0)
            atomicMax(reinterpret_cast<unsigned int*>(a.amax_out), __float_as_uint(amax_local));
    }
}

template <class D>
const void* async_fn(int rmax)
{
    switch (rmax) {
    case 2: return (const void*)fused_rows_async_kernel<D, 2>;
    case 4: return (const void*)fused_rows_async_kernel<D, 4>;
    case 8: return (const void*)fused_rows_async_kernel<D, 8>;
    default: return nullptr;
    }
}

// the dynamic shared memory bound, raised once per device and kernel
cudaError_t allow_smem(const void* fn, size_t bytes)
{
    static std::mutex mu;
    static std::set<std::pair<int, const void*>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(mu);
    if (done.count({dev, fn}))
        return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess)
        done.insert({dev, fn});
    return e;
}

template <class D>
cudaError_t launch_t(const FusedArgs& a, const LaunchCfg& c)
{
    const int rmax = a.R <= 2 ? 2 : a.R <= 4 ? 4 : 8;
    const void* fn = async_fn<D>(rmax);
    if (!fn)
        return cudaErrorInvalidValue;
    const int Hv = a.H / 8;
    const int threads = (Hv + 31) / 32 * 32;
    cudaError_t e = allow_smem(fn, async_smem_bytes(rmax, async_max_threads<D>(rmax)));
    if (e != cudaSuccess)
        return e;
    const int grid = a.T < c.sms ? a.T : c.sms;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    int na = 0;
    cfg.gridDim = dim3(grid < 1 ? 1 : grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = async_smem_bytes(a.R, threads);
    cfg.stream = c.stream;
    if (c.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (c.used_cluster)
        *c.used_cluster = 1;
    void* args[] = {const_cast<FusedArgs*>(&a)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

bool fused_rows_async_supported(int dtype, int H, int R, bool lamport)
{
    if (lamport || (dtype != AR_DT_BF16 && dtype != AR_DT_FP16) || R < 1 || R > 8 || H % 8 != 0)
        return false;
    return H / 8 <= one_vec_threads_for(2, R);
}

cudaError_t launch_fused_rows_async(int dtype, const FusedArgs& a, const LaunchCfg& c)
{
    if (!fused_rows_async_supported(dtype, a.H, a.R, a.lamport != 0))
        return cudaErrorInvalidValue;
    return dtype == AR_DT_BF16 ? launch_t<Bf16>(a, c) : launch_t<Fp16>(a, c);
}

}  // namespace arf
