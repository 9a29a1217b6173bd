// Launch selection for the register-resident row kernels (one element type
// per translation unit so the instantiations compile in parallel).
#pragma once

#include <mutex>
#include <map>
#include <utility>

#include "fused_rows.cuh"

namespace arf {

template <class D, int RMAX, bool WARP_ROW>
static const void* rows_fn_vpt(int vpt)
{
    switch (vpt) {
    case 1: return (const void*)fused_rows_kernel<D, RMAX, 1, WARP_ROW>;
    case 2: return (const void*)fused_rows_kernel<D, RMAX, 2, WARP_ROW>;
    case 4: return (const void*)fused_rows_kernel<D, RMAX, 4, WARP_ROW>;
    case 8:
        if constexpr (WARP_ROW)
            return nullptr;
        else
            return (const void*)fused_rows_kernel<D, RMAX, 8, WARP_ROW>;
    default: return nullptr;
    }
}

template <class D, bool WARP_ROW>
static const void* rows_fn(int rmax, int vpt)
{
    switch (rmax) {
    case 2: return rows_fn_vpt<D, 2, WARP_ROW>(vpt);
    case 4: return rows_fn_vpt<D, 4, WARP_ROW>(vpt);
    case 8: return rows_fn_vpt<D, 8, WARP_ROW>(vpt);
    case 16: return rows_fn_vpt<D, 16, WARP_ROW>(vpt);
    default: return nullptr;
    }
}

static inline int blocks_per_sm(const void* fn, int threads)
{
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> cache;
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(fn, threads);
    auto it = cache.find(key);
    if (it != cache.end())
        return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, 0) != cudaSuccess || n < 1)
        n = 1;
    cache[key] = n;
    return n;
}

static inline int pow2_at_least(int x)
{
    int p = 1;
    while (p < x)
        p <<= 1;
    return p;
}

// Geometry:
//   WARP_ROW: 8 warps per block, one row per warp, VPT = ceil(Hv / 32) in
//             {1, 2, 4} (hidden <= 1024).
//   CTA_ROW : one row per block; one vector per thread up to 896 threads
//             (hidden <= 7168; up to 1024 threads, hidden <= 8192, with at
//             most 4 ranks), else VPT in {2, 4, 8} with <= 512 threads
//             (hidden <= 32768).
// Grid: enough blocks for every row, capped at what is resident at once
// (rows are then strided over the resident blocks).
template <class D>
cudaError_t launch_fused_rows_t(int variant, const FusedArgs& a, const LaunchCfg& c)
{
    const int Hv = a.H / 8;
    const int rmax = a.R <= 2 ? 2 : a.R <= 4 ? 4 : a.R <= 8 ? 8 : 16;
    const void* fn;
    int threads, grid;
    if (variant == AR_VARIANT_WARP_ROW) {
        const int vpt = pow2_at_least((Hv + 31) / 32);
        if (vpt > 4)
            return cudaErrorInvalidValue;
        fn = rows_fn<D, true>(rmax, vpt);
        threads = 256;
        const int need = (a.T + 7) / 8;
        const int cap = c.sms * blocks_per_sm(fn, threads);
        grid = need < cap ? need : cap;
    } else {
        // one vector per thread up to 896 threads, else <= 512 threads
        // (two vectors per thread measured 208 us vs 188 us at H = 7168)
        const int one_vec_max = rmax <= 4 ? 1024 : 896;
        const int vpt = Hv <= one_vec_max ? 1 : pow2_at_least((Hv + 511) / 512);
        if (vpt > 8)
            return cudaErrorInvalidValue;
        fn = rows_fn<D, false>(rmax, vpt);
        threads = ((Hv + vpt - 1) / vpt + 31) / 32 * 32;
        const int cap = c.sms * blocks_per_sm(fn, threads);
        grid = a.T < cap ? a.T : cap;
    }
    if (!fn)
        return cudaErrorInvalidValue;
    if (grid < 1)
        grid = 1;
    void* args[] = {const_cast<FusedArgs*>(&a)};
    return cudaLaunchKernel(fn, dim3(grid), dim3(threads), args, 0, c.stream);
}

}  // namespace arf
