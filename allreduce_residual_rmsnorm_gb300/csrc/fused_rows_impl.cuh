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
    case 3:
        // 16-bit rows, at most 4 ranks (the load batch must divide 3 vectors)
        if constexpr (!WARP_ROW && RMAX <= 4 && D::bytes == 2)
            return (const void*)fused_rows_kernel<D, RMAX, 3, WARP_ROW>;
        else
            return nullptr;
    case 4: return (const void*)fused_rows_kernel<D, RMAX, 4, WARP_ROW>;
    case 8:
        if constexpr (WARP_ROW)
            return nullptr;
        else
            return (const void*)fused_rows_kernel<D, RMAX, 8, WARP_ROW>;
    default: return nullptr;
    }
}

// two rows per SM (16-bit): two vectors per thread with at most 4 ranks, one
// vector per thread with 5..8
template <class D>
static const void* rows_light_fn(int rmax)
{
    if constexpr (D::bytes == 2) {
        switch (rmax) {
        case 2: return (const void*)fused_rows_kernel<D, 2, 2, false, false, true>;
        case 4: return (const void*)fused_rows_kernel<D, 4, 2, false, false, true>;
        case 8: return (const void*)fused_rows_kernel<D, 8, 1, false, false, true>;
        default: return nullptr;
        }
    }
    return nullptr;
}

// one or two vectors per thread, one row per block, buffer mode only (no
// Lamport code)
template <class D, int VPT>
static const void* rows_buf_fn_vpt(int rmax)
{
    switch (rmax) {
    case 2: return (const void*)fused_rows_kernel<D, 2, VPT, false, false, false, false, true>;
    case 4: return (const void*)fused_rows_kernel<D, 4, VPT, false, false, false, false, true>;
    case 8: return (const void*)fused_rows_kernel<D, 8, VPT, false, false, false, false, true>;
    case 16: return (const void*)fused_rows_kernel<D, 16, VPT, false, false, false, false, true>;
    default: return nullptr;
    }
}

template <class D>
static const void* rows_buf_fn(int rmax, int vpt)
{
    return vpt == 1 ? rows_buf_fn_vpt<D, 1>(rmax) : vpt == 2 ? rows_buf_fn_vpt<D, 2>(rmax) : nullptr;
}

template <class D>
static const void* rows_ahead_fn()
{
    if constexpr (D::bytes == 2)
        return (const void*)fused_rows_kernel<D, 8, 1, false, false, false, true>;
    return nullptr;
}

// one-vector-per-thread row kernels launched with a cluster
template <class D>
static const void* rows_cluster_fn(int rmax)
{
    switch (rmax) {
    case 2: return (const void*)fused_rows_kernel<D, 2, 1, false, true>;
    case 4: return (const void*)fused_rows_kernel<D, 4, 1, false, true>;
    case 8: return (const void*)fused_rows_kernel<D, 8, 1, false, true>;
    case 16: return (const void*)fused_rows_kernel<D, 16, 1, false, true>;
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

// clusters of C CTAs that can be resident at once (cached)
static inline int max_clusters(const void* fn, int threads, int C)
{
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> cache;
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(fn, threads * 16 + C);
    auto it = cache.find(key);
    if (it != cache.end())
        return it->second;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = C;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(threads);
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1)
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
//   CTA_ROW : one row per block; one vector per thread up to
//             one_vec_threads (bf16 / fp16: 896 threads, hidden <= 7168, or
//             1024 threads, hidden <= 8192, with at most 4 ranks; fp32: 512
//             threads, hidden <= 4096), else VPT in {2, 3, 4, 8} with <= 512
//             threads (hidden <= 32768; 3 for 16-bit rows of 1025..1536
//             vectors with at most 4 ranks, 2 for the two-rows-per-SM form).
//             With LaunchCfg::cluster = C > 1, one row per cluster of C CTAs
//             (one vector per thread, the row's sum of squares combined through
//             distributed shared memory) for token counts below the SM count.
// Grid: enough blocks (clusters) for every row, capped at what is resident at
// once (rows are then strided over the resident blocks).
template <class D>
cudaError_t launch_fused_rows_t(int variant, const FusedArgs& a, const LaunchCfg& c)
{
    const int Hv = a.H / 8;
    const int rmax = a.R <= 2 ? 2 : a.R <= 4 ? 4 : a.R <= 8 ? 8 : 16;
    const void* fn;
    int threads, grid;
    int C = variant == AR_VARIANT_WARP_ROW ? 1 : c.cluster;
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
        const int one_vec_max = one_vec_threads<D>(rmax);
        // a row split over a cluster of C CTAs: one vector per thread only
        if (C > 1 && (Hv + C - 1) / C > one_vec_max)
            C = 1;
        int vpt = (Hv + C - 1) / C <= one_vec_max ? 1 : pow2_at_least((Hv + 511) / 512);
        // Light 16-bit rows (513..1023 vectors, at most 4 ranks, at most 2304
        // rank-vectors = 36 KB of partials per row), with at least two rows
        // per SM: two rows per SM at two vectors per thread instead of one
        // row per SM at one vector per thread with the next row loaded ahead.
        // Measured (us, back-to-back / inputs evicted, T=8192, two rows per
        // SM vs one): R=3, H=4104 73.6 / 81.0 vs 87.6 / 99.1; R=2, H=6144
        // 83.7 / 89.1 vs 86.0 / 98.5; R=3, H=6144 95.9 / 104.7 vs 98.2 /
        // 110.6; R=4, H=4608 88.3 / 89.9 vs 88.2 / 90.0.  Heavier rows do
        // better with the look-ahead: R=4, H=6144 110.8 / 116.4 vs 105.8 /
        // 116.1; R=3, H=7168 116.4 / 119.0 vs 107.7 / 119.5; R=3, H=8192
        // 133.8 / 132.3 vs 118.9 / 129.5; R=2, H=8192 106.9 / 115.5 vs
        // 103.0 / 114.9.  Between them R=4, H=5120 (100.1 / 98.9 vs 95.0 /
        // 105.8) and H=5632 (102.3 / 108.8 vs 101.6 / 112.7) split the two
        // timings and take the look-ahead.
        bool light = false;
        // (buffer mode only: this instantiation carries no Lamport code)
        if (D::bytes == 2 && C == 1 && rmax <= 4 && Hv > 512 && Hv < 1024 &&
            a.R * Hv <= 2304 && a.T >= 2 * c.sms && !a.lamport) {
            vpt = 2;
            light = true;
        }
        // 16-bit rows of 449..512 vectors with 5..8 ranks: the one-vector
        // kernel takes 68 registers there, one block of 480..512 threads per
        // SM, and with 8 ranks it has no registers for the next row's
        // loads.  At most 512 threads leave up to 128 registers: with 6..8
        // ranks the next row's rank and residual vectors are loaded ahead as
        // for <= 4 ranks (114 registers); with 5 ranks two blocks of <= 64
        // registers share the SM instead.  Measured (us, back-to-back /
        // inputs evicted; before -> 64 registers -> look-ahead), T=8192,
        // H=4096, residual + norm: R=8 116.9 / 129.1 -> 118.1 / 125.4 ->
        // 109.4 / 116.6 (0.99 of the copy bandwidth); R=7 109.9 / 121.4 ->
        // 107.8 / 115.8 -> 102.2 / 109.1; R=6 106.9 / 119.2 -> 96.0 / 106.3
        // -> 95.7 / 104.4; R=5 103.3 / 115.6 -> 86.5 / 96.8 -> 90.7 / 100.7.
        // R=8 with NVFP4 output 133.3 -> 120.5 -> 114.5, with FP8 output
        // 122.8 -> 124.4 -> 115.4; R=8, T=512 9.3 / 15.4 -> 8.3 / 15.3 ->
        // 8.8 / 13.0.  Narrower rows already hold two or more 68-register
        // blocks per SM, and neither form wins there (look-ahead, R=8:
        // H=1024 114.2 -> 108.4, H=2048 112.2 -> 108.6, but with NVFP4
        // output 107.8 -> 114.4, H=1536 86.5 -> 92.8, H=2560 136.3 -> 180.5;
        // 64 registers: H=3072 86.3 -> 96.0), so they keep the plain kernel.
        bool ahead = false;
        if (D::bytes == 2 && C == 1 && rmax == 8 && Hv > 448 && Hv <= 512) {
            // the look-ahead instantiation carries no Lamport code
            if (a.R >= 6 && a.T > c.sms && !a.lamport)
                ahead = true;
            else if (a.T >= 2 * c.sms)
                light = true;
        }
        // 1025..1536 vectors of a 16-bit row with at most 4 ranks: three
        // vectors per thread (up to 512 threads) instead of four (up to 384);
        // measured R=2, H=10240, T=16384: 256.4 vs 312.3 us; R=4, H=10240,
        // T=2048: 51.6 vs 76.6 us; R=3, H=12288, T=1024: 28.4 vs 43.2 us.
        if (D::bytes == 2 && C == 1 && rmax <= 4 && Hv > 1024 && Hv <= 1536)
            vpt = 3;
        if (vpt > 8)
            return cudaErrorInvalidValue;
        fn = light ? rows_light_fn<D>(rmax)
             : ahead ? rows_ahead_fn<D>()
             : (C > 1 && vpt == 1) ? rows_cluster_fn<D>(rmax) : rows_fn<D, false>(rmax, vpt);
        if (vpt != 1)
            C = 1;
        threads = ((Hv + C * vpt - 1) / (C * vpt) + 31) / 32 * 32;
        if (C == 1) {
            int cap = c.sms * blocks_per_sm(fn, threads);
            grid = a.T < cap ? a.T : cap;
            // Few rows per block (decode-sized buffer calls, small prefills):
            // the buffer-mode instantiation, whose kernel carries no Lamport
            // code.  Measured (µs back-to-back, CUDA graphs with PDL; with
            // the Lamport code -> without): R=4, H=8192 with FP8 output at
            // T=256 / 512 / 1024 6.37 / 11.60 / 19.17 -> 5.84 / 10.45 / 18.87,
            // but T=2048 39.5 -> 40.2; R=4, H=7168, T=384 8.30 -> 7.46; R=4,
            // H=4096, T=512 5.55 -> 5.06; R=8, H=7168 with NVFP4 output at
            // T=512 / 608 15.09 / 16.76 -> 14.65 / 15.98; R=8, T=8192 178.2 ->
            // 179.2.  Hence 2..7 rows per block (with one row per block,
            // R=8, T=128, H=4096, nothing gained: 2.98 µs either way).  Also
            // for two vectors per thread: R=8, H=8192, T=256 7.49 -> 7.12.
            if (vpt <= 2 && !light && !ahead && !a.lamport) {
                const void* fb = rows_buf_fn<D>(rmax, vpt);
                const int capb = c.sms * blocks_per_sm(fb, threads);
                const int gb = a.T < capb ? a.T : capb;
                const int rpb = (a.T + gb - 1) / gb;
                if (fb && rpb >= 2 && rpb <= 7) {
                    fn = fb;
                    grid = gb;
                }
            }
        } else {
            int ncl = max_clusters(fn, threads, C);
            if (ncl < 1)
                ncl = 1;
            grid = (a.T < ncl ? a.T : ncl) * C;
        }
    }
    if (!fn)
        return cudaErrorInvalidValue;
    if (grid < 1)
        grid = 1;
    if (c.used_cluster)
        *c.used_cluster = C;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    int na = 0;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = c.stream;
    if (C > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = C;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (c.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    void* args[] = {const_cast<FusedArgs*>(&a)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace arf
