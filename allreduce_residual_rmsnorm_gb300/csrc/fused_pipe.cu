// Bulk-copy pipelined fused epilogue for large token counts.
//
// Same arithmetic as the register-resident row kernels (TensorRT-LLM
// allReduceFusionKernels.cu: allreduce_sum, add128, rms_norm, fused_op), but
// the bytes move differently:
//
//   * persistent blocks, one per SM, rows strided over the grid;
//   * one producer lane streams the input rows of its rows in slice groups
//     (at most 2 x NC vectors of one source row; the R rank partials of a
//     group, then the residual's) into a ring of S shared-memory stages with
//     1-D bulk async copies (cp.async.bulk, the TMA engine) that signal an
//     mbarrier per stage ("full") with their byte count;
//   * consumer warps wait on "full", fold the stage into fp32 accumulators
//     held in registers (rank order, as the oracle), and release the stage
//     ("empty", one arrival per consumer warp);
//   * so the copy engine keeps up to S transfers in flight per SM
//     while the consumers reduce, normalise, quantise and store the previous
//     row -- memory-level parallelism without registers.
//
// Every wait is bounded by FusedArgs::timeout_ns (mbarrier try_wait + the
// global timer).  A wait that gives up records AR_ERR_TIMEOUT in the
// workspace status word, tells the block to stop, and the producer lane still
// waits (bounded) for its copies in flight before the block exits.
#include "fused_core.cuh"

#include <mutex>
#include <set>
#include <utility>

namespace arf {

namespace {

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

// try_wait with a suspend-time hint: a waiting warp sleeps in the barrier
// unit (up to `hint_ns`) instead of spinning through issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// Wait for completion of the phase with parity `parity`; false after timeout_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    if (mbar_try_wait(bar, parity, 1000u))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity, 1000u)) {
        if (globaltimer_ns() - t0 > timeout_ns)
            return false;
    }
    return true;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

constexpr int kMaxStages = 32;
constexpr uint32_t kSmemLimit = 232448;  // 227 KB opt-in dynamic shared memory per block
constexpr uint32_t kSmemTail = 2048;     // barriers, reduction slots, flags
constexpr uint32_t kRingTarget = 163840; // bytes of stages per block

}  // namespace

// row_rstd of the consumer warps that also publishes, between the same two
// barriers, one snapshot of the abort flag taken by a single thread: every
// consumer warp then takes the same decision to stop after this row.  (A warp
// reading the flag on its own could leave while the others, having read it
// before the producer set it, wait for it at the next row's barrier.)
__device__ __forceinline__ float consumer_row_rstd(DF ss, DF* slots, float* rstd_slot,
                                                   int* stop_slot, volatile int* abort_flag,
                                                   int warp, int lane, int nw, int H, float eps,
                                                   NamedSync sync, bool& stop)
{
    ss = df_warp_sum(ss);
    if (lane == 0)
        slots[warp] = ss;
    sync();
    if (warp == 0) {
        DF v = lane < nw ? slots[lane] : DF{0.0f, 0.0f};
        v = df_warp_sum(v);
        if (lane == 0) {
            *rstd_slot = inv_rms(v, H, eps);
            *stop_slot = *abort_flag;
        }
    }
    sync();
    stop = *reinterpret_cast<volatile int*>(stop_slot) != 0;
    return *rstd_slot;
}

// Ring position: stage index and the parity of its current use.
struct Ring {
    uint32_t s = 0, ph = 0;
    __device__ __forceinline__ void next(uint32_t S)
    {
        if (++s == S) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// Stage = one "slice group" of one source row: KPS consecutive k-slices, where
// k-slice k holds vectors [k * NC, (k + 1) * NC) -- one vector per consumer
// thread.  Stages of a row come in the order (group j, source u): the R rank
// partials of group j, then its residual, then group j + 1.  A consumer
// therefore finishes the rank sum of KPS vectors before the next group
// arrives and keeps only the packed y of the row in registers; and a stage is
// at most KPS * NC vectors (KPS = 2, or 3 for three vectors per thread: at
// most 24 KB of bf16 at NC = 512) whatever the hidden size, so the ring holds
// 6 to 10 copies in flight even for 32768-wide rows.
template <int VPT>
__host__ __device__ constexpr int pipe_kps()
{
    return VPT == 3 ? 3 : (VPT < 2 ? VPT : 2);
}

template <class D, int VPT>
__global__ void __launch_bounds__(544, 1)
fused_pipe_kernel(const FusedArgs a, const int S, const int NC)
{
    using V = typename D::Vec;
    constexpr int EB = D::bytes;
    constexpr int VB = 8 * EB;
    constexpr int KPS = pipe_kps<VPT>();
    constexpr int NG = VPT / KPS;           // slice groups per row
    extern __shared__ __align__(1024) uint8_t smem[];
    const int H = a.H;
    const int Hv = H >> 3;
    const int R = a.R;
    const int pat = a.pattern;
    const uint32_t row_bytes = (uint32_t)H * EB;
    const uint32_t group_bytes = (uint32_t)(KPS * NC * VB);   // stage capacity
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * group_bytes);
    uint64_t* empty = full + kMaxStages;
    DF* red = reinterpret_cast<DF*>(empty + kMaxStages);   // [2][32]
    float* rstd_sh = reinterpret_cast<float*>(red + 64);   // [2]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(rstd_sh + 2);
    int* stop_sh = const_cast<int*>(abort_flag) + 1;       // [2]: per-row snapshots of abort_flag
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int ncw = NC >> 5;
    const uint64_t tmo = a.timeout_ns;
    const uint32_t smem0 = smem_addr(smem);
    const uint32_t full0 = smem_addr(full);
    const uint32_t empty0 = smem_addr(empty);

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, (uint32_t)ncw);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // ------------------------------------------------------------ producer
    if (warp == ncw) {
        if (lane == 0) {
            Ring ring;
            uint32_t issued = 0;
            bool ok = true;
            for (int row = blockIdx.x; ok && row < a.T; row += gridDim.x) {
                const size_t roff = (size_t)row * row_bytes;
                for (int j = 0; ok && j < NG; ++j) {
                    // bytes of group j inside the row (every group holds at least
                    // one vector: checked at launch)
                    const uint32_t goff = (uint32_t)j * group_bytes;
                    const uint32_t gb = row_bytes - goff < group_bytes ? row_bytes - goff : group_bytes;
                    for (int u = 0; u <= R; ++u) {
                        // a stage's previous use must have been released by every consumer warp
                        if (issued >= (uint32_t)S && !mbar_wait(empty0 + 8u * ring.s, ring.ph ^ 1u, tmo)) {
                            record_error(a.state, AR_ERR_TIMEOUT, -2);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        const uint8_t* src = (u < R ? a.partial[u] : a.residual_in) + roff + goff;
                        mbar_arrive_expect_tx(full0 + 8u * ring.s, gb);
                        bulk_g2s(smem0 + ring.s * group_bytes, src, gb, full0 + 8u * ring.s);
                        ++issued;
                        ring.next((uint32_t)S);
                    }
                }
            }
            // tail: every issued copy must have landed before the block may exit
            // (at most one use per stage is outstanding).  This wait is bounded
            // by at least 200 ms whatever the caller's timeout, so that a tiny
            // timeout cannot end the block while copies still write its shared
            // memory.
            const uint64_t tail_tmo = tmo > 200000000ull ? tmo : 200000000ull;
            const uint32_t n_tail = issued < (uint32_t)S ? issued : (uint32_t)S;
            for (uint32_t k = 0; k < n_tail; ++k) {
                // step back k+1 positions from the next free position
                uint32_t s = ring.s, ph = ring.ph;
                for (uint32_t j = 0; j <= k; ++j) {
                    if (s == 0) {
                        s = (uint32_t)S;
                        ph ^= 1u;
                    }
                    --s;
                }
                if (!mbar_wait(full0 + 8u * s, ph, tail_tmo))
                    record_error(a.state, AR_ERR_TIMEOUT, -3);
            }
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    const int g = tid;
    float qscale = 0.0f;
    if (pat & (AR_QUANT_FP8 | AR_QUANT_NVFP4))
        qscale = *a.scale_factor;
    float amax_unused = 0.0f;

    Ring ring;
    int parity = 0;
    for (int row = blockIdx.x; row < a.T; row += gridDim.x) {
        const size_t roff = (size_t)row * row_bytes;
        DF2 ss = {};
        V yv[VPT];
        bool ok = true;
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            float acc[KPS][8];
            V xr[KPS];
            for (int u = 0; ok && u <= R; ++u) {
                // one outcome per warp, so that its lanes stay converged
                if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8u * ring.s, ring.ph, tmo))) {
                    if (lane == 0)
                        record_error(a.state, AR_ERR_TIMEOUT, -1);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                const uint8_t* st = smem + (size_t)ring.s * group_bytes;
                V w[KPS];
#pragma unroll
                for (int kk = 0; kk < KPS; ++kk) {
                    const int v = g + (j * KPS + kk) * NC;
                    w[kk] = v < Hv ? *reinterpret_cast<const V*>(st + (size_t)(g + kk * NC) * VB)
                                   : zero_vec<V>();
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty0 + 8u * ring.s);
                ring.next((uint32_t)S);
#pragma unroll
                for (int kk = 0; kk < KPS; ++kk) {
                    if (u == 0) {
                        if (a.acc)
                            elem_start8<D>(acc[kk], w[kk]);
                        else
                            unpack8<D>(w[kk], acc[kk]);
                    } else if (u < R) {
                        if (a.acc)
                            elem_add8<D>(acc[kk], w[kk]);
                        else
                            add8<D>(acc[kk], w[kk]);
                    } else {
                        xr[kk] = w[kk];
                    }
                }
            }
#pragma unroll
            for (int kk = 0; kk < KPS; ++kk) {
                const int k = j * KPS + kk;
                const int v = g + k * NC;
                if (ok && v < Hv) {
                    if (a.acc)
                        elem_finish8<D>(acc[kk]);
                    yv[k] = residual_vec<D>(acc[kk], xr[kk], ss);
                    if (pat & AR_RESIDUAL_OUT)
                        st_vec(a.residual_out + roff + (size_t)v * VB, yv[k]);
                } else {
                    yv[k] = zero_vec<V>();
                }
            }
        }
        bool stop = false;
        const float rstd = consumer_row_rstd(df2_merge(ss), red + parity * 32, &rstd_sh[parity],
                                             &stop_sh[parity], abort_flag, warp, lane, ncw, H,
                                             a.eps, NamedSync{NC}, stop);
        parity ^= 1;
        if (stop)
            break;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = g + k * NC;
            float gf[8];
            load_gamma<D>(a.gamma, v, v < Hv, gf);   // L1-resident across rows
            normalize_vec<D>(a, pat, row, v, v < Hv, yv[k], gf, rstd, qscale, amax_unused);
        }
    }
}

// ---------------------------------------------------------------- launch

namespace {

template <class D>
const void* pipe_fn(int vpt)
{
    switch (vpt) {
    case 1: return (const void*)fused_pipe_kernel<D, 1>;
    case 2: return (const void*)fused_pipe_kernel<D, 2>;
    case 4: return (const void*)fused_pipe_kernel<D, 4>;
    case 3:
        // 16-bit only: a three-slice fp32 group would be 48 KB (a 3-stage ring)
        if constexpr (D::bytes == 2)
            return (const void*)fused_pipe_kernel<D, 3>;
        else
            return nullptr;
    case 6: return (const void*)fused_pipe_kernel<D, 6>;
    case 8: return (const void*)fused_pipe_kernel<D, 8>;
    default: return nullptr;
    }
}

template <class D>
cudaError_t launch_t(const FusedArgs& a, const LaunchCfg& c)
{
    const int Hv = a.H / 8;
    // at most 512 consumer threads: more consumer warps cost more barrier
    // arrivals per byte than they win in latency hiding (measured at H = 7168).
    // Vectors per thread: ceil(Hv / 512), rounded up to an even count above 3
    // (two-slice groups); 3 (one three-slice group per source row) and 6
    // rather than 4 and 8 keep up to 16 consumer warps (bf16 R = 8,
    // H = 10240: 220.5 vs 258.0 us; H = 12288: 218.1 vs 229.9 us; H = 20480:
    // 242.4 vs 284.2 us; R = 4, H = 20480: 314.0 vs 377.2 us).
    const int q = (Hv + 511) / 512;
    const int vpt = (q <= 3 && (q < 3 || D::bytes == 2)) ? q : (q + 1) / 2 * 2;
    const void* fn = pipe_fn<D>(vpt);
    if (!fn)
        return cudaErrorInvalidValue;
    const int NC = ((Hv + vpt - 1) / vpt + 31) / 32 * 32;
    const int kps = vpt == 3 ? 3 : (vpt < 2 ? vpt : 2);
    // every slice group must hold at least one vector of the row
    if (NC * (vpt - kps) >= Hv)
        return cudaErrorInvalidValue;
    const uint32_t stage_bytes = (uint32_t)(kps * NC * 8 * D::bytes);
    // ring depth: ~160 KB of copies in flight per SM (a sweep at H = 7168 was
    // flat from 10 to 12 stages and lost bandwidth above 16 and below 8)
    int S = (int)(kRingTarget / stage_bytes);
    if (S < 4)
        S = 4;
    const int S_fit = (int)((kSmemLimit - kSmemTail) / stage_bytes);
    if (S > S_fit)
        S = S_fit;
    if (S > kMaxStages)
        S = kMaxStages;
    if (S < 2)
        return cudaErrorInvalidValue;
    const uint32_t smem = (uint32_t)S * stage_bytes + kSmemTail;
    // the shared-memory opt-in is a per-device function attribute: set once
    // per (device, instantiation)
    static std::mutex mu;
    static std::set<std::pair<int, const void*>> attr_set;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return e;
        std::lock_guard<std::mutex> lk(mu);
        if (!attr_set.count({dev, fn})) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemLimit);
            if (e != cudaSuccess)
                return e;
            attr_set.insert({dev, fn});
        }
    }
    int grid = c.sms < a.T ? c.sms : a.T;
    if (grid < 1)
        grid = 1;
    int Sarg = S, NCarg = NC;
    void* args[] = {const_cast<FusedArgs*>(&a), &Sarg, &NCarg};
    return cudaLaunchKernel(fn, dim3(grid), dim3(NC + 32), args, smem, c.stream);
}

}  // namespace

bool fused_pipe_supported(int dtype, int H, int R)
{
    return dtype_supported(dtype) && H % 8 == 0 && H <= AR_MAX_HIDDEN && R >= 1 && R <= AR_MAX_RANKS;
}

cudaError_t launch_fused_pipe(int dtype, const FusedArgs& a, const LaunchCfg& c)
{
    if (a.lamport || a.amax_out || !fused_pipe_supported(dtype, a.H, a.R))
        return cudaErrorNotSupported;
    switch (dtype) {
    case AR_DT_BF16: return launch_t<Bf16>(a, c);
    case AR_DT_FP16: return launch_t<Fp16>(a, c);
    case AR_DT_FP32: return launch_t<F32>(a, c);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace arf
