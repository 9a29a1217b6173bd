// Bulk-copy pipelined fused epilogue for large token counts.
//
// Same arithmetic as the register-resident row kernels (TensorRT-LLM
// allReduceFusionKernels.cu: allreduce_sum, add128, rms_norm, fused_op), but
// the bytes move differently:
//
//   * persistent blocks, one per SM, rows strided over the grid; one thread
//     per 16-byte vector of a row (<= 896 threads), as the row kernel;
//   * every input row a block needs -- the R rank partials, then the
//     residual, for each of its rows in turn -- is one 1-D bulk async copy
//     (cp.async.bulk, the TMA engine) into a ring of S row-sized shared-memory
//     stages (as many as fit: ~1.7 rows of 9 at R = 8, H = 7168), each
//     signalling a per-stage mbarrier with its byte count;
//   * the threads wait on those barriers, fold each stage into fp32 registers
//     (rank order, as the oracle), and need no per-stage release: the block
//     barrier that the row's sum of squares needs anyway proves that every
//     thread has read the row's stages, and right after it thread 0 refills
//     the freed stages with the next rows' copies;
//   * so the copy engine keeps about S rows' worth of bytes in flight per SM
//     while the block reduces, normalises, quantises and stores.
//
// Every wait is bounded by FusedArgs::timeout_ns (mbarrier try_wait with a
// suspend hint + the global timer).  A wait that gives up records
// AR_ERR_TIMEOUT in the workspace status word and the block stops after the
// row's barrier; thread 0 then waits (bounded) for its copies still in flight
// before the block exits.
#include "fused_core.cuh"

#include <mutex>

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

}  // namespace

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

// Producer state, held by thread 0: the next unit to issue and its ring slot.
// Unit u of this block is rank (u % U) of the block's row (u / U); rank R is
// the residual row.
struct Producer {
    uint32_t next = 0;
    uint32_t s = 0;
    int row = 0;
    int rank = 0;
};

template <class D, int VPT>
__global__ void __launch_bounds__(VPT == 1 ? 896 : 512, 1)
fused_pipe_kernel(const FusedArgs a, const int S, const int NT)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int H = a.H;
    const int Hv = H >> 3;
    const int R = a.R;
    const int U = R + 1;                          // stage loads per row
    const int pat = a.pattern;
    const uint32_t stage_bytes = (uint32_t)H * 2;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * stage_bytes);
    DF* red = reinterpret_cast<DF*>(full + kMaxStages);   // [2][32]
    float* rstd_sh = reinterpret_cast<float*>(red + 64);  // [2]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(rstd_sh + 2);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int nw = NT >> 5;
    const uint64_t tmo = a.timeout_ns;
    const uint32_t smem0 = smem_addr(smem);
    const uint32_t full0 = smem_addr(full);

    const int nrows = a.T > (int)blockIdx.x ? (a.T - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const uint32_t total = (uint32_t)nrows * (uint32_t)U;

    Producer pr;
    pr.row = blockIdx.x;
    // issue units while fewer than S are outstanding (thread 0 only)
    auto issue_upto = [&](uint32_t consumed) {
        while (pr.next < total && pr.next - consumed < (uint32_t)S) {
            const uint8_t* src = pr.rank < R ? a.partial[pr.rank] : a.residual_in;
            src += (size_t)pr.row * stage_bytes;
            mbar_arrive_expect_tx(full0 + 8u * pr.s, stage_bytes);
            bulk_g2s(smem0 + pr.s * stage_bytes, src, stage_bytes, full0 + 8u * pr.s);
            ++pr.next;
            if (++pr.s == (uint32_t)S)
                pr.s = 0;
            if (++pr.rank == U) {
                pr.rank = 0;
                pr.row += gridDim.x;
            }
        }
    };

    if (tid == 0) {
        for (int s = 0; s < S; ++s)
            mbar_init(full0 + 8u * s, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        issue_upto(0);
    }
    __syncthreads();

    const int g = tid;
    float qscale = 0.0f;
    if (pat & (AR_QUANT_FP8 | AR_QUANT_NVFP4))
        qscale = *a.scale_factor;
    float amax_unused = 0.0f;

    Ring ring;
    uint32_t consumed = 0;
    int parity = 0;
    for (int k = 0; k < nrows; ++k) {
        const int row = blockIdx.x + k * gridDim.x;
        const size_t roff = (size_t)row * stage_bytes;
        float acc[VPT][8];
        uint4 xr[VPT];
        bool ok = true;
        for (int u = 0; u < U; ++u) {
            if (!mbar_wait(full0 + 8u * ring.s, ring.ph, tmo)) {
                record_error(a.state, AR_ERR_TIMEOUT, -1);
                *abort_flag = 1;
                ok = false;
                break;
            }
            const uint8_t* st = smem + (size_t)ring.s * stage_bytes;
            ring.next((uint32_t)S);
#pragma unroll
            for (int kk = 0; kk < VPT; ++kk) {
                const int v = g + kk * NT;
                if (v < Hv) {
                    const uint4 w = *reinterpret_cast<const uint4*>(st + (size_t)v * 16);
                    if (u == 0)
                        unpack8<D>(w, acc[kk]);
                    else if (u < R)
                        add8<D>(acc[kk], w);
                    else
                        xr[kk] = w;
                }
            }
        }

        DF ss = {0.0f, 0.0f};
        uint4 yv[VPT];
#pragma unroll
        for (int kk = 0; kk < VPT; ++kk) {
            const int v = g + kk * NT;
            if (ok && v < Hv) {
                yv[kk] = residual_vec<D>(acc[kk], xr[kk], ss);
                if (pat & AR_RESIDUAL_OUT)
                    st_vec(a.residual_out + roff + (size_t)v * 16, yv[kk]);
            } else {
                yv[kk] = make_uint4(0, 0, 0, 0);
            }
        }

        // sum of squares; the first barrier also frees this row's stages, so
        // thread 0 refills them before the normalisation
        ss = df_warp_sum(ss);
        if (lane == 0)
            red[parity * 32 + warp] = ss;
        __syncthreads();
        if (*abort_flag)
            break;
        consumed += (uint32_t)U;
        if (tid == 0)
            issue_upto(consumed);
        if (warp == 0) {
            DF t = lane < nw ? red[parity * 32 + lane] : DF{0.0f, 0.0f};
            t = df_warp_sum(t);
            if (lane == 0)
                rstd_sh[parity] = inv_rms(t, H, a.eps);
        }
        __syncthreads();
        const float rstd = rstd_sh[parity];
        parity ^= 1;

#pragma unroll
        for (int kk = 0; kk < VPT; ++kk) {
            const int v = g + kk * NT;
            float gf[8];
            load_gamma<D>(a.gamma, v, v < Hv, gf);
            normalize_vec<D>(a, pat, row, v, v < Hv, yv[kk], gf, rstd, qscale, amax_unused);
        }
    }

    // after an abort, copies may still be in flight into this block's shared
    // memory: thread 0 waits (bounded) for every issued, unconsumed unit
    if (tid == 0 && *abort_flag) {
        Ring r2 = ring;
        for (uint32_t c = consumed; c < pr.next; ++c) {
            (void)mbar_wait(full0 + 8u * r2.s, r2.ph, tmo);
            r2.next((uint32_t)S);
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
    case 8: return (const void*)fused_pipe_kernel<D, 8>;
    default: return nullptr;
    }
}

int pow2_at_least(int x)
{
    int p = 1;
    while (p < x)
        p <<= 1;
    return p;
}

template <class D>
cudaError_t launch_t(const FusedArgs& a, const LaunchCfg& c)
{
    const int Hv = a.H / 8;
    // one 16-byte vector per thread up to 896 threads, else <= 512 threads
    const int vpt = Hv <= 896 ? 1 : pow2_at_least((Hv + 511) / 512);
    const void* fn = pipe_fn<D>(vpt);
    if (!fn)
        return cudaErrorInvalidValue;
    const int NT = ((Hv + vpt - 1) / vpt + 31) / 32 * 32;
    const uint32_t stage_bytes = (uint32_t)a.H * 2;
    // as many stages as fit: the ring holds ~1.7 rows at R = 8, H = 7168
    int S = (int)((kSmemLimit - kSmemTail) / stage_bytes);
    if (S > kMaxStages)
        S = kMaxStages;
    if (S < 2)
        return cudaErrorInvalidValue;
    const uint32_t smem = (uint32_t)S * stage_bytes + kSmemTail;
    static std::mutex mu;
    static bool attr_set[2][9] = {};
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!attr_set[D::id][vpt]) {
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kSmemLimit);
            if (e != cudaSuccess)
                return e;
            attr_set[D::id][vpt] = true;
        }
    }
    int grid = c.sms < a.T ? c.sms : a.T;
    if (grid < 1)
        grid = 1;
    int Sarg = S, NTarg = NT;
    void* args[] = {const_cast<FusedArgs*>(&a), &Sarg, &NTarg};
    return cudaLaunchKernel(fn, dim3(grid), dim3(NT), args, smem, c.stream);
}

}  // namespace

// The ring must hold one whole row (R partial rows + the residual row): its
// stages are released only by the row's block barrier.
bool fused_pipe_supported(int dtype, int H, int R)
{
    (void)dtype;
    if (H % 8 != 0 || H > AR_MAX_HIDDEN || R < 1 || R > AR_MAX_RANKS)
        return false;
    uint64_t S = (kSmemLimit - kSmemTail) / ((uint64_t)H * 2);
    if (S > kMaxStages)
        S = kMaxStages;
    return S >= (uint64_t)R + 1;
}

cudaError_t launch_fused_pipe(int dtype, const FusedArgs& a, const LaunchCfg& c)
{
    if (a.lamport || a.amax_out || !fused_pipe_supported(dtype, a.H, a.R))
        return cudaErrorNotSupported;
    return dtype == AR_DT_BF16 ? launch_t<Bf16>(a, c) : launch_t<Fp16>(a, c);
}

}  // namespace arf
