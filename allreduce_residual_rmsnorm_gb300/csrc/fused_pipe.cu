// Bulk-copy pipelined fused epilogue for large token counts.
//
// Same arithmetic as the register-resident row kernels (TensorRT-LLM
// allReduceFusionKernels.cu: allreduce_sum, add128, rms_norm, fused_op), but
// the bytes move differently:
//
//   * persistent blocks, one per SM, rows strided over the grid;
//   * one producer lane streams every input row of its rows -- the R rank
//     partials, then the residual -- into a ring of S shared-memory stages
//     with 1-D bulk async copies (cp.async.bulk, the TMA engine) that signal
//     an mbarrier per stage ("full") with their byte count;
//   * consumer warps wait on "full", fold the stage into fp32 accumulators
//     held in registers (rank order, as the oracle), and release the stage
//     ("empty", one arrival per consumer warp);
//   * so the copy engine keeps up to S row-sized transfers in flight per SM
//     while the consumers reduce, normalise, quantise and store the previous
//     row -- memory-level parallelism without registers.
//
// Every wait is bounded by FusedArgs::timeout_ns (mbarrier try_wait + the
// global timer).  A wait that gives up records AR_ERR_TIMEOUT in the
// workspace status word, tells the block to stop, and the producer lane still
// waits (bounded) for its copies in flight before the block exits.
#include "ar_common.cuh"
#include "ar_internal.h"

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

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for completion of the phase with parity `parity`; false after timeout_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
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

__device__ __forceinline__ void consumer_sync(int nthreads)
{
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

constexpr int kMaxStages = 32;
constexpr uint32_t kSmemLimit = 232448;  // 227 KB opt-in dynamic shared memory per block
constexpr uint32_t kSmemTail = 2048;     // barriers, reduction slots, flags

}  // namespace

template <class D, int VPT>
__global__ void __launch_bounds__(544, 1)
fused_pipe_kernel(const FusedArgs a, const int S, const int NC)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int H = a.H;
    const int Hv = H >> 3;
    const int R = a.R;
    const int pat = a.pattern;
    const uint32_t stage_bytes = (uint32_t)H * 2;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * stage_bytes);
    uint64_t* empty = full + kMaxStages;
    DF* red = reinterpret_cast<DF*>(empty + kMaxStages);   // [2][32]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 64);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int ncw = NC >> 5;
    const uint64_t tmo = a.timeout_ns;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), (uint32_t)ncw);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // ------------------------------------------------------------ producer
    if (warp == ncw) {
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int row = blockIdx.x; ok && row < a.T; row += gridDim.x) {
                const size_t roff = (size_t)row * stage_bytes;
                for (int u = 0; u <= R; ++u, ++it) {
                    const uint32_t s = it % (uint32_t)S;
                    const uint32_t n = it / (uint32_t)S;
                    if (n > 0 && !mbar_wait(smem_addr(&empty[s]), (n - 1) & 1u, tmo)) {
                        record_error(a.state, AR_ERR_TIMEOUT, -2);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    const uint8_t* src = u < R ? a.partial[u] + roff : a.residual_in + roff;
                    mbar_arrive_expect_tx(smem_addr(&full[s]), stage_bytes);
                    bulk_g2s(smem_addr(smem + (size_t)s * stage_bytes), src, stage_bytes,
                             smem_addr(&full[s]));
                }
            }
            // tail: every issued copy must have landed before the block may exit
            const uint32_t issued = it;
            for (uint32_t k = issued > (uint32_t)S ? issued - S : 0; k < issued; ++k) {
                const uint32_t s = k % (uint32_t)S;
                if (!mbar_wait(smem_addr(&full[s]), (k / (uint32_t)S) & 1u, tmo))
                    record_error(a.state, AR_ERR_TIMEOUT, -3);
            }
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    const int g = tid;
    uint4 gv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = g + k * NC;
        gv[k] = v < Hv ? ld_keep(a.gamma + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
    }
    float qscale = 0.0f;
    if (pat & (AR_QUANT_FP8 | AR_QUANT_NVFP4))
        qscale = *a.scale_factor;

    uint32_t it = 0;
    int parity = 0;
    for (int row = blockIdx.x; row < a.T; row += gridDim.x) {
        const size_t roff = (size_t)row * stage_bytes;
        float acc[VPT][8];
        uint4 xr[VPT];
        bool ok = true;
        for (int u = 0; u <= R; ++u, ++it) {
            const uint32_t s = it % (uint32_t)S;
            if (!mbar_wait(smem_addr(&full[s]), (it / (uint32_t)S) & 1u, tmo)) {
                record_error(a.state, AR_ERR_TIMEOUT, -1);
                *abort_flag = 1;
                ok = false;
                break;
            }
            const uint8_t* st = smem + (size_t)s * stage_bytes;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = g + k * NC;
                if (v < Hv) {
                    const uint4 w = *reinterpret_cast<const uint4*>(st + (size_t)v * 16);
                    if (u == R) {
                        xr[k] = w;
                    } else if (u == 0) {
                        unpack8<D>(w, acc[k]);
                    } else {
                        float t[8];
                        unpack8<D>(w, t);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            acc[k][i] = __fadd_rn(acc[k][i], t[i]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&empty[s]));
        }

        DF ss = {0.0f, 0.0f};
        uint4 yv[VPT];
        if (ok) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = g + k * NC;
                if (v < Hv) {
                    float af[8], xf[8];
                    unpack8<D>(pack8<D>(acc[k]), af);
                    unpack8<D>(xr[k], xf);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        af[i] = __fadd_rn(af[i], xf[i]);
                    const uint4 y = pack8<D>(af);
                    yv[k] = y;
                    if (pat & AR_RESIDUAL_OUT)
                        st_vec(a.residual_out + roff + (size_t)v * 16, y);
                    float yf[8];
                    unpack8<D>(y, yf);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        df_add_term(ss, __fmul_rn(yf[i], yf[i]));
                } else {
                    yv[k] = make_uint4(0, 0, 0, 0);
                }
            }
        }
        ss = df_warp_sum(ss);
        if (lane == 0)
            red[parity * 32 + warp] = ss;
        consumer_sync(NC);
        if (*abort_flag)
            break;
        DF tot = red[parity * 32];
        for (int w = 1; w < ncw; ++w)
            tot = df_add(tot, red[parity * 32 + w]);
        parity ^= 1;
        const float ss32 = df_round(tot);
        const float ms = __fdiv_rn(ss32, (float)H);
        const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.eps)));

#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = g + k * NC;
            const bool okv = v < Hv;
            float yf[8], gf[8], nf[8];
            unpack8<D>(yv[k], yf);
            unpack8<D>(gv[k], gf);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                nf[i] = __fmul_rn(__fmul_rn(yf[i], rstd), gf[i]);
            const uint4 nv = pack8<D>(nf);
            if (okv && (pat & AR_NORM_OUT))
                st_vec(a.norm_out + roff + (size_t)v * 16, nv);
            if (pat & (AR_QUANT_FP8 | AR_QUANT_NVFP4)) {
                float nq[8];
                unpack8<D>(nv, nq);
                if (pat & AR_QUANT_FP8) {
                    float t[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        t[i] = __fmul_rn(nq[i], qscale);
                    const uint2 c = e4m3x8(t);
                    if (okv)
                        st_u2(a.quant_out + (size_t)row * H + (size_t)v * 8, c.x, c.y);
                } else {
                    float bm = 0.0f;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        bm = fmaxf(bm, fabsf(nq[i]));
                    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
                    const uint32_t sf = e4m3_byte(__fmul_rn(qscale, __fdiv_rn(bm, 6.0f)));
                    const float dec = e4m3_to_f32(sf);
                    const float enc = dec == 0.0f ? 0.0f : __fdiv_rn(qscale, dec);
                    float t[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        t[i] = __fmul_rn(nq[i], enc);
                    const uint32_t codes = e2m1x8(t);
                    if (okv) {
                        *reinterpret_cast<uint32_t*>(a.quant_out + (size_t)row * (H / 2) +
                                                     (size_t)v * 4) = codes;
                        if ((v & 1) == 0)
                            a.scale_out[(size_t)row * (H / 16) + (v >> 1)] = (uint8_t)sf;
                    }
                }
            }
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
    const int vpt = pow2_at_least((Hv + 511) / 512);
    const void* fn = pipe_fn<D>(vpt);
    if (!fn)
        return cudaErrorInvalidValue;
    const int NC = ((Hv + vpt - 1) / vpt + 31) / 32 * 32;
    const uint32_t stage_bytes = (uint32_t)a.H * 2;
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
    int Sarg = S, NCarg = NC;
    void* args[] = {const_cast<FusedArgs*>(&a), &Sarg, &NCarg};
    return cudaLaunchKernel(fn, dim3(grid), dim3(NC + 32), args, smem, c.stream);
}

}  // namespace

bool fused_pipe_supported(int dtype, int H, int R)
{
    (void)dtype;
    return H % 8 == 0 && H <= AR_MAX_HIDDEN && R >= 1 && R <= AR_MAX_RANKS;
}

cudaError_t launch_fused_pipe(int dtype, const FusedArgs& a, const LaunchCfg& c)
{
    if (a.lamport || a.amax_out)
        return cudaErrorNotSupported;
    return dtype == AR_DT_BF16 ? launch_t<Bf16>(a, c) : launch_t<Fp16>(a, c);
}

}  // namespace arf
