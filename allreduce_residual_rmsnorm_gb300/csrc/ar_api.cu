// C ABI of libarfusion: workspace life cycle, staging, argument checks and
// kernel dispatch.  Declarations and the contract of every entry point are in
// include/ar_fusion.h.
//
// Workspace layout (TensorRT-LLM allReduceFusionKernels.cu, Workspace; the
// FlashInfer workspace note), one device allocation, each region 256-byte
// aligned:
//   [buffer  R * maxT * H * elem]  rank r at r * maxT * H elements
//   [flags   R * AR_BARRIER_FLAG_COUNT * 4]  reserved (zero)
//   [lamport 3 slots of R * max(oneshot, maxT) * H * elem], -0.0f words when idle;
//            within the slot, rank r at r * tokens * H elements of the call
//   [state   struct ar_fusion_state]
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <new>
#include <string>

#include "ar_common.cuh"
#include "ar_internal.h"

namespace arf {
cudaError_t launch_fused_rows_bf16(int variant, const FusedArgs& a, const LaunchCfg& c);
cudaError_t launch_fused_rows_fp16(int variant, const FusedArgs& a, const LaunchCfg& c);
cudaError_t launch_fused_rows_fp32(int variant, const FusedArgs& a, const LaunchCfg& c);

cudaError_t launch_fused_rows(int dtype, int variant, const FusedArgs& a, const LaunchCfg& c)
{
    switch (dtype) {
    case AR_DT_BF16: return launch_fused_rows_bf16(variant, a, c);
    case AR_DT_FP16: return launch_fused_rows_fp16(variant, a, c);
    case AR_DT_FP32: return launch_fused_rows_fp32(variant, a, c);
    default: return cudaErrorInvalidValue;
    }
}
}  // namespace arf

using namespace arf;

struct ar_fusion_ws {
    int R, maxT, H, dtype;
    int device, sms;
    bool owned;
    uint8_t* base;
    uint64_t total, buffer_off, buffer_bytes, flag_off, flag_bytes, lamport_off, slot_bytes,
        state_off;
    int variant, mode, last_variant, last_cluster;
    uint64_t timeout_ns;
    int cluster, pdl;           // launch options of the fused call (0 cluster = auto)
    int acc;                    // AR_ACC_FP32 or AR_ACC_ELEMENT
    int sf_layout;              // AR_SF_LINEAR or AR_SF_SWIZZLED
};

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what)
{
    return fail(AR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }
inline bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

struct Layout {
    uint64_t buffer_off, buffer_bytes, flag_off, flag_bytes, lamport_off, slot_bytes, state_off,
        total;
};

Layout layout_of(int R, int maxT, int H, int dtype)
{
    Layout L;
    const uint64_t elem = (uint64_t)elem_bytes(dtype);
    const uint64_t tok = (uint64_t)(maxT > AR_ONESHOT_MAX_TOKENS ? maxT : AR_ONESHOT_MAX_TOKENS);
    L.buffer_off = 0;
    L.buffer_bytes = (uint64_t)R * maxT * H * elem;
    L.flag_off = align256(L.buffer_off + L.buffer_bytes);
    L.flag_bytes = (uint64_t)R * AR_BARRIER_FLAG_COUNT * 4;
    L.lamport_off = align256(L.flag_off + L.flag_bytes);
    L.slot_bytes = (uint64_t)R * tok * H * elem;
    L.state_off = align256(L.lamport_off + 3 * L.slot_bytes);
    L.total = align256(L.state_off + sizeof(ar_fusion_state));
    return L;
}

int check_shape(int tp_size, int max_token_num, int hidden_dim, int dtype)
{
    if (!dtype_supported(dtype))
        return fail(AR_ERR_UNSUPPORTED, "dtype %d is not bf16 (0), fp16 (1) or fp32 (2)", dtype);
    if (tp_size < 1 || tp_size > AR_MAX_RANKS)
        return fail(AR_ERR_UNSUPPORTED, "tp_size %d outside 1..%d", tp_size, AR_MAX_RANKS);
    if (max_token_num < 1)
        return fail(AR_ERR_INVALID, "max_token_num %d < 1", max_token_num);
    if (hidden_dim <= 0 || hidden_dim % 8 != 0)
        return fail(AR_ERR_INVALID, "hidden_dim %d is not a positive multiple of 8", hidden_dim);
    if (hidden_dim > AR_MAX_HIDDEN)
        return fail(AR_ERR_UNSUPPORTED, "hidden_dim %d > %d", hidden_dim, AR_MAX_HIDDEN);
    return AR_OK;
}

// -------------------------------------------------------- small kernels

__global__ void fill_u32_kernel(uint32_t* p, uint64_t n, uint32_t v)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        p[i] = v;
}

__global__ void init_state_kernel(ar_fusion_state* st, uint64_t comm_size)
{
    st->counter = 0;
    st->flag = 0;
    st->lamport_flag = 0;
    st->clear_elem_bytes = 0;
    st->comm_size = comm_size;
    st->clear_size = 0;
    st->status = 0;
    st->detail = -1;
    st->calls = 0;
}

// Copy one rank's [T][H] partial into the workspace.  Lamport: into slot
// (lamport_flag % 3) at rank * T * H elements, with every -0.0f word written as
// +0.0f (the push loop of the one-shot kernel).  Buffer: plain copy.
__global__ void stage_kernel(const uint4* src, uint8_t* region, uint64_t slot_bytes,
                             uint64_t rank_off_bytes, uint64_t nvec, int lamport,
                             const ar_fusion_state* st)
{
    // a fused call launched with programmatic dependent launch may be
    // scheduled now; it still waits for this copy to complete before reading
    pdl_trigger();
    uint8_t* dst = region + rank_off_bytes;
    if (lamport) {
        // one polling load per block (polling loads bypass L1: one per
        // thread would queue thousands of requests on one L2 line)
        __shared__ uint32_t flag_sh;
        if (threadIdx.x == 0)
            flag_sh = *reinterpret_cast<const volatile uint32_t*>(&st->lamport_flag);
        __syncthreads();
        dst += (uint64_t)(flag_sh % 3u) * slot_bytes;
    }
    uint4* d = reinterpret_cast<uint4*>(dst);
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        uint4 v = ld_stream(src + i);
        if (lamport) {
            v.x = v.x == 0x80000000u ? 0u : v.x;
            v.y = v.y == 0x80000000u ? 0u : v.y;
            v.z = v.z == 0x80000000u ? 0u : v.z;
            v.w = v.w == 0x80000000u ? 0u : v.w;
        }
        d[i] = v;
    }
}

unsigned grid_for(uint64_t items, int threads, int sms)
{
    uint64_t b = (items + threads - 1) / threads;
    const uint64_t cap = (uint64_t)sms * 16;
    if (b > cap)
        b = cap;
    return b < 1 ? 1u : (unsigned)b;
}

int init_regions(ar_fusion_ws* ws, cudaStream_t s)
{
    cudaError_t e = cudaMemsetAsync(ws->base + ws->buffer_off, 0, ws->lamport_off, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(buffer, flags)");
    const uint64_t words = 3 * ws->slot_bytes / 4;
    fill_u32_kernel<<<grid_for(words, 256, ws->sms), 256, 0, s>>>(
        reinterpret_cast<uint32_t*>(ws->base + ws->lamport_off), words, 0x80000000u);
    init_state_kernel<<<1, 1, 0, s>>>(reinterpret_cast<ar_fusion_state*>(ws->base + ws->state_off),
                                      ws->slot_bytes);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "workspace init kernels");
    return AR_OK;
}

ar_fusion_state* state_of(ar_fusion_ws* ws)
{
    return reinterpret_cast<ar_fusion_state*>(ws->base + ws->state_off);
}

int resolve_mode(const ar_fusion_ws* ws, int mode, int tokens)
{
    if (mode == AR_MODE_AUTO)
        mode = ws->mode;
    if (mode == AR_MODE_AUTO)
        mode = tokens <= AR_ONESHOT_MAX_TOKENS ? AR_MODE_LAMPORT : AR_MODE_BUFFER;
    return mode;
}

bool valid_pattern(int p)
{
    const int q = p & (AR_QUANT_FP8 | AR_QUANT_NVFP4);
    if (p & ~(AR_RESIDUAL_OUT | AR_NORM_OUT | AR_QUANT_FP8 | AR_QUANT_NVFP4))
        return false;
    if (q == (AR_QUANT_FP8 | AR_QUANT_NVFP4))
        return false;
    const int base = p & (AR_RESIDUAL_OUT | AR_NORM_OUT);
    if (q)
        return base == AR_RESIDUAL_OUT || base == (AR_RESIDUAL_OUT | AR_NORM_OUT);
    return base == AR_NORM_OUT || base == (AR_RESIDUAL_OUT | AR_NORM_OUT);
}

// Common checks of ar_fusion_run / ar_fusion_norm_amax.  Fills `a` (pointers,
// mode) on success.  `calib` = calibration pass (no outputs, no Lamport).
int prepare(ar_fusion_ws* ws, const void* const* partials, int nranks, int tokens, int hidden,
            int dtype, const void* residual_in, const void* gamma, float eps, int pattern,
            void* residual_out, void* norm_out, void* quant_out, void* scale_out,
            const float* scale_factor, bool calib, FusedArgs& a, bool& launch)
{
    launch = false;
    if (!ws)
        return fail(AR_ERR_INVALID, "workspace is NULL");
    if (!dtype_supported(dtype))
        return fail(AR_ERR_UNSUPPORTED, "dtype %d is not bf16 (0), fp16 (1) or fp32 (2)", dtype);
    if (dtype != ws->dtype)
        return fail(AR_ERR_INVALID, "dtype %d differs from the workspace's %d", dtype, ws->dtype);
    if (nranks < 1 || nranks > AR_MAX_RANKS)
        return fail(AR_ERR_UNSUPPORTED, "nranks %d outside 1..%d", nranks, AR_MAX_RANKS);
    if (tokens < 0)
        return fail(AR_ERR_INVALID, "tokens %d < 0", tokens);
    if (hidden <= 0 || hidden % 8 != 0)
        return fail(AR_ERR_INVALID, "hidden_dim %d is not a positive multiple of 8", hidden);
    if (hidden > AR_MAX_HIDDEN)
        return fail(AR_ERR_UNSUPPORTED, "hidden_dim %d > %d", hidden, AR_MAX_HIDDEN);
    if (!calib) {
        if (!valid_pattern(pattern))
            return fail(AR_ERR_INVALID, "unsupported pattern 0x%x", pattern);
        if ((pattern & AR_QUANT_NVFP4) && hidden % 16 != 0)
            return fail(AR_ERR_INVALID, "NVFP4 needs hidden_dim %% 16 == 0 (got %d)", hidden);
    }
    const bool staged = partials == nullptr;
    int mode = AR_MODE_BUFFER;
    if (staged) {
        if (nranks != ws->R)
            return fail(AR_ERR_INVALID, "staged partials: nranks %d != tp_size %d", nranks, ws->R);
        if (hidden != ws->H)
            return fail(AR_ERR_INVALID, "staged partials: hidden %d != workspace hidden %d",
                        hidden, ws->H);
        if (tokens > ws->maxT)
            return fail(AR_ERR_CAPACITY, "tokens %d > max_token_num %d", tokens, ws->maxT);
        mode = calib ? AR_MODE_BUFFER : resolve_mode(ws, AR_MODE_AUTO, tokens);
        if (mode != AR_MODE_LAMPORT && mode != AR_MODE_BUFFER)
            return fail(AR_ERR_INVALID, "bad staged mode %d", mode);
    }
    if (tokens == 0)
        return AR_OK;

    // pointers: element arrays aligned for the vector accesses (16 bytes,
    // 32 for fp32), byte outputs to 16 bytes
    const auto va = [dtype](const void* p) { return vec_aligned(p, dtype); };
    if (!residual_in || !gamma)
        return fail(AR_ERR_INVALID, "residual_in and gamma must be non-NULL");
    if (!va(residual_in) || !va(gamma))
        return fail(AR_ERR_INVALID, "residual_in / gamma not vector aligned");
    if (!calib) {
        if ((pattern & AR_RESIDUAL_OUT) && (!residual_out || !va(residual_out)))
            return fail(AR_ERR_INVALID, "residual_out NULL or not vector aligned");
        if ((pattern & AR_NORM_OUT) && (!norm_out || !va(norm_out)))
            return fail(AR_ERR_INVALID, "norm_out NULL or not vector aligned");
        if (pattern & (AR_QUANT_FP8 | AR_QUANT_NVFP4)) {
            if (!quant_out || !aligned16(quant_out))
                return fail(AR_ERR_INVALID, "quant_out NULL or not 16-byte aligned");
            if (!scale_factor || ((uintptr_t)scale_factor & 3))
                return fail(AR_ERR_INVALID, "scale_factor NULL or misaligned");
        }
        if ((pattern & AR_QUANT_NVFP4) && (!scale_out || !aligned16(scale_out)))
            return fail(AR_ERR_INVALID, "scale_out NULL or not 16-byte aligned");
    }

    memset(&a, 0, sizeof a);
    if (!staged) {
        for (int r = 0; r < nranks; ++r) {
            if (!partials[r] || !va(partials[r]))
                return fail(AR_ERR_INVALID, "partials[%d] NULL or not vector aligned", r);
            a.partial[r] = static_cast<const uint8_t*>(partials[r]);
        }
    } else if (mode == AR_MODE_BUFFER) {
        for (int r = 0; r < nranks; ++r)
            a.partial[r] = ws->base + ws->buffer_off +
                           (uint64_t)r * ws->maxT * ws->H * elem_bytes(ws->dtype);
    } else {
        a.lamport = 1;
        a.lamport_base = ws->base + ws->lamport_off;
        a.slot_bytes = ws->slot_bytes;
    }
    a.R = nranks;
    a.T = tokens;
    a.H = hidden;
    a.pattern = calib ? 0 : pattern;
    a.residual_in = static_cast<const uint8_t*>(residual_in);
    a.gamma = static_cast<const uint8_t*>(gamma);
    a.eps = eps;
    if (!calib) {
        a.residual_out = (pattern & AR_RESIDUAL_OUT) ? static_cast<uint8_t*>(residual_out) : nullptr;
        a.norm_out = (pattern & AR_NORM_OUT) ? static_cast<uint8_t*>(norm_out) : nullptr;
        a.quant_out = (pattern & (AR_QUANT_FP8 | AR_QUANT_NVFP4)) ? static_cast<uint8_t*>(quant_out)
                                                                  : nullptr;
        a.scale_out = (pattern & AR_QUANT_NVFP4) ? static_cast<uint8_t*>(scale_out) : nullptr;
        a.scale_factor = (pattern & (AR_QUANT_FP8 | AR_QUANT_NVFP4)) ? scale_factor : nullptr;
    }
    a.state = state_of(ws);
    a.timeout_ns = ws->timeout_ns;
    a.acc = ws->acc;
    a.sf_layout = ws->sf_layout;
    launch = true;
    return AR_OK;
}

int pick_variant(const ar_fusion_ws* ws, const FusedArgs& a)
{
    int v = ws->variant;
    if (v == AR_VARIANT_BULK_PIPE && (a.lamport || !fused_pipe_supported(ws->dtype, a.H, a.R)))
        v = AR_VARIANT_AUTO;
    if (v == AR_VARIANT_WARP_ROW && a.H > 1024)
        v = AR_VARIANT_AUTO;
    if (v != AR_VARIANT_AUTO)
        return v;
    // One row per warp only up to hidden 512 (at hidden 1024 the block
    // version is faster: 131.5 vs 156.5 us at 32768 tokens).
    if (a.H <= 512)
        return AR_VARIANT_WARP_ROW;
    // Rows that fit one vector per thread of a row block, with at most 8
    // ranks, stay on the register-resident kernel (R = 8, T = 8192, H = 7168:
    // 180-186 us vs 193-214 us for the pipe).  Wider rows (several vectors per
    // thread), and more than 8 ranks of rows over 8 KB, move to the bulk-copy
    // pipe once the inputs exceed ~L2 (96 MiB): bf16 R = 8, H = 16384,
    // T = 4096: 223.8 vs 297.2 us; H = 32768: 260.9 vs 344.9 us; bf16 R = 16,
    // H = 8192: 192.2 vs 240.0 us; R = 12, H = 7168: 135.1 vs 146.6 us; fp32
    // R = 16, H = 4096: 192.5 vs 252.1 us.  Rows of 8 KB or less make stages
    // too small for the pipe (bf16 R = 16, H = 4096: 121.4 vs 103.3 us;
    // H = 1024: 392 vs 102 us), and below ~L2 the row kernel's L2 hits win
    // (fp32 R = 8, H = 7168, T = 304: 11.2 vs 15.2 us).
    const int Hv = a.H / 8;
    const uint64_t eb = (uint64_t)elem_bytes(ws->dtype);
    const uint64_t in_bytes = (uint64_t)(a.R + 1) * a.T * a.H * eb;
    // The row kernel also keeps 16-bit rows of up to 1536 vectors with at most
    // 4 ranks (three vectors per thread: R = 4, H = 10240, T = 13104: 276.4 vs
    // 353.9 us; R = 3, H = 12288: 352.5 vs 409.7 us) and, with two ranks, up
    // to 2048 vectors (R = 2, H = 16384: 394.5 vs 394.6 us; H = 20480:
    // 1071.7 vs 468.1 us).  fp32 rows beyond one vector per thread take the
    // pipe at any rank count (R = 2, H = 12288: 453.5 vs 530.6 us).
    const bool row_holds = eb == 2 && ((a.R <= 4 && Hv <= 1536) || (a.R <= 2 && Hv <= 2048));
    const bool wide = Hv > one_vec_threads_for((int)eb, a.R) && !row_holds;
    const bool many_ranks = a.R > 8 && (uint64_t)a.H * eb > 8192;
    if (!a.lamport && !a.amax_out && in_bytes >= (96ull << 20) && (wide || many_ranks) &&
        fused_pipe_supported(ws->dtype, a.H, a.R))
        return AR_VARIANT_BULK_PIPE;
    return AR_VARIANT_CTA_ROW;
}

// CTAs per row when the caller left the choice to the library (cluster 0):
// one.  A cluster split measured slower wherever the row kernel is used by
// default: decode sizes (R = 8, T = 128, H = 4096: 7.65 vs 7.09 us), bf16
// prefill (R = 8, T = 8192, H = 7168: 231.8 vs 180.1 us), and the wide rows
// that it helps (fp32 R = 8, H = 7168: 391.0 vs 494.4 us at 8192 tokens) run
// on the bulk-copy pipe instead (229 us).
int auto_cluster(const ar_fusion_ws* ws)
{
    return ws->cluster > 0 ? ws->cluster : 1;
}

int launch_fused(ar_fusion_ws* ws, const FusedArgs& a, cudaStream_t s)
{
    LaunchCfg c{ws->sms, s};
    c.pdl = ws->pdl;
    const int variant = pick_variant(ws, a);
    c.cluster = auto_cluster(ws);
    ws->last_variant = variant;
    ws->last_cluster = 1;
    c.used_cluster = &ws->last_cluster;
    cudaError_t e = variant == AR_VARIANT_BULK_PIPE ? launch_fused_pipe(ws->dtype, a, c)
                                                    : launch_fused_rows(ws->dtype, variant, a, c);
    if (e != cudaSuccess)
        return cuda_fail(e, "fused kernel launch");
    return AR_OK;
}

}  // namespace

int arf::set_last_error(int code, const char* msg)
{
    g_err = msg;
    return code;
}

// ======================================================================= ABI

extern "C" {

int ar_fusion_version(void) { return 10000; }

const char* ar_fusion_last_error(void) { return g_err.c_str(); }

int ar_fusion_workspace_bytes(int tp_size, int max_token_num, int hidden_dim, int dtype,
                              size_t* bytes)
{
    if (!bytes)
        return fail(AR_ERR_INVALID, "bytes is NULL");
    int rc = check_shape(tp_size, max_token_num, hidden_dim, dtype);
    if (rc)
        return rc;
    *bytes = (size_t)layout_of(tp_size, max_token_num, hidden_dim, dtype).total;
    return AR_OK;
}

int ar_fusion_workspace_create(int tp_size, int max_token_num, int hidden_dim, int dtype,
                               void* device_mem, size_t device_mem_bytes, void* stream,
                               ar_fusion_ws** out)
{
    if (!out)
        return fail(AR_ERR_INVALID, "out is NULL");
    *out = nullptr;
    int rc = check_shape(tp_size, max_token_num, hidden_dim, dtype);
    if (rc)
        return rc;
    const Layout L = layout_of(tp_size, max_token_num, hidden_dim, dtype);
    if (device_mem && (device_mem_bytes < L.total || ((uintptr_t)device_mem & 255)))
        return fail(AR_ERR_INVALID, "device_mem too small (%zu < %llu) or not 256-byte aligned",
                    device_mem_bytes, (unsigned long long)L.total);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    ar_fusion_ws* ws = new (std::nothrow) ar_fusion_ws();
    if (!ws)
        return fail(AR_ERR_INVALID, "out of host memory");
    ws->R = tp_size;
    ws->maxT = max_token_num;
    ws->H = hidden_dim;
    ws->dtype = dtype;
    ws->device = dev;
    ws->sms = sms;
    ws->owned = device_mem == nullptr;
    ws->total = L.total;
    ws->buffer_off = L.buffer_off;
    ws->buffer_bytes = L.buffer_bytes;
    ws->flag_off = L.flag_off;
    ws->flag_bytes = L.flag_bytes;
    ws->lamport_off = L.lamport_off;
    ws->slot_bytes = L.slot_bytes;
    ws->state_off = L.state_off;
    ws->variant = AR_VARIANT_AUTO;
    ws->last_variant = AR_VARIANT_AUTO;
    ws->last_cluster = 0;
    ws->cluster = 0;
    // programmatic dependent launch by default: the row kernels wait on the
    // device for the preceding grid before their first read, and measured
    // faster with it wherever they run (us per call, CUDA graphs: R=8,
    // T=128, H=4096 3.29 -> 2.98, Lamport 6.45 -> 5.77; R=2, T=16, H=512
    // Lamport 3.29 -> 2.66; R=4, T=2048, H=8192 FP8 40.6 -> 40.1; R=8,
    // T=8192, H=7168 NVFP4 178.4 -> 177.8)
    ws->pdl = 1;
    ws->acc = AR_ACC_FP32;
    ws->sf_layout = AR_SF_LINEAR;
    ws->mode = AR_MODE_AUTO;
    ws->timeout_ns = 2000000000ull;
    if (ws->owned) {
        void* p = nullptr;
        e = cudaMalloc(&p, L.total);
        if (e != cudaSuccess) {
            delete ws;
            return cuda_fail(e, "cudaMalloc(workspace)");
        }
        ws->base = static_cast<uint8_t*>(p);
    } else {
        ws->base = static_cast<uint8_t*>(device_mem);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = init_regions(ws, s);
    if (rc == AR_OK) {
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess)
            rc = cuda_fail(e, "cudaStreamSynchronize(create)");
    }
    if (rc != AR_OK) {
        if (ws->owned)
            cudaFree(ws->base);
        delete ws;
        return rc;
    }
    *out = ws;
    return AR_OK;
}

int ar_fusion_workspace_destroy(ar_fusion_ws* ws)
{
    if (!ws)
        return AR_OK;
    int rc = AR_OK;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        rc = cuda_fail(e, "cudaDeviceSynchronize(destroy)");
    if (ws->owned) {
        e = cudaFree(ws->base);
        if (e != cudaSuccess && rc == AR_OK)
            rc = cuda_fail(e, "cudaFree(workspace)");
    }
    delete ws;
    return rc;
}

int ar_fusion_workspace_info(const ar_fusion_ws* ws, ar_fusion_ws_info* info)
{
    if (!ws || !info)
        return fail(AR_ERR_INVALID, "workspace or info is NULL");
    memset(info, 0, sizeof *info);
    info->tp_size = ws->R;
    info->max_token_num = ws->maxT;
    info->hidden_dim = ws->H;
    info->dtype = ws->dtype;
    info->elem_bytes = elem_bytes(ws->dtype);
    info->oneshot_max_tokens = AR_ONESHOT_MAX_TOKENS;
    info->total_bytes = ws->total;
    info->buffer_bytes = ws->buffer_bytes;
    info->flag_bytes = ws->flag_bytes;
    info->lamport_comm_bytes = ws->slot_bytes;
    info->lamport_buffer_bytes = 3 * ws->slot_bytes;
    info->state_bytes = sizeof(ar_fusion_state);
    info->base = ws->base;
    info->buffer = ws->base + ws->buffer_off;
    info->flags = ws->base + ws->flag_off;
    info->lamport = ws->base + ws->lamport_off;
    info->state = ws->base + ws->state_off;
    info->last_variant = ws->last_variant;
    info->last_cluster = ws->last_cluster;
    return AR_OK;
}

int ar_fusion_workspace_copy_state(ar_fusion_ws* ws, void* stream, ar_fusion_state* out)
{
    if (!ws || !out)
        return fail(AR_ERR_INVALID, "workspace or out is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(out, state_of(ws), sizeof *out, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "reading workspace state");
    return AR_OK;
}

int ar_fusion_workspace_status(ar_fusion_ws* ws, void* stream, int* detail)
{
    ar_fusion_state st;
    int rc = ar_fusion_workspace_copy_state(ws, stream, &st);
    if (rc)
        return rc;
    if (detail)
        *detail = st.detail;
    if (st.status != 0)
        return fail(st.status, "device reported status %d (detail %d)", st.status, st.detail);
    return AR_OK;
}

int ar_fusion_workspace_reset(ar_fusion_ws* ws, void* stream)
{
    if (!ws)
        return fail(AR_ERR_INVALID, "workspace is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint64_t words = 3 * ws->slot_bytes / 4;
    fill_u32_kernel<<<grid_for(words, 256, ws->sms), 256, 0, s>>>(
        reinterpret_cast<uint32_t*>(ws->base + ws->lamport_off), words, 0x80000000u);
    init_state_kernel<<<1, 1, 0, s>>>(state_of(ws), ws->slot_bytes);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "workspace reset kernels");
    return AR_OK;
}

int ar_fusion_workspace_set_timeout_ns(ar_fusion_ws* ws, uint64_t ns)
{
    if (!ws || ns == 0)
        return fail(AR_ERR_INVALID, "workspace NULL or timeout 0");
    ws->timeout_ns = ns;
    return AR_OK;
}

int ar_fusion_workspace_set_variant(ar_fusion_ws* ws, int variant)
{
    if (!ws || variant < AR_VARIANT_AUTO || variant > AR_VARIANT_BULK_PIPE)
        return fail(AR_ERR_INVALID, "workspace NULL or variant %d unknown", variant);
    ws->variant = variant;
    return AR_OK;
}

int ar_fusion_workspace_set_launch(ar_fusion_ws* ws, int cluster_size, int pdl)
{
    if (!ws)
        return fail(AR_ERR_INVALID, "workspace is NULL");
    if (cluster_size != 0 && cluster_size != 1 && cluster_size != 2 && cluster_size != 4 &&
        cluster_size != 8)
        return fail(AR_ERR_INVALID, "cluster_size %d is not 0 (auto), 1, 2, 4 or 8", cluster_size);
    if (pdl != 0 && pdl != 1)
        return fail(AR_ERR_INVALID, "pdl %d is not 0 or 1", pdl);
    ws->cluster = cluster_size;
    ws->pdl = pdl;
    return AR_OK;
}

int ar_fusion_workspace_set_accumulate(ar_fusion_ws* ws, int accumulate)
{
    if (!ws || (accumulate != AR_ACC_FP32 && accumulate != AR_ACC_ELEMENT))
        return fail(AR_ERR_INVALID, "workspace NULL or accumulate %d unknown", accumulate);
    ws->acc = accumulate;
    return AR_OK;
}

int ar_fusion_workspace_set_scale_layout(ar_fusion_ws* ws, int layout)
{
    if (!ws || (layout != AR_SF_LINEAR && layout != AR_SF_SWIZZLED))
        return fail(AR_ERR_INVALID, "workspace NULL or scale layout %d unknown", layout);
    ws->sf_layout = layout;
    return AR_OK;
}

int ar_fusion_workspace_set_mode(ar_fusion_ws* ws, int mode)
{
    if (!ws || mode < AR_MODE_AUTO || mode > AR_MODE_BUFFER)
        return fail(AR_ERR_INVALID, "workspace NULL or mode %d unknown", mode);
    ws->mode = mode;
    return AR_OK;
}

int ar_fusion_workspace_stage(ar_fusion_ws* ws, int rank, const void* src, int tokens, int mode,
                              void* stream)
{
    if (!ws)
        return fail(AR_ERR_INVALID, "workspace is NULL");
    if (rank < 0 || rank >= ws->R)
        return fail(AR_ERR_INVALID, "rank %d outside 0..%d", rank, ws->R - 1);
    if (mode < AR_MODE_AUTO || mode > AR_MODE_BUFFER)
        return fail(AR_ERR_INVALID, "mode %d unknown", mode);
    if (tokens < 0)
        return fail(AR_ERR_INVALID, "tokens %d < 0", tokens);
    if (tokens > ws->maxT)
        return fail(AR_ERR_CAPACITY, "tokens %d > max_token_num %d", tokens, ws->maxT);
    if (tokens == 0)
        return AR_OK;
    if (!src || !vec_aligned(src, ws->dtype))
        return fail(AR_ERR_INVALID, "src NULL or not vector aligned");
    mode = resolve_mode(ws, mode, tokens);
    const uint64_t eb = (uint64_t)elem_bytes(ws->dtype);
    const uint64_t plane = (uint64_t)tokens * ws->H * eb;
    const uint64_t nvec = plane / 16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (mode == AR_MODE_LAMPORT) {
        stage_kernel<<<grid_for(nvec, 256, ws->sms), 256, 0, s>>>(
            static_cast<const uint4*>(src), ws->base + ws->lamport_off, ws->slot_bytes,
            (uint64_t)rank * plane, nvec, 1, state_of(ws));
    } else {
        stage_kernel<<<grid_for(nvec, 256, ws->sms), 256, 0, s>>>(
            static_cast<const uint4*>(src), ws->base + ws->buffer_off, 0,
            (uint64_t)rank * ws->maxT * ws->H * eb, nvec, 0, state_of(ws));
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return cuda_fail(e, "stage kernel launch");
    return AR_OK;
}

int ar_fusion_workspace_partial_ptr(ar_fusion_ws* ws, int rank, int tokens, int mode,
                                    void* stream, void** out)
{
    if (!ws || !out)
        return fail(AR_ERR_INVALID, "workspace or out is NULL");
    *out = nullptr;
    if (rank < 0 || rank >= ws->R)
        return fail(AR_ERR_INVALID, "rank %d outside 0..%d", rank, ws->R - 1);
    if (mode < AR_MODE_AUTO || mode > AR_MODE_BUFFER)
        return fail(AR_ERR_INVALID, "mode %d unknown", mode);
    if (tokens < 1)
        return fail(AR_ERR_INVALID, "tokens %d < 1", tokens);
    if (tokens > ws->maxT)
        return fail(AR_ERR_CAPACITY, "tokens %d > max_token_num %d", tokens, ws->maxT);
    mode = resolve_mode(ws, mode, tokens);
    const uint64_t eb = (uint64_t)elem_bytes(ws->dtype);
    if (mode == AR_MODE_BUFFER) {
        *out = ws->base + ws->buffer_off + (uint64_t)rank * ws->maxT * ws->H * eb;
        return AR_OK;
    }
    ar_fusion_state st;
    int rc = ar_fusion_workspace_copy_state(ws, stream, &st);
    if (rc)
        return rc;
    *out = ws->base + ws->lamport_off + (uint64_t)(st.lamport_flag % 3u) * ws->slot_bytes +
           (uint64_t)rank * tokens * ws->H * eb;
    return AR_OK;
}

int ar_fusion_run(ar_fusion_ws* ws, const void* const* partials, int nranks, int tokens,
                  int hidden_dim, int dtype, const void* residual_in, const void* gamma,
                  float eps, int pattern, void* residual_out, void* norm_out, void* quant_out,
                  void* scale_out, const float* scale_factor, void* stream)
{
    FusedArgs a;
    bool launch = false;
    int rc = prepare(ws, partials, nranks, tokens, hidden_dim, dtype, residual_in, gamma, eps,
                     pattern, residual_out, norm_out, quant_out, scale_out, scale_factor, false, a,
                     launch);
    if (rc || !launch)
        return rc;
    return launch_fused(ws, a, static_cast<cudaStream_t>(stream));
}

int ar_fusion_norm_amax(ar_fusion_ws* ws, const void* const* partials, int nranks, int tokens,
                        int hidden_dim, int dtype, const void* residual_in, const void* gamma,
                        float eps, float* amax_out, void* stream)
{
    if (!amax_out || ((uintptr_t)amax_out & 3))
        return fail(AR_ERR_INVALID, "amax_out NULL or misaligned");
    FusedArgs a;
    bool launch = false;
    int rc = prepare(ws, partials, nranks, tokens, hidden_dim, dtype, residual_in, gamma, eps, 0,
                     nullptr, nullptr, nullptr, nullptr, nullptr, true, a, launch);
    if (rc)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMemsetAsync(amax_out)");
    if (!launch)
        return AR_OK;
    a.amax_out = amax_out;
    const LaunchCfg c{ws->sms, s};
    const int variant = a.H <= 512 ? AR_VARIANT_WARP_ROW : AR_VARIANT_CTA_ROW;
    e = launch_fused_rows(ws->dtype, variant, a, c);
    if (e != cudaSuccess)
        return cuda_fail(e, "amax kernel launch");
    return AR_OK;
}

int ar_fusion_sum(const void* const* bufs, int nranks, size_t n, int dtype, void* out,
                  void* stream)
{
    return ar_fusion_sum_ex(bufs, nranks, n, dtype, AR_ACC_FP32, out, stream);
}

int ar_fusion_sum_ex(const void* const* bufs, int nranks, size_t n, int dtype, int accumulate,
                     void* out, void* stream)
{
    if (accumulate != AR_ACC_FP32 && accumulate != AR_ACC_ELEMENT)
        return fail(AR_ERR_INVALID, "accumulate %d unknown", accumulate);
    if (!dtype_supported(dtype))
        return fail(AR_ERR_UNSUPPORTED, "dtype %d is not bf16 (0), fp16 (1) or fp32 (2)", dtype);
    if (nranks < 1 || nranks > AR_MAX_RANKS)
        return fail(AR_ERR_UNSUPPORTED, "nranks %d outside 1..%d", nranks, AR_MAX_RANKS);
    if (n == 0)
        return AR_OK;
    const uintptr_t emask = (uintptr_t)elem_bytes(dtype) - 1;
    if (!bufs || !out || ((uintptr_t)out & emask))
        return fail(AR_ERR_INVALID, "bufs / out NULL or out misaligned");
    SumArgs a;
    memset(&a, 0, sizeof a);
    for (int r = 0; r < nranks; ++r) {
        if (!bufs[r] || ((uintptr_t)bufs[r] & emask))
            return fail(AR_ERR_INVALID, "bufs[%d] NULL or misaligned", r);
        a.in[r] = static_cast<const uint8_t*>(bufs[r]);
    }
    a.out = static_cast<uint8_t*>(out);
    a.R = nranks;
    a.n = n;
    a.acc = accumulate;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "device query");
    e = launch_vector_sum(dtype, a, LaunchCfg{sms, static_cast<cudaStream_t>(stream)});
    if (e != cudaSuccess)
        return cuda_fail(e, "sum kernel launch");
    return AR_OK;
}

}  // extern "C"
