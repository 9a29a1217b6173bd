// ar_fusion_run_noalloc: the one-shot (Lamport-slot) fused call with its
// scratch in a fixed device array instead of a caller- or library-allocated
// workspace, for callers that may not allocate device memory.
//
// Who cannot allocate: code that runs inside a host framework which owns the
// whole device-memory budget (a serving engine that sizes one pool at start-up
// and forbids side allocations by its plugins), and code on a latency-critical
// path where cudaMalloc / cudaFree -- which can synchronise the device -- are
// not allowed.  Such callers still pass their own inputs and outputs; only the
// scratch (three Lamport slots and the slot state) comes from here.
//
// The scratch is one file-scope array of AR_NOALLOC_SCRATCH_BYTES per GPU
// that loads the library, held until the process exits.  Host code cannot use
// the array's name as a device address (on the host it names a stand-in
// object), so the device address is looked up once per device with
// cudaGetSymbolAddress and passed to the kernels.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "ar_common.cuh"
#include "ar_internal.h"

namespace {

constexpr uint64_t kSlotBytes = AR_NOALLOC_SLOT_BYTES;
constexpr uint64_t kStateOff = 3 * kSlotBytes;

static_assert(kStateOff + 256 <= AR_NOALLOC_SCRATCH_BYTES, "scratch layout");

// [slot 0 | slot 1 | slot 2 | ar_fusion_state], shared by every call on a device
static __device__ __align__(256) uint8_t g_noalloc_scratch[AR_NOALLOC_SCRATCH_BYTES];

// failures are reported through ar_fusion_last_error()
int nfail(int code, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    return arf::set_last_error(code, buf);
}

__global__ void noalloc_init_kernel(uint8_t* scratch)
{
    uint32_t* w = reinterpret_cast<uint32_t*>(scratch);
    const uint64_t words = kStateOff / 4;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += stride)
        w[i] = 0x80000000u;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        ar_fusion_state* st = reinterpret_cast<ar_fusion_state*>(scratch + kStateOff);
        st->counter = 0;
        st->flag = 0;
        st->lamport_flag = 0;
        st->clear_elem_bytes = 0;
        st->comm_size = kSlotBytes;
        st->clear_size = 0;
        st->status = 0;
        st->detail = -1;
        st->calls = 0;
    }
}

// Copy the caller's R partials into the current slot (lamport_flag % 3, rank r
// at r * plane bytes) with every -0.0f word written as +0.0f.  The status word
// is left alone: a device-side error stays recorded until
// ar_fusion_noalloc_status reads and clears it.
__global__ void noalloc_stage_kernel(arf::FusedArgs a, uint8_t* scratch, uint64_t plane_vecs)
{
    ar_fusion_state* st = reinterpret_cast<ar_fusion_state*>(scratch + kStateOff);
    // one polling load per block (they bypass L1; one per thread would queue
    // thousands of requests on one L2 line)
    __shared__ uint32_t flag_sh;
    if (threadIdx.x == 0)
        flag_sh = *reinterpret_cast<volatile uint32_t*>(&st->lamport_flag);
    __syncthreads();
    const uint32_t flag = flag_sh;
    uint4* slot = reinterpret_cast<uint4*>(scratch + (uint64_t)(flag % 3u) * kSlotBytes);
    const uint64_t total = plane_vecs * (uint64_t)a.R;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const uint64_t r = i / plane_vecs, j = i - r * plane_vecs;
        uint4 v = arf::ld_stream(a.partial[r] + j * 16);
        v.x = v.x == 0x80000000u ? 0u : v.x;
        v.y = v.y == 0x80000000u ? 0u : v.y;
        v.z = v.z == 0x80000000u ? 0u : v.z;
        v.w = v.w == 0x80000000u ? 0u : v.w;
        slot[i] = v;
    }
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

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

// Per-device set-up: device address of the scratch array (looked up with the
// device current) and the one-time sentinel fill, on the caller's stream.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
uint8_t* g_scratch_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

int setup(int dev, cudaStream_t s, uint8_t** scratch, int* sms)
{
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return nfail(AR_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return nfail(AR_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        noalloc_init_kernel<<<n * 4, 256, 0, s>>>(static_cast<uint8_t*>(p));
        e = cudaGetLastError();
        if (e != cudaSuccess)
            return nfail(AR_ERR_CUDA, "scratch init launch: %s", cudaGetErrorString(e));
        g_sms[dev] = n;
        g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *scratch = g_scratch_ptr[dev];
    *sms = g_sms[dev];
    return AR_OK;
}

}  // namespace

extern "C" {

int ar_fusion_run_noalloc(const void* const* partials, int nranks, int tokens, int hidden_dim,
                          int dtype, const void* residual_in, const void* gamma, float eps,
                          int pattern, void* residual_out, void* norm_out, void* quant_out,
                          void* scale_out, const float* scale_factor, void* stream)
{
    if (!arf::dtype_supported(dtype))
        return nfail(AR_ERR_UNSUPPORTED, "dtype %d is not bf16 (0), fp16 (1) or fp32 (2)", dtype);
    if (nranks < 1 || nranks > AR_MAX_RANKS)
        return nfail(AR_ERR_UNSUPPORTED, "nranks %d outside 1..%d", nranks, AR_MAX_RANKS);
    if (tokens < 0)
        return nfail(AR_ERR_INVALID, "tokens %d < 0", tokens);
    if (hidden_dim <= 0 || hidden_dim % 8 != 0)
        return nfail(AR_ERR_INVALID, "hidden_dim %d is not a positive multiple of 8", hidden_dim);
    if (hidden_dim > AR_MAX_HIDDEN)
        return nfail(AR_ERR_UNSUPPORTED, "hidden_dim %d > %d", hidden_dim, AR_MAX_HIDDEN);
    if (!valid_pattern(pattern))
        return nfail(AR_ERR_INVALID, "unsupported pattern 0x%x", pattern);
    if ((pattern & AR_QUANT_NVFP4) && hidden_dim % 16 != 0)
        return nfail(AR_ERR_INVALID, "NVFP4 needs hidden_dim %% 16 == 0 (got %d)", hidden_dim);
    const uint64_t plane = (uint64_t)tokens * hidden_dim * arf::elem_bytes(dtype);
    if (plane * (uint64_t)nranks > kSlotBytes)
        return nfail(AR_ERR_CAPACITY,
                     "nranks * tokens * hidden_dim * elem = %llu bytes exceeds the fixed scratch "
                     "slot of %llu bytes",
                     (unsigned long long)(plane * (uint64_t)nranks),
                     (unsigned long long)kSlotBytes);
    if (tokens == 0)
        return AR_OK;
    if (!partials)
        return nfail(AR_ERR_INVALID, "partials is NULL");
    const auto va = [dtype](const void* p) { return arf::vec_aligned(p, dtype); };
    if (!residual_in || !gamma || !va(residual_in) || !va(gamma))
        return nfail(AR_ERR_INVALID, "residual_in / gamma NULL or not vector aligned");
    if ((pattern & AR_RESIDUAL_OUT) && (!residual_out || !va(residual_out)))
        return nfail(AR_ERR_INVALID, "residual_out NULL or not vector aligned");
    if ((pattern & AR_NORM_OUT) && (!norm_out || !va(norm_out)))
        return nfail(AR_ERR_INVALID, "norm_out NULL or not vector aligned");
    if (pattern & (AR_QUANT_FP8 | AR_QUANT_NVFP4)) {
        if (!quant_out || !aligned16(quant_out))
            return nfail(AR_ERR_INVALID, "quant_out NULL or not 16-byte aligned");
        if (!scale_factor || ((uintptr_t)scale_factor & 3))
            return nfail(AR_ERR_INVALID, "scale_factor NULL or misaligned");
    }
    if ((pattern & AR_QUANT_NVFP4) && (!scale_out || !aligned16(scale_out)))
        return nfail(AR_ERR_INVALID, "scale_out NULL or not 16-byte aligned");

    arf::FusedArgs a;
    memset(&a, 0, sizeof a);
    for (int r = 0; r < nranks; ++r) {
        if (!partials[r] || !va(partials[r]))
            return nfail(AR_ERR_INVALID, "partials[%d] NULL or not vector aligned", r);
        a.partial[r] = static_cast<const uint8_t*>(partials[r]);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return nfail(AR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return nfail(AR_ERR_UNSUPPORTED, "device %d beyond %d", dev, kMaxDevices);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* scratch = nullptr;
    int sms = 0;
    int rc = setup(dev, s, &scratch, &sms);
    if (rc)
        return rc;

    a.R = nranks;
    a.T = tokens;
    a.H = hidden_dim;
    a.pattern = pattern;
    a.residual_in = static_cast<const uint8_t*>(residual_in);
    a.gamma = static_cast<const uint8_t*>(gamma);
    a.eps = eps;
    a.residual_out = (pattern & AR_RESIDUAL_OUT) ? static_cast<uint8_t*>(residual_out) : nullptr;
    a.norm_out = (pattern & AR_NORM_OUT) ? static_cast<uint8_t*>(norm_out) : nullptr;
    a.quant_out = (pattern & (AR_QUANT_FP8 | AR_QUANT_NVFP4)) ? static_cast<uint8_t*>(quant_out)
                                                              : nullptr;
    a.scale_out = (pattern & AR_QUANT_NVFP4) ? static_cast<uint8_t*>(scale_out) : nullptr;
    a.scale_factor = (pattern & (AR_QUANT_FP8 | AR_QUANT_NVFP4)) ? scale_factor : nullptr;
    a.lamport = 1;
    a.lamport_base = scratch;
    a.slot_bytes = kSlotBytes;
    a.state = reinterpret_cast<ar_fusion_state*>(scratch + kStateOff);
    a.timeout_ns = 2000000000ull;

    const uint64_t plane_vecs = plane / 16;
    uint64_t blocks = (plane_vecs * nranks + 255) / 256;
    if (blocks > (uint64_t)sms * 8)
        blocks = (uint64_t)sms * 8;
    noalloc_stage_kernel<<<(unsigned)blocks, 256, 0, s>>>(a, scratch, plane_vecs);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return nfail(AR_ERR_CUDA, "stage launch: %s", cudaGetErrorString(e));
    const arf::LaunchCfg c{sms, s};
    e = arf::launch_fused_rows(dtype, hidden_dim <= 512 ? AR_VARIANT_WARP_ROW : AR_VARIANT_CTA_ROW,
                               a, c);
    if (e != cudaSuccess)
        return nfail(AR_ERR_CUDA, "fused kernel launch: %s", cudaGetErrorString(e));
    return AR_OK;
}

int ar_fusion_noalloc_status(void* stream, int* detail)
{
    if (detail)
        *detail = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return nfail(AR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return nfail(AR_ERR_UNSUPPORTED, "device %d beyond %d", dev, kMaxDevices);
    uint8_t* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_setup_mu);
        scratch = g_scratch_ptr[dev];
    }
    if (!scratch)
        return AR_OK;  // no call has run on this device yet
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t word[2] = {0, -1};  // status, detail
    uint8_t* at = scratch + kStateOff + offsetof(ar_fusion_state, status);
    e = cudaMemcpyAsync(word, at, sizeof word, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
        return nfail(AR_ERR_CUDA, "reading the scratch status: %s", cudaGetErrorString(e));
    if (word[0] != AR_OK) {
        static const int32_t clean[2] = {0, -1};
        e = cudaMemcpyAsync(at, clean, sizeof clean, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(s);
        if (e != cudaSuccess)
            return nfail(AR_ERR_CUDA, "clearing the scratch status: %s", cudaGetErrorString(e));
    }
    if (detail)
        *detail = word[1];
    return word[0];
}

}  // extern "C"
