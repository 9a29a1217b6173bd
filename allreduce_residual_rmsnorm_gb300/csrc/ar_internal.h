// Host/device shared internals of libarfusion (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ar_fusion.h"

namespace arf {

// Everything one fused launch needs, passed by value as the kernel parameter.
struct FusedArgs {
    const uint8_t* partial[AR_MAX_RANKS];  // per-rank [T][H] bases (unused in Lamport mode)
    int R, T, H, pattern;
    const uint8_t* residual_in;
    const uint8_t* gamma;
    float eps;
    uint8_t* residual_out;
    uint8_t* norm_out;
    uint8_t* quant_out;
    uint8_t* scale_out;
    const float* scale_factor;
    float* amax_out;            // calibration pass: atomic max of |n| (as uint bits)
    // Lamport (one-shot) staged mode
    int lamport;
    uint8_t* lamport_base;      // slot k at lamport_base + k * slot_bytes
    uint64_t slot_bytes;
    ar_fusion_state* state;     // status word always; slot state in Lamport mode
    uint64_t timeout_ns;
    int acc;                    // 1: round the rank sum to the element type after every add
    int sf_layout;              // NVFP4 scale bytes: AR_SF_LINEAR or AR_SF_SWIZZLED
};

struct LaunchCfg {
    int sms;                    // multiprocessor count of the current device
    cudaStream_t stream;
    int cluster = 1;            // CTAs per row (one-row-per-block kernel), 1, 2, 4 or 8
    int pdl = 0;                // programmatic dependent launch
    int* used_cluster = nullptr;  // out: CTAs per row the row kernel was launched with
};

// Kernel launchers (return cudaError_t of the launch).  `variant` is a
// concrete AR_VARIANT_* (never AUTO).
cudaError_t launch_fused_rows(int dtype, int variant, const FusedArgs& a, const LaunchCfg& c);
cudaError_t launch_fused_pipe(int dtype, const FusedArgs& a, const LaunchCfg& c);
bool fused_pipe_supported(int dtype, int H, int R);

struct SumArgs {
    const uint8_t* in[AR_MAX_RANKS];
    uint8_t* out;
    int R;
    uint64_t n;
    int acc;                    // 1: round to the element type after every add
};
cudaError_t launch_vector_sum(int dtype, const SumArgs& a, const LaunchCfg& c);

// Element types and the alignment their vector accesses need: 16 bytes for
// bf16 / fp16 (128-bit), 32 bytes for fp32 (256-bit).
inline bool dtype_supported(int dtype)
{
    return dtype == AR_DT_BF16 || dtype == AR_DT_FP16 || dtype == AR_DT_FP32;
}
inline int elem_bytes(int dtype) { return dtype == AR_DT_FP32 ? 4 : 2; }
inline bool vec_aligned(const void* p, int dtype)
{
    return ((uintptr_t)p & (dtype == AR_DT_FP32 ? 31u : 15u)) == 0;
}

// Threads of a one-vector-per-thread row block (one row per block): bf16 /
// fp16 up to 896 (72 registers each) with up to 8 ranks, 1024 (64 registers)
// with up to 4; fp32 vectors take twice the registers: up to 512.  Rows of
// more vectors take several vectors per thread.
__host__ __device__ constexpr int one_vec_threads_for(int elem_bytes, int nranks)
{
    return elem_bytes == 4 ? 512 : (nranks <= 4 ? 1024 : 896);
}

// Record `msg` as the calling thread's ar_fusion_last_error() text; returns code.
int set_last_error(int code, const char* msg);

}  // namespace arf
