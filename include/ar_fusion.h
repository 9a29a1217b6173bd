/*
 * ar_fusion.h -- C ABI of the GB300 allreduce-fusion epilogue library
 * (libarfusion.so, sm_103a).
 *
 * The operation (per token row t of a [tokens][hidden] problem, element type D
 * = bf16, fp16 or fp32; round_D is the identity for fp32):
 *
 *   s_h  = P_0[t][h] + P_1[t][h] + ... + P_{R-1}[t][h]  (fp32, rank order)
 *   a_h  = round_D(s_h)
 *   y_h  = round_D(a_h + residual_in[t][h])                -> residual_out
 *   rstd = 1 / sqrt(sum_h y_h^2 / hidden + eps)            (fp32)
 *   n_h  = round_D((y_h * rstd) * gamma_h)                 -> norm_out
 *   optional: FP8 E4M3 per-tensor codes of n, or NVFP4 codes + E4M3 block
 *   scales of n                                            -> quant_out, scale_out
 *
 * Sources (page title, function):
 *   TensorRT-LLM cpp/tensorrt_llm/kernels/allReduceFusionKernels.cu --
 *     allreduce_sum (fp32 accumulation in rank order, Fp32Acc), add128 and
 *     fused_op (residual add, optional outputs), rms_norm (sum of squares,
 *     acc / hidden_dim + eps, x * s * gamma), allreduce_fusion_op (argument
 *     checks and the four output patterns), LamportComm and
 *     allreduce_fusion_kernel_oneshot_lamport (triple-buffered slots, -0.0
 *     sentinel, retired-slot clear), lamport_initialize, Workspace.
 *   FlashInfer docs, flashinfer.comm.trtllm_create_ipc_workspace_for_all_reduce_fusion
 *     (workspace regions [buffer, flags, lamport x3], metadata fields).
 *   mscclpp python/mscclpp_benchmark/allreduce.cu -- vectorSum (plain R-way sum).
 *
 * One GPU.  The R rank partials that a tensor-parallel all-reduce would
 * exchange are R device buffers: either caller-owned pointers, or regions of
 * the workspace filled with ar_fusion_workspace_stage().  Nothing crosses
 * GPUs.
 *
 * Conventions for every entry point:
 *   - Device pointers are plain CUDA device addresses; `stream` is a
 *     cudaStream_t passed as void* (NULL = legacy default stream).
 *   - All calls that launch work are asynchronous on `stream` and never
 *     synchronise the device.  Exceptions, stated per call: create, destroy,
 *     status and copy_state synchronise `stream`.
 *   - Every call returns an ar_status code and never throws or aborts.  Invalid
 *     arguments are rejected before anything is launched.  The message for the
 *     last failure on the calling thread is ar_fusion_last_error().
 *   - All device pointers must be 16-byte aligned, fp32 element arrays 32-byte
 *     aligned (AR_ERR_INVALID otherwise).
 *   - The caller owns every tensor; the library owns the workspace object and,
 *     unless the caller supplied it, the workspace memory.
 *   - Launching calls may be captured into a CUDA graph once the same call
 *     (same shapes and options) has run uncaptured, which fills the
 *     library's host-side launch caches.  The Lamport slot state lives in
 *     device memory, so every replay reads the slot its own staging filled
 *     and retires the previous one.
 *   - Device-side waits are bounded: a wait that gives up records
 *     AR_ERR_TIMEOUT in the workspace status word (ar_fusion_workspace_status)
 *     instead of hanging the GPU.
 */
#ifndef AR_FUSION_H
#define AR_FUSION_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ constants -- */

/* Element types of partials, residual, gamma and the residual / norm
 * outputs.  AR_DT_FP32 is the 4-byte exchange type of FlashInfer's
 * trtllm_create_ipc_workspace_for_all_reduce_fusion(use_fp32_lamport=True):
 * the workspace regions hold fp32 elements, and every rounding to the element
 * type is the identity.  fp32 device pointers (partials, residual_in, gamma,
 * residual_out, norm_out; fp32 sum inputs and output on the vector path) must
 * be 32-byte aligned. */
enum ar_dtype {
    AR_DT_BF16 = 0,
    AR_DT_FP16 = 1,
    AR_DT_FP32 = 2
};

/* Output pattern bits.  Valid patterns are the four of allreduce_fusion_op
 * (TensorRT-LLM allReduceFusionKernels.cu), with QUANT = exactly one of
 * AR_QUANT_FP8 / AR_QUANT_NVFP4:
 *     RESIDUAL_OUT | QUANT            NORM_OUT
 *     RESIDUAL_OUT | NORM_OUT         RESIDUAL_OUT | NORM_OUT | QUANT      */
enum ar_pattern {
    AR_RESIDUAL_OUT = 1,
    AR_NORM_OUT = 2,
    AR_QUANT_FP8 = 4,
    AR_QUANT_NVFP4 = 8
};

enum ar_status {
    AR_OK = 0,
    AR_ERR_INVALID = -1,      /* bad argument (null, misaligned, bad pattern ...) */
    AR_ERR_UNSUPPORTED = -2,  /* valid request outside what the kernels implement */
    AR_ERR_CUDA = -3,         /* a CUDA runtime call failed; see ar_fusion_last_error */
    AR_ERR_TIMEOUT = -4,      /* a bounded device-side wait gave up */
    AR_ERR_CAPACITY = -5      /* staged tokens > max_token_num of the workspace
                                 (or beyond the no-allocation scratch) */
};

/* Accumulation of the rank sum (TensorRT-LLM allReduceFusionKernels.cu:
 * allreduce_sum with Fp32Acc, the default of use_fp32_acc, or chained add128
 * in the element type; mscclpp allreduce.cu vectorSum adds in the element
 * type). */
enum ar_accumulate {
    AR_ACC_FP32 = 0,          /* fp32, rank order, rounded to the element type once */
    AR_ACC_ELEMENT = 1        /* rounded to the element type after every addition */
};

/* Layout of the NVFP4 block-scale bytes (scale_out). */
enum ar_scale_layout {
    AR_SF_LINEAR = 0,         /* [tokens][hidden/16], row-major */
    AR_SF_SWIZZLED = 1        /* tiles of 128 rows x 4 blocks, see ar_fusion_workspace_set_scale_layout */
};

/* Where ar_fusion_run reads the partials from when `partials` is NULL. */
enum ar_mode {
    AR_MODE_AUTO = 0,         /* tokens <= AR_ONESHOT_MAX_TOKENS -> LAMPORT, else BUFFER */
    AR_MODE_LAMPORT = 1,      /* current Lamport slot: polled for the -0.0 sentinel,
                                 retired slot cleared, slot index advanced */
    AR_MODE_BUFFER = 2        /* the buffer region, rank r at r * max_token_num * hidden */
};

/* Kernel variant.  AUTO: one row per warp for hidden <= 512; the bulk-copy
 * pipe for inputs ((nranks + 1) * tokens * hidden elements) of at least
 * 96 MiB outside Lamport mode when a row needs more than one vector of 8
 * elements per thread of a row block (bf16/fp16: hidden > 7168 with more
 * than 4 ranks, > 12288 with 3 or 4, > 16384 with 1 or 2; fp32: > 4096), or
 * nranks > 8 with rows of more than 8 KB; else one row per thread block. */
enum ar_variant {
    AR_VARIANT_AUTO = 0,
    AR_VARIANT_WARP_ROW = 1,  /* one row per warp (small hidden) */
    AR_VARIANT_CTA_ROW = 2,   /* one row per thread block, loads straight to registers */
    AR_VARIANT_BULK_PIPE = 3  /* persistent blocks, rank rows streamed into shared
                                 memory by bulk async copies (large token counts) */
};

#define AR_MAX_RANKS 16
/* Token count up to which AR_MODE_AUTO uses the Lamport (one-shot) slots. The
 * page's kOneShotMaxToken lives in a header that is not on the pages; this
 * value is ours. */
#define AR_ONESHOT_MAX_TOKENS 128
/* Barrier flag words per rank in the flags region (the page's
 * kBarrierFlagCount is not on the pages; ours).  Reserved: one GPU needs no
 * cross-rank barrier. */
#define AR_BARRIER_FLAG_COUNT 256
#define AR_MAX_HIDDEN 32768

typedef struct ar_fusion_ws ar_fusion_ws;   /* opaque, library-owned */

/* Workspace description (FlashInfer workspace metadata fields, plus device
 * addresses of each region).  Byte sizes are 64-bit: the page's `int` sizes
 * overflow at 8 ranks x 8192 tokens x 7168 hidden. */
typedef struct ar_fusion_ws_info {
    int32_t tp_size;               /* R */
    int32_t max_token_num;
    int32_t hidden_dim;
    int32_t dtype;                 /* enum ar_dtype */
    int32_t elem_bytes;            /* sizeof(D): 2, or 4 for AR_DT_FP32 */
    int32_t oneshot_max_tokens;    /* AR_ONESHOT_MAX_TOKENS */
    uint64_t total_bytes;          /* whole workspace */
    uint64_t buffer_bytes;         /* R * max_token_num * hidden * elem */
    uint64_t flag_bytes;           /* R * AR_BARRIER_FLAG_COUNT * 4 */
    uint64_t lamport_comm_bytes;   /* one slot: R * max(oneshot, max_token_num) * hidden * elem */
    uint64_t lamport_buffer_bytes; /* three slots */
    uint64_t state_bytes;          /* the state block (struct ar_fusion_state) */
    void* base;                    /* device address of the workspace */
    void* buffer;                  /* base + 0 */
    void* flags;
    void* lamport;                 /* slot k at lamport + k * lamport_comm_bytes */
    void* state;                   /* struct ar_fusion_state */
    int32_t last_variant;          /* enum ar_variant the last fused launch used (0: none yet) */
    int32_t last_cluster;          /* CTAs per row of that launch (1: no cluster; 0: none yet) */
} ar_fusion_ws_info;

/* Device-resident state (the page's 5-int flag array, widened).  Read it with
 * ar_fusion_workspace_copy_state.  Order of the first fields follows the page:
 * counter, flag, lamport flag, lamport comm size, clear size. */
typedef struct ar_fusion_state {
    uint32_t counter;        /* blocks finished in the current launch (0 between calls) */
    uint32_t flag;           /* reserved (non-Lamport flag; unused on one GPU) */
    uint32_t lamport_flag;   /* current slot = lamport_flag % 3 */
    uint32_t clear_elem_bytes; /* bytes per element of clear_size: the element size of
                                  the call that filled the retired slot (2 or 4) */
    uint64_t comm_size;      /* bytes of one Lamport slot */
    uint64_t clear_size;     /* elements of the retired slot still to be cleared */
    int32_t status;          /* AR_OK or the first device-side error (AR_ERR_TIMEOUT) */
    int32_t detail;          /* where it happened (see ar_fusion_workspace_status), or -1 */
    uint64_t calls;          /* Lamport-mode calls since create / reset */
} ar_fusion_state;

/* ------------------------------------------------------------ workspace -- */

/* Bytes of device memory a workspace needs (for caller-supplied memory).
 * Regions, in order and each 256-byte aligned: buffer, flags, three Lamport
 * slots, state.  Returns AR_OK or AR_ERR_INVALID / AR_ERR_UNSUPPORTED. */
int ar_fusion_workspace_bytes(int tp_size, int max_token_num, int hidden_dim, int dtype,
                              size_t* bytes);

/* Create a workspace (Workspace constructor of TensorRT-LLM
 * allReduceFusionKernels.cu; FlashInfer trtllm_create_ipc_workspace_for_all_reduce_fusion).
 *   tp_size        R, 1..AR_MAX_RANKS
 *   max_token_num  largest `tokens` of a call that reads staged partials
 *                  (it sizes the buffer region and the Lamport slots), >= 1;
 *                  calls with caller partials may pass more tokens
 *   hidden_dim     row length, multiple of 8, <= AR_MAX_HIDDEN
 *   dtype          enum ar_dtype
 *   device_mem     NULL: the library allocates (cudaMalloc) and frees the memory.
 *                  Otherwise caller-owned device memory of at least
 *                  ar_fusion_workspace_bytes() bytes, 256-byte aligned, which
 *                  must outlive the workspace.
 *   stream         stream for the initialisation kernels (the Lamport region
 *                  is filled with -0.0f words, lamport_initialize; the rest is
 *                  zeroed); this call synchronises it.
 *   out            receives the handle.
 * Errors: AR_ERR_INVALID, AR_ERR_UNSUPPORTED, AR_ERR_CUDA (allocation). */
int ar_fusion_workspace_create(int tp_size, int max_token_num, int hidden_dim, int dtype,
                               void* device_mem, size_t device_mem_bytes, void* stream,
                               ar_fusion_ws** out);

/* Synchronise the device, free library-owned memory, free the handle.
 * NULL is accepted (no-op). */
int ar_fusion_workspace_destroy(ar_fusion_ws* ws);

/* Fill *info.  No CUDA call.  Errors: AR_ERR_INVALID for a NULL argument. */
int ar_fusion_workspace_info(const ar_fusion_ws* ws, ar_fusion_ws_info* info);

/* Copy the device state block to host memory *out (synchronises `stream`).
 * Errors: AR_ERR_INVALID for a NULL argument, AR_ERR_CUDA if the copy fails. */
int ar_fusion_workspace_copy_state(ar_fusion_ws* ws, void* stream, ar_fusion_state* out);

/* Synchronise `stream`, read the device status word: returns AR_OK, the
 * recorded device error (AR_ERR_TIMEOUT), or AR_ERR_CUDA.  *detail (may be
 * NULL) receives where the first wait gave up: row * 32 + rank for a Lamport
 * poll; for the bulk-copy pipe -1 (a stage wait of the consumers), -2 (the
 * producer waiting for a free stage) or -3 (its final wait for copies in
 * flight); -1 when nothing failed. */
int ar_fusion_workspace_status(ar_fusion_ws* ws, void* stream, int* detail);

/* Re-initialise on `stream`: Lamport region back to -0.0f words, slot index
 * and clear size to 0, status to AR_OK.  Asynchronous. */
int ar_fusion_workspace_reset(ar_fusion_ws* ws, void* stream);

/* Bound, in nanoseconds, of each device-side wait of later launches
 * (default 2e9): the Lamport polls and the bulk-copy pipe's stage waits.  The
 * pipe's final wait for its own copies in flight is bounded by at least
 * 200 ms whatever this value.  Host-side setting; no CUDA call.  Errors:
 * AR_ERR_INVALID for 0. */
int ar_fusion_workspace_set_timeout_ns(ar_fusion_ws* ws, uint64_t ns);

/* Force a kernel variant (enum ar_variant) or staged-read mode (enum
 * ar_mode) for later calls on this workspace; AUTO restores the default
 * choice.  A forced variant that cannot run a call (the bulk-copy pipe in
 * Lamport mode, one row per warp above hidden 1024) falls back to AUTO's
 * choice for that call.  Host-side settings; no CUDA
 * call.  Errors: AR_ERR_INVALID for a NULL workspace or an unknown value. */
int ar_fusion_workspace_set_variant(ar_fusion_ws* ws, int variant);
int ar_fusion_workspace_set_mode(ar_fusion_ws* ws, int mode);

/* Launch options of later fused calls on this workspace (host-side; no CUDA
 * call).  cluster_size: CTAs per token row for the one-row-per-block kernel
 * (TensorRT-LLM allReduceFusionKernels.cu, allreduce_fusion_kernel_launcher
 * splits a token over a thread-block cluster and combines the sum of squares
 * through distributed shared memory, rms_norm): 0 = automatic (one CTA per
 * row: the split measured slower wherever the library picks the row
 * kernel), 1 = no cluster, 2, 4 or 8;
 * used only where each CTA of the cluster still holds one vector (8
 * elements) per thread.  pdl: 1 (the default) = programmatic dependent
 * launch (the same launcher's programmaticStreamSerialization attribute):
 * the fused kernel may be scheduled while the preceding kernel on the
 * stream finishes and waits on the device for its results before its first
 * read, which is safe after any kernel; 0 = plain stream order.  The
 * bulk-copy pipe always launches in plain stream order.  Errors:
 * AR_ERR_INVALID. */
int ar_fusion_workspace_set_launch(ar_fusion_ws* ws, int cluster_size, int pdl);

/* Accumulation of the rank sum of later fused calls (enum ar_accumulate;
 * default AR_ACC_FP32).  Host-side; no CUDA call.  Errors: AR_ERR_INVALID. */
int ar_fusion_workspace_set_accumulate(ar_fusion_ws* ws, int accumulate);

/* Layout of the NVFP4 scale bytes written by later fused calls (enum
 * ar_scale_layout; default AR_SF_LINEAR).  TensorRT-LLM's fused_op writes the
 * scales through cvt_quant_to_fp4_get_sf_out_offset, a header that is not on
 * the pages; AR_SF_SWIZZLED is the block-scale layout that tensor-core NVFP4
 * matrix multiplies consume: with kb = hidden/16 blocks per row and
 * kt = ceil(kb / 4), the scale of (row m, block k) is at byte
 *     ((m / 128) * kt + k / 4) * 512 + (m % 32) * 16 + ((m / 32) % 4) * 4 + k % 4
 * so scale_out must hold ceil(tokens / 128) * 128 * kt * 4 bytes; padding
 * bytes (rows >= tokens, blocks >= kb) are not written -- zero them once if
 * the consumer reads them.  Host-side; no CUDA call.  Errors: AR_ERR_INVALID. */
int ar_fusion_workspace_set_scale_layout(ar_fusion_ws* ws, int layout);

/* Stage rank `rank`'s partial [tokens][hidden] (device pointer `src`) into the
 * workspace, standing in for the one-shot push of
 * allreduce_fusion_kernel_oneshot_lamport (on one GPU nothing is pushed over
 * NVLink; the bytes are copied by a kernel).
 *   mode AR_MODE_LAMPORT: into the current slot (lamport_flag % 3, read on the
 *     device) at rank * tokens * hidden elements; every 32-bit word equal to
 *     the -0.0f sentinel (0x80000000) is written as +0.0f.
 *   mode AR_MODE_BUFFER: into the buffer region at rank * max_token_num *
 *     hidden elements, unchanged.
 *   mode AR_MODE_AUTO: LAMPORT if tokens <= AR_ONESHOT_MAX_TOKENS, else BUFFER
 *     (or the mode forced with ar_fusion_workspace_set_mode).
 * Errors: AR_ERR_INVALID (rank, pointer, mode), AR_ERR_CAPACITY. */
int ar_fusion_workspace_stage(ar_fusion_ws* ws, int rank, const void* src, int tokens, int mode,
                              void* stream);

/* Device address where rank `rank`'s partial of a `tokens`-row call is staged,
 * for producers that write it in place instead of calling
 * ar_fusion_workspace_stage (a matmul epilogue, or a peer's push where the
 * ranks are GPUs).  mode as in ar_fusion_workspace_stage:
 *   AR_MODE_BUFFER: buffer region + rank * max_token_num * hidden elements;
 *     host arithmetic, no CUDA call.
 *   AR_MODE_LAMPORT: current slot + rank * tokens * hidden elements; reads the
 *     slot index from the device (synchronises `stream`).  The producer must
 *     write every element of the [tokens][hidden] block and no 32-bit word
 *     equal to 0x80000000 (write such a -0.0f word as +0.0f, as the staging
 *     kernel does), ordered before the ar_fusion_run that reads it; the slot
 *     changes with every Lamport call.
 * `*out` receives the address (16-byte aligned; 32-byte for fp32).
 * Errors: AR_ERR_INVALID (NULL, rank, mode, tokens < 1), AR_ERR_CAPACITY
 * (tokens > max_token_num), AR_ERR_CUDA. */
int ar_fusion_workspace_partial_ptr(ar_fusion_ws* ws, int rank, int tokens, int mode,
                                    void* stream, void** out);

/* ---------------------------------------------------------- fused call -- */

/* The fused epilogue (allreduce_fusion_op, TensorRT-LLM allReduceFusionKernels.cu).
 *   ws            workspace (status word; staged partials when partials == NULL)
 *   partials      host array of `nranks` device pointers, each [tokens][hidden] D
 *                 (read only), or NULL to read the partials staged in `ws`
 *                 (AR_MODE_AUTO unless forced: Lamport slot for tokens <=
 *                 AR_ONESHOT_MAX_TOKENS, else buffer region)
 *   nranks        R, 1..AR_MAX_RANKS; must equal tp_size when partials == NULL
 *   tokens        rows, >= 0 (0: nothing launched, AR_OK)
 *   hidden_dim    row length, multiple of 8 (of 16 with AR_QUANT_NVFP4),
 *                 <= AR_MAX_HIDDEN; must equal the workspace's when staged
 *   dtype         enum ar_dtype; must equal the workspace's
 *   residual_in   [tokens][hidden] D
 *   gamma         [hidden] D
 *   eps           RMSNorm epsilon (fp32)
 *   pattern       one of the four valid ar_pattern combinations
 *   residual_out  [tokens][hidden] D, written if AR_RESIDUAL_OUT, else ignored
 *   norm_out      [tokens][hidden] D, written if AR_NORM_OUT, else ignored
 *   quant_out     AR_QUANT_FP8: [tokens][hidden] E4M3 bytes;
 *                 AR_QUANT_NVFP4: [tokens][hidden/2] bytes, element 2k in the
 *                 low nibble of byte k
 *   scale_out     AR_QUANT_NVFP4: [tokens][hidden/16] E4M3 block-scale bytes
 *                 (row-major, linear); ignored otherwise
 *   scale_factor  device fp32 scalar: AR_QUANT_FP8: the multiplier 1/scale;
 *                 AR_QUANT_NVFP4: the global encode scale gs (block scale =
 *                 E4M3(gs * blockmax / 6), codes = E2M1(n * gs / blockscale))
 *   stream        CUDA stream
 * Errors (before any launch): AR_ERR_INVALID (null / misaligned pointers, bad
 * pattern, hidden not a multiple of 8 / 16, dtype or hidden mismatch),
 * AR_ERR_UNSUPPORTED (nranks outside 1..16, hidden too large),
 * AR_ERR_CAPACITY (staged and tokens > max_token_num), AR_ERR_CUDA (launch).
 * Device-side: a Lamport-mode wait that gives up sets AR_ERR_TIMEOUT in the
 * status word; outputs of that call are then undefined. */
int ar_fusion_run(ar_fusion_ws* ws, const void* const* partials, int nranks, int tokens,
                  int hidden_dim, int dtype, const void* residual_in, const void* gamma,
                  float eps, int pattern, void* residual_out, void* norm_out, void* quant_out,
                  void* scale_out, const float* scale_factor, void* stream);

/* Calibration pass for the per-tensor quantisers: the same sum, residual add
 * and RMSNorm as ar_fusion_run, writing only amax = max |n| over the whole
 * tensor to the device fp32 *amax_out (overwritten).  Reads caller partials,
 * or the buffer region when partials == NULL (never the Lamport slots, whose
 * state it leaves alone).  Same argument rules as ar_fusion_run. */
int ar_fusion_norm_amax(ar_fusion_ws* ws, const void* const* partials, int nranks, int tokens,
                        int hidden_dim, int dtype, const void* residual_in, const void* gamma,
                        float eps, float* amax_out, void* stream);

/* ---------------------------------------------------------- plain sum -- */

/* out[i] = round_D(in_0[i] + ... + in_{R-1}[i]) in fp32, rank order, for i < n
 * (mscclpp allreduce.cu vectorSum, accumulating in fp32).
 *   bufs    host array of `nranks` device pointers, n elements of D each
 *   nranks  1..AR_MAX_RANKS;  n any size (no alignment tail restriction)
 *   out     n elements of D; may alias none of the inputs
 * Pointers need only element alignment here; 16-byte aligned inputs (bf16,
 * fp16) or 32-byte aligned inputs (fp32) take the vector path.  Errors: AR_ERR_INVALID, AR_ERR_UNSUPPORTED, AR_ERR_CUDA. */
int ar_fusion_sum(const void* const* bufs, int nranks, size_t n, int dtype, void* out,
                  void* stream);

/* ar_fusion_sum with a choice of accumulation (enum ar_accumulate):
 * AR_ACC_ELEMENT rounds every partial sum to the element type, as mscclpp's
 * vectorSum does with half-precision adds.  ar_fusion_sum is AR_ACC_FP32.
 * Errors as ar_fusion_sum, and AR_ERR_INVALID for an unknown accumulate. */
int ar_fusion_sum_ex(const void* const* bufs, int nranks, size_t n, int dtype, int accumulate,
                     void* out, void* stream);

/* ------------------------------------------------- no-allocation call -- */

/* Fixed scratch of ar_fusion_run_noalloc: three slots and the slot state,
 * one array per GPU that loads the library, kept until the process exits. */
#define AR_NOALLOC_SLOT_BYTES (4u << 20)
#define AR_NOALLOC_SCRATCH_BYTES (3u * AR_NOALLOC_SLOT_BYTES + 256u)

/* The one-shot fused call (same operation, arguments and results as
 * ar_fusion_run with caller partials) for callers that must not allocate
 * device memory: code inside a host framework that owns the whole device
 * memory budget and forbids plugins to allocate, or code on a latency-critical
 * path where cudaMalloc / cudaFree (which can synchronise the device) are not
 * allowed.  The pages have no counterpart: there the workspace is always
 * allocated (TensorRT-LLM Workspace, FlashInfer workspace creation).
 *
 * No workspace: the partials (host array of `nranks` device pointers, each
 * [tokens][hidden] D) are staged by a kernel into one of three slots of a
 * fixed device array of AR_NOALLOC_SCRATCH_BYTES, with the -0.0f sentinel
 * flip, then read, summed, normalised and quantised by the Lamport-mode kernel,
 * which refills the previous call's slot with the sentinel and advances the
 * slot index -- all on `stream`.  Nothing is allocated: no cudaMalloc,
 * cudaFree or allocating library call.
 *
 * Limits: nranks * tokens * hidden_dim * sizeof(D) <= AR_NOALLOC_SLOT_BYTES, else
 * AR_ERR_CAPACITY before anything runs.  Other argument rules and errors as
 * ar_fusion_run.
 * Set-up: the first call on each device (the device current at the call)
 * looks up the array's device address (cudaGetSymbolAddress) and launches a
 * one-time fill of it on `stream`; make that first call before any stream
 * capture.
 * Sharing: every call on a device uses the same array and leaves the slot
 * state for the next call; calls whose work overlaps on the GPU (different
 * streams without ordering between them) race on it and give undefined
 * results.  Serialise them (one stream, or events).  Consecutive calls may
 * change element type, ranks and sizes: each call clears exactly the bytes
 * its predecessor left in the retired slot.
 * Device-side errors: a bounded wait that gives up (only possible when calls
 * overlap) records AR_ERR_TIMEOUT in the array's status word, which later
 * calls do not erase; read it with ar_fusion_noalloc_status. */
int ar_fusion_run_noalloc(const void* const* partials, int nranks, int tokens, int hidden_dim,
                          int dtype, const void* residual_in, const void* gamma, float eps,
                          int pattern, void* residual_out, void* norm_out, void* quant_out,
                          void* scale_out, const float* scale_factor, void* stream);

/* Device-side status of ar_fusion_run_noalloc on the current device (no
 * counterpart on the pages).  Synchronises `stream`, then returns the first
 * device-side error recorded by a no-allocation call since set-up or since
 * the previous ar_fusion_noalloc_status call (AR_OK if none; AR_ERR_TIMEOUT
 * when a wait gave up, outputs of that call undefined) and clears it.
 * *detail (may be NULL) receives where it happened -- row * 32 + rank for a
 * wait on a rank's data -- or -1.  Before the first no-allocation call on the
 * device it returns AR_OK and touches nothing.  Allocates nothing; returns
 * AR_ERR_CUDA if reading the status word fails. */
int ar_fusion_noalloc_status(void* stream, int* detail);

/* ---------------------------------------------------------- utilities -- */

/* Message for the last failed call on this thread ("" if none). */
const char* ar_fusion_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int ar_fusion_version(void);

#ifdef __cplusplus
}
#endif

#endif /* AR_FUSION_H */
