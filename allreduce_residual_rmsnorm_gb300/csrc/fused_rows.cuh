// Register-resident fused epilogue: one row per warp or one row per block.
//
// Per token row (TensorRT-LLM allReduceFusionKernels.cu: allreduce_sum,
// fused_op, add128, rms_norm):
//   s = sum_r f(P_r)  (fp32, rank order)    a = rnd(s)
//   y = rnd(f(a) + f(x))                    -> residual_out
//   ss = sum y^2 (double-float pair, rounded once)
//   rstd = 1 / sqrt(ss / H + eps)           (IEEE div / sqrt)
//   n = rnd((y * rstd) * gamma)             -> norm_out, FP8 / NVFP4 codes
//
// Each row is split into vectors of 8 elements (16 bytes, or 32 bytes of
// fp32 moved by 256-bit accesses); the thread with index g in its group of G
// threads owns vectors v = g + k*G (k < VPT), so every warp-wide load or store
// instruction covers 512 (1024) contiguous bytes.  The
// summed row stays in registers between the sum of squares and the
// normalisation: every input byte is read once.  An NVFP4 block (16
// elements) is the vector pair (2j, 2j+1), held by neighbouring lanes, so the
// block maximum takes one xor-1 shuffle.
//
// In Lamport mode the partials come from the current workspace slot and are
// polled (bounded) until no 32-bit word holds the -0.0f sentinel; the
// retired slot is refilled with the sentinel in the same launch and the block
// that takes the last atomic ticket advances the slot index
// (LamportComm::update without a spin).
#pragma once

#include <stddef.h>

#include "fused_core.cuh"


namespace arf {

// Threads of a one-vector-per-thread row block (one_vec_threads_for).
template <class D>
__host__ __device__ constexpr int one_vec_threads(int rmax)
{
    return one_vec_threads_for(D::bytes, rmax);
}

// Block size bound: one_vec_threads for one vector per thread; wider rows
// (several vectors per thread) and the two-rows-per-SM form at most 512; one
// row per warp: 8 warps.
template <class D, int RMAX, int VPT, bool WARP_ROW, bool LIGHT = false, bool AHEAD = false>
constexpr int rows_max_threads()
{
    return WARP_ROW ? 256 : (LIGHT || AHEAD) ? 512 : (VPT == 1 ? one_vec_threads<D>(RMAX) : 512);
}

// LIGHT, two rows per SM: blocks of <= 512 threads within 64 registers, so
// that two blocks (two rows) share an SM and one row's reductions overlap the
// other's loads.  Two forms (the launcher picks them, see
// launch_fused_rows_t): 16-bit rows of 513..1024 vectors with at most 4
// ranks at two vectors per thread and one vector per load batch, and 16-bit
// rows of 449..512 vectors with 5 ranks at one vector per thread (whose
// unbounded build takes more than 64 registers, one block per SM).
// AHEAD: one vector per thread with 5..8 ranks in blocks of <= 512 threads,
// whose register budget (up to 128) holds the next row's eight rank vectors
// and residual vector: the look-ahead below, otherwise taken only with at
// most 4 ranks.
template <bool LIGHT>
__host__ __device__ constexpr int rows_min_blocks()
{
    return LIGHT ? 2 : 1;
}

// Lamport launches of at most this many blocks (every launch of the one-shot
// token range) take their slot ticket right after reading the slot state
// instead of at the end.
constexpr unsigned kEarlyTicketBlocks = 128;

// s[kk] (+)= rank batch r0..r0+RB-1 of vector g + (k0 + kk) * G; ELEM rounds
// every partial sum to the element type.
template <class D, int KCH, int RB, bool ELEM>
__device__ __forceinline__ void fold_ranks(float (&s)[KCH][8],
                                           const typename D::Vec (&raw)[KCH][RB], int r0,
                                           int R, int g, int k0, int G, int Hv)
{
#pragma unroll
    for (int kk = 0; kk < KCH; ++kk) {
        if (g + (k0 + kk) * G < Hv) {
#pragma unroll
            for (int rr = 0; rr < RB; ++rr) {
                if (r0 + rr < R) {
                    if (r0 + rr == 0) {
                        if (ELEM)
                            elem_start8<D>(s[kk], raw[kk][rr]);
                        else
                            unpack8<D>(raw[kk][rr], s[kk]);
                    } else {
                        if (ELEM)
                            elem_add8<D>(s[kk], raw[kk][rr]);
                        else
                            add8<D>(s[kk], raw[kk][rr]);
                    }
                }
            }
        }
    }
}

// CLUSTER: the kernel is launched with a thread-block cluster and one row
// spans its CTAs (a separate instantiation, so the common one-CTA-per-row
// kernel carries none of the cluster code).
template <class D, int RMAX, int VPT, bool WARP_ROW, bool CLUSTER = false, bool LIGHT = false,
          bool AHEAD = false, bool BUF = false>
__global__ void __launch_bounds__(rows_max_threads<D, RMAX, VPT, WARP_ROW, LIGHT, AHEAD>(),
                                  rows_min_blocks<LIGHT>())
fused_rows_kernel(const FusedArgs a)
{
    using V = typename D::Vec;
    constexpr int EB = D::bytes;           // element bytes
    constexpr int VB = 8 * EB;             // vector bytes
    // partial vectors in flight per thread: 16 x 16 B (bf16 / fp16), 8 x 32 B
    // (fp32; within 128 registers at 512 threads).  fp32 batchings measured
    // at (R, T, H) = (8, 4096, 4096) / (4, 2048, 8192) / (8, 128, 4096):
    // 8 loads of up to 8 ranks 115.3 / 80.8 / 8.3 us, 4 loads of up to 4
    // ranks 124.9 / 93.1 / 9.0 us, 2 loads at 1024 threads 154.3 / 86.0 / 9.2 us.
    constexpr int LOADS = EB == 4 ? 8 : 16;
    // ranks loaded per batch
    constexpr int RBMAX = 8;
    constexpr int RB = RMAX < RBMAX ? RMAX : RBMAX;
    // vectors per batch (one in the two-rows-per-SM form)
    constexpr int KCH = LIGHT ? 1 : ((LOADS / RB) > VPT ? VPT : (LOADS / RB));
    static_assert(!LIGHT || (D::bytes == 2 && !WARP_ROW && !CLUSTER &&
                             ((VPT == 2 && RMAX <= 4) || (VPT == 1 && RMAX == 8))),
                  "two rows per SM: 16-bit; two vectors per thread with at most 4 ranks, "
                  "or one vector per thread with 5..8");
    static_assert(!AHEAD || (D::bytes == 2 && VPT == 1 && RMAX == 8 && !WARP_ROW && !CLUSTER &&
                             !LIGHT),
                  "look-ahead of 5..8 ranks: 16-bit, one vector per thread, <= 512 threads");
    static_assert(!BUF || (VPT <= 2 && !WARP_ROW && !CLUSTER && !LIGHT && !AHEAD),
                  "buffer-mode instantiation: row-block kernels of one or two vectors");
    static_assert(VPT % KCH == 0, "batch must divide VPT");
    static_assert(RMAX % RB == 0, "rank batch must divide RMAX");

    const int H = a.H;
    const int Hv = H >> 3;
    const int R = a.R;
    const int pat = a.pattern;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int G, g, row, row_step;
    if (WARP_ROW) {
        G = 32;
        g = lane;
        row = blockIdx.x * nwarps + warp;
        row_step = gridDim.x * nwarps;
    } else if (!CLUSTER) {
        G = blockDim.x;
        g = threadIdx.x;
        row = blockIdx.x;
        row_step = gridDim.x;
    } else {
        // one row per cluster of C CTAs: CTA `crank` holds vectors
        // [crank * blockDim, (crank + 1) * blockDim)
        G = blockDim.x * cluster_size();
        g = cluster_rank() * blockDim.x + threadIdx.x;
        row = cluster_id();
        row_step = cluster_count();
    }
    const unsigned C = CLUSTER ? cluster_size() : 1u;

    // Lamport mode (run time).  The look-ahead form for 6..8 ranks, the
    // two-rows-per-SM form for <= 4 ranks and the BUF instantiation are
    // launched in buffer mode only and carry no Lamport code (µs without it,
    // T=8192, back-to-back / inputs evicted: R=8, H=4096 109.7 / 116.2 ->
    // 106.0 / 109.7; R=3, H=4104 79.0 / 86.8 -> 71.2 / 79.8; R=2, H=6144
    // 81.4 / 92.3 -> 79.0 / 88.8; R=3, H=5120 83.9 / 90.3 -> 86.4 / 86.5).
    // The two-rows form for 5 ranks keeps it (82.95 / 92.1 -> 85.5 / 95.8
    // without).
#define AR_LAMPORT ((AHEAD || BUF || (LIGHT && VPT == 2)) ? 0 : a.lamport)

    // inputs and the slot state may be written by the preceding grid
    pdl_wait();

    // rank r's row data: a caller pointer (constant-bank parameter, no
    // register copy) or, in Lamport mode, slot + r * plane
    uint32_t flag = 0;
    const uint8_t* slot = nullptr;
    unsigned ticket = 0;
    const size_t plane = (size_t)a.T * H * EB;
    if (AR_LAMPORT) {
        // The slot state's first 32 bytes in one load, once per block
        // (shared through shared memory) or, with one row per warp, once per
        // warp: polling loads bypass L1, and every thread reading the words
        // on its own sent ~6,000 requests for one L2 line at R=8, T=128,
        // H=4096 (Lamport call with PDL 6.25 -> 5.55 us; R=4 5.77 -> 5.05;
        // fp32 8.06 -> 7.48).  For one-row-per-warp blocks the block barrier
        // measured slower than a load per warp (3.69 -> 3.78 us at R=2,
        // T=16, H=512).
        static_assert(offsetof(ar_fusion_state, lamport_flag) == 8 &&
                          offsetof(ar_fusion_state, clear_elem_bytes) == 12 &&
                          offsetof(ar_fusion_state, clear_size) == 24,
                      "state words read by one 32-byte load");
        uint32_t st[3];   // lamport_flag, clear_elem_bytes, clear_size (low, high)
        uint32_t st_hi;
        if (WARP_ROW) {
            const V32 sv = ld_poll32(a.state);   // the state is 256-byte aligned
            st[0] = sv.lo.z;
            st[1] = sv.lo.w;
            st[2] = sv.hi.z;
            st_hi = sv.hi.w;
        } else {
            __shared__ uint32_t st_sh[4];
            if (threadIdx.x == 0) {
                const V32 sv = ld_poll32(a.state);
                st_sh[0] = sv.lo.z;
                st_sh[1] = sv.lo.w;
                st_sh[2] = sv.hi.z;
                st_sh[3] = sv.hi.w;
            }
            __syncthreads();
            st[0] = st_sh[0];
            st[1] = st_sh[1];
            st[2] = st_sh[2];
            st_hi = st_sh[3];
        }
        // Slot ticket.  The last block to take one advances the state at its
        // end; a ticket proves only that its block has read the state, so it
        // is taken here and its latency hides behind the row (Lamport call
        // with PDL, µs: 2 blocks 3.59 -> 3.28, 16 blocks 5.12 -> 4.72, 64
        // blocks 5.23 -> 4.94, 128 blocks (R=8, T=128, H=4096) 5.6 -> 5.2-5.3,
        // R=4 4.55 -> 4.10).  Larger launches (Lamport forced beyond the
        // one-shot token range) take theirs at the end: tickets taken at
        // once queue on one word.
        if (gridDim.x <= kEarlyTicketBlocks) {
            if (WARP_ROW)
                __syncthreads();   // every warp of the block has read the state
            if (threadIdx.x == 0)
                ticket = atomicAdd(&a.state->counter, 1u);
        }
        flag = st[0];
        const uint32_t clear_eb = st[1];
        const uint64_t clear_elems = (uint64_t)st[2] | ((uint64_t)st_hi << 32);
        slot = a.lamport_base + (size_t)(flag % 3u) * a.slot_bytes;
        // refill the retired slot with the sentinel (clear loop of the one-shot
        // kernel) over the bytes its last user wrote: that call's element size,
        // which need not be this call's (never beyond the slot)
        uint8_t* clr = a.lamport_base + (size_t)((flag + 2u) % 3u) * a.slot_bytes;
        uint64_t nvec = clear_elems * clear_eb / 16;
        if (nvec > a.slot_bytes / 16)
            nvec = a.slot_bytes / 16;
        const uint64_t nth = (uint64_t)gridDim.x * blockDim.x;
        const uint4 sent = make_uint4(0x80000000u, 0x80000000u, 0x80000000u, 0x80000000u);
        for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += nth)
            st_vec(clr + i * 16, sent);
    }
#define AR_RANK_PTR(r) (AR_LAMPORT ? slot + (size_t)(r) * plane : a.partial[(r)])

    float qscale = 0.0f;
    if (pat & (AR_QUANT_FP8 | AR_QUANT_NVFP4))
        qscale = *a.scale_factor;

    __shared__ DF red[2][32];
    __shared__ float rstd_sh[2];
    // this CTA's row partial, read by the cluster as one 8-byte load
    // (ld_dsmem_f2): DF alone is only 4-byte aligned
    __shared__ __align__(8) DF part[2];
    int parity = 0;
    float amax_local = 0.0f;

    // One vector per thread, one row per block, at most 4 ranks: the next
    // row's rank vectors and residual vector are loaded into registers as soon
    // as this row's sum is formed, so those loads are in flight through this
    // row's reduction barriers, normalisation and stores.  Measured (us,
    // back-to-back / inputs evicted): R=4, T=2048, H=8192 with FP8 output
    // 45.4 / 54.4 -> 39.9 / 50.3; R=4, T=8192, H=7168 128.7 / 140.1 ->
    // 120.3 / 131.2.  With 8 or 16 ranks the 896-thread blocks have registers
    // for two ranks ahead only, which measured slower (R=8, H=7168: 180 ->
    // 221 us), so those rows load as before; so did two vectors per thread
    // at 512 threads with the same look-ahead (R=4, H=8192: 65.9 us).  Rows
    // of <= 512 vectors with 6..8 ranks take it in the AHEAD instantiation
    // (R=8, T=8192, H=4096: 116.9 -> 109.4 us).  The row then works on
    // `pre` / `pre_x` in place (no register copies).
    constexpr bool PIPE = !WARP_ROW && !CLUSTER && VPT == 1 && (RMAX <= 4 || AHEAD);
    V pre[KCH][RB];
    V pre_x[KCH];
    const auto load_first = [&](int r_) {
#pragma unroll
        for (int kk = 0; kk < KCH; ++kk) {
            const int v = g + kk * G;
            if (v < Hv) {
                const size_t o = (size_t)r_ * H * EB + (size_t)v * VB;
#pragma unroll
                for (int rr = 0; rr < RB; ++rr)
                    if (rr < R)
                        pre[kk][rr] = AR_LAMPORT ? ld_poll_v<D>(AR_RANK_PTR(rr) + o)
                                                : ld_stream_v<D>(AR_RANK_PTR(rr) + o);
                pre_x[kk] = ld_stream_v<D>(a.residual_in + o);
            }
        }
    };
    if (PIPE && row < a.T)
        load_first(row);

    for (; row < a.T; row += row_step) {
        const size_t roff = (size_t)row * H * EB;
        DF2 ss = {};
        V yv[VPT];

        // One-row-per-block, staged or caller partials: while this row is
        // loaded and reduced, have the copy engine pull the block's next row
        // (R partial rows + the residual row) into L2, so that its loads start
        // from L2 instead of exposing DRAM latency at every row boundary.
        // (Measured at R = 8, T = 8192, H = 7168: one row ahead 187.8 us, two
        // 189.8 us, three 200.3 us, none 214.1 us.)
        if (!WARP_ROW && !AR_LAMPORT && threadIdx.x < (unsigned)(R + 1)) {
            const int nrow = row + row_step;
            // this CTA's slice of the row (the whole row without a cluster)
            const size_t off = (size_t)(g - threadIdx.x) * VPT * VB;
            const size_t len = (size_t)blockDim.x * VPT * VB;
            const size_t rowb = (size_t)H * EB;
            if (nrow < a.T && off < rowb) {
                const uint8_t* src = (int)threadIdx.x < R ? AR_RANK_PTR(threadIdx.x) : a.residual_in;
                const size_t n = off + len <= rowb ? len : rowb - off;
                prefetch_l2_bulk(src + (size_t)nrow * rowb + off, (uint32_t)n);
            }
        }

#pragma unroll
        for (int k0 = 0; k0 < VPT; k0 += KCH) {
            float s[KCH][8];
            // with PIPE (one chunk, one rank batch) the row's vectors are
            // already in `pre` / `pre_x`: work on them in place
            V xr_own[KCH];
            V (&xr)[KCH] = PIPE ? pre_x : xr_own;
#pragma unroll
            for (int r0 = 0; r0 < RMAX; r0 += RB) {
                if (r0 >= R)
                    break;
                V raw_own[KCH][RB];
                V (&raw)[KCH][RB] = PIPE ? pre : raw_own;
                // ---- loads of this batch (all in flight together)
#pragma unroll
                for (int kk = 0; kk < KCH; ++kk) {
                    const int v = g + (k0 + kk) * G;
                    if (PIPE) {
                        // loaded by load_first
                    } else if (v < Hv) {
#pragma unroll
                        for (int rr = 0; rr < RB; ++rr)
                            if (r0 + rr < R)
                                raw[kk][rr] = AR_LAMPORT ? ld_poll_v<D>(AR_RANK_PTR(r0 + rr) + roff + (size_t)v * VB)
                                                        : ld_stream_v<D>(AR_RANK_PTR(r0 + rr) + roff + (size_t)v * VB);
                        if (r0 == 0)
                            xr[kk] = ld_stream_v<D>(a.residual_in + roff + (size_t)v * VB);
                    }
                }
                // ---- Lamport: re-poll until no sentinel word is left (bounded)
                if (AR_LAMPORT) {
                    bool pend = false;
#pragma unroll
                    for (int kk = 0; kk < KCH; ++kk)
#pragma unroll
                        for (int rr = 0; rr < RB; ++rr)
                            if (r0 + rr < R && g + (k0 + kk) * G < Hv)
                                pend |= has_sentinel(raw[kk][rr]);
                    if (pend) {
                        const uint64_t t0 = globaltimer_ns();
                        while (true) {
                            pend = false;
                            int first = -1;
#pragma unroll
                            for (int kk = 0; kk < KCH; ++kk) {
                                const int v = g + (k0 + kk) * G;
#pragma unroll
                                for (int rr = 0; rr < RB; ++rr)
                                    if (r0 + rr < R && v < Hv && has_sentinel(raw[kk][rr])) {
                                        raw[kk][rr] = ld_poll_v<D>(AR_RANK_PTR(r0 + rr) + roff + (size_t)v * VB);
                                        if (has_sentinel(raw[kk][rr])) {
                                            pend = true;
                                            if (first < 0)
                                                first = r0 + rr;
                                        }
                                    }
                            }
                            if (!pend)
                                break;
                            if (globaltimer_ns() - t0 > a.timeout_ns) {
                                record_error(a.state, AR_ERR_TIMEOUT, row * 32 + first);
                                break;
                            }
                            __nanosleep(256);
                        }
                    }
                }
                // ---- fold this rank batch into the fp32 sum (rank order); the
                // accumulation choice is taken once, outside the unrolled fold
                if (!a.acc)
                    fold_ranks<D, KCH, RB, false>(s, raw, r0, R, g, k0, G, Hv);
                else
                    fold_ranks<D, KCH, RB, true>(s, raw, r0, R, g, k0, G, Hv);
            }
            // ---- residual add, sum of squares
#pragma unroll
            for (int kk = 0; kk < KCH; ++kk) {
                const int k = k0 + kk;
                const int v = g + k * G;
                if (v < Hv) {
                    if (a.acc)
                        elem_finish8<D>(s[kk]);
                    const V y = residual_vec<D>(s[kk], xr[kk], ss);
                    yv[k] = y;
                    if (pat & AR_RESIDUAL_OUT)
                        st_vec(a.residual_out + roff + (size_t)v * VB, y);
                } else {
                    yv[k] = zero_vec<V>();
                }
            }
        }
        if (PIPE && row + row_step < a.T)
            load_first(row + row_step);

        // ---- sum of squares over the row
        float rstd;
        const DF ssm = df2_merge(ss);
        if (WARP_ROW) {
            rstd = inv_rms(df_warp_sum(ssm), H, a.eps);
        } else if (!CLUSTER) {
            rstd = row_rstd(ssm, red[parity], &rstd_sh[parity], warp, lane, nwarps, H, a.eps,
                            BlockSync{});
            parity ^= 1;
        } else {
            // block partial -> part[parity]; after the cluster barrier every
            // warp reads the C partials (rank order) through distributed
            // shared memory.  Partials alternate by row parity, so one cluster
            // barrier per row suffices (a CTA can only overwrite part[p] two
            // rows later, after every CTA has passed the next barrier).
            const DF sw = df_warp_sum(ssm);
            if (lane == 0)
                red[parity][warp] = sw;
            __syncthreads();
            if (warp == 0) {
                DF v = lane < nwarps ? red[parity][lane] : DF{0.0f, 0.0f};
                v = df_warp_sum(v);
                if (lane == 0)
                    part[parity] = v;
            }
            cluster_barrier();
            DF t = {0.0f, 0.0f};
            if ((unsigned)lane < C) {
                const float2 q = ld_dsmem_f2(&part[parity], (unsigned)lane);
                t = DF{q.x, q.y};
            }
            rstd = inv_rms(df_warp_sum(t), H, a.eps);
            parity ^= 1;
        }

        // ---- normalise, optional outputs (gamma re-read per row: L1-resident)
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = g + k * G;
            float gf[8];
            load_gamma<D>(a.gamma, v, v < Hv, gf);
            normalize_vec<D>(a, pat, row, v, v < Hv, yv[k], gf, rstd, qscale, amax_local);
        }
    }

#undef AR_RANK_PTR

    // no CTA may leave while another CTA of its cluster can still read its
    // row partial
    if (CLUSTER)
        cluster_barrier();
    pdl_trigger();

    if (a.amax_out) {
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1)
            amax_local = fmaxf(amax_local, __shfl_xor_sync(0xffffffffu, amax_local, m));
        if (lane == 0)
            atomicMax(reinterpret_cast<unsigned int*>(a.amax_out), __float_as_uint(amax_local));
    }

    // Slot state: the block holding the last ticket advances it.  Only the next launch
    // reads it, and kernel completion (stream order, or griddepcontrol.wait
    // under programmatic dependent launch) already makes every write of this
    // grid visible there, so no fence is needed (one measured 0.2-0.4 us).
    if (AR_LAMPORT) {
        const bool early = gridDim.x <= kEarlyTicketBlocks;
        if (!early)
            __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned prev = early ? ticket : atomicAdd(&a.state->counter, 1u);
            if (prev == gridDim.x - 1) {
                a.state->lamport_flag = (flag + 1u) % 3u;
                a.state->clear_size = (uint64_t)R * a.T * H;
                a.state->clear_elem_bytes = EB;
                a.state->calls += 1;
                a.state->counter = 0;
            }
        }
    }
#undef AR_LAMPORT
}

}  // namespace arf
