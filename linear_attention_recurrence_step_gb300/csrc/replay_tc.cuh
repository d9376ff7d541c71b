// replay_tc.cuh -- replay of a long accepted prefix as one tensor-core
// contraction (tcgen05.mma, tf32 operands, accumulator in tensor memory).
//
// The replay fold of "metaltile-std gated_delta_replay.rs" (kernel
// state_replay), s <- g_t s + delta_t k_t over the steps t that are accepted
// and unmasked, is linear in the state and does not read the state to form
// its updates, so it closes to
//     s_out = Gam s_in + sum_t w_t delta_t k_t,
//     w_t   = prod of g_x over the folded steps x after t,  Gam = prod of all
// and for every (b, hv) tile the sum is a dense product
//     S_out = Gam S_in + (delta^T diag(w)) K      (Dv x Dk, contraction over T).
// replay_weights_kernel forms w and Gam (a suffix product per tile);
// replay_tc_kernel runs the contraction: tape rows arrive by cp.async in a
// ring several stages ahead, eight warps turn each 16-step stage into
// operand tiles in shared memory (delta scaled by w as A, k rows as B, both
// split into tf32 hi + lo terms, K-major core-matrix layout), one thread
// issues three tcgen05.mma per 8 steps (a_lo b_hi + a_hi b_lo + a_hi b_hi)
// into a 128-lane f32 accumulator in tensor memory, and the commit of each
// stage to an mbarrier frees its operand buffer for the stage after next.  Long calls split the steps over several CTAs per tile; their
// partial sums are added in a fixed order by replay_reduce_kernel, so
// results are run-to-run deterministic.
//
// Rows of the tile beyond Dv and steps that are not folded enter as exact
// zeros (never loaded), so whatever unused tape slots hold cannot reach the
// state.  Every wait on an mbarrier is bounded (about a second of clock);
// on expiry the CTA writes NaN to its outputs instead of hanging, raises the
// library's wait-expiry flag (gdn_wait_status), releases its tensor memory
// and exits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tile.cuh"

namespace gdn {

constexpr int kTcRows = 128;       // accumulator lanes = state rows per CTA
constexpr int kTcThreads = 256;    // eight warps: two per 32 tensor-memory lanes
constexpr int kTcSteps = 16;       // steps staged per pipeline stage
constexpr int kTcWeightsThreads = 1024;
constexpr long long kTcWaitCycles = 2000000000ll;  // default bound on an mbarrier wait (~1 s)

__host__ __device__ constexpr int tc_cols(int dk) {  // tensor-memory columns to allocate
    return dk <= 32 ? 32 : dk <= 64 ? 64 : dk <= 128 ? 128 : 256;
}

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ unsigned smem_addr(const void *p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of
// 8 rows x 16 bytes, `lbo` bytes apart along K and `sbo` bytes apart along
// M / N (bits 46-48 hold the descriptor version 1).
__device__ __forceinline__ uint64_t tc_desc(unsigned addr, unsigned lbo, unsigned sbo) {
    return (uint64_t)((addr >> 4) & 0x3fffu) | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::tf32: f32 accumulator, tf32 A and B, both
// K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t tc_idesc_tf32(int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcRows >> 4) << 24);
}
__device__ __forceinline__ void tc_mma_tf32(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(da), "l"(db), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void tc_commit(unsigned mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
                 : "memory");
}
// Bounded wait for phase `parity` of an mbarrier; false when the bound expired.
__device__ __forceinline__ bool mbar_wait(unsigned mbar, unsigned parity, long long bound = kTcWaitCycles) {
    uint32_t done = 0;
    const long long t0 = clock64();
    while (!done) {
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(mbar), "r"(parity)
            : "memory");
        if (!done && clock64() - t0 > bound) return false;
    }
    return true;
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
        "[%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]);
}
// x ~ hi + lo: the tensor core reads an f32 operand as tf32 by dropping its
// 13 low mantissa bits (truncation, checked on the GPU for kind::tf32), so hi
// is x itself and lo = x - trunc(x) (exact in f32, below 2^-10 |x|).
__device__ __forceinline__ void tc_split(float x, float &hi, float &lo) {
    hi = x;
    lo = x - __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

// ------------------------------------------------------------ decay weights
// One CTA per (b, hv): w_t (0 for steps that are not folded) and Gam.  Each
// thread takes a segment of consecutive steps; the exclusive suffix products
// of the segment products come from a block-wide scan (warp shuffles, then
// one warp over the warps' totals), so no thread walks the segments in turn.
template <typename TIn>
__global__ void __launch_bounds__(kTcWeightsThreads) replay_weights_kernel(const ReplayTcArgs a) {
    pdl_trigger();
    pdl_wait();
    constexpr int NW = kTcWeightsThreads / 32;
    __shared__ float wtot[NW];  // each warp's product, then the product of the warps after it
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t n = blockIdx.x;
    const int64_t b = n / a.Hv, hv = n - b * a.Hv;
    int64_t steps = a.steps;
    if (a.acc_b) {
        const int64_t ab = (int64_t)a.acc_b[b];
        steps = ab < 0 ? 0 : (ab < steps ? ab : steps);
    }
    const TIn *glp = static_cast<const TIn *>(a.g_log);
    const int64_t L = (a.T + kTcWeightsThreads - 1) / kTcWeightsThreads;
    const int64_t s0 = tid * L, s1 = min(a.T, s0 + L);
    // the decay of step t, 1 when t is not folded (loads depend on indices only)
    auto gfold = [&](int64_t t) {
        const float gv = ld_f32(glp + (b * a.T + t) * a.Hv + hv);
        const bool on = t < steps && (!a.mask || a.mask[b * a.T + t] != 0u);
        return on ? gv : 1.f;
    };
    // Up to kWCache steps per thread (T <= kWCache * threads) stay in
    // registers between the two passes, loaded all at once; longer tapes walk
    // the steps and load them again in the second pass.  The products are
    // taken in the same order either way.
    constexpr int kWCache = 8;
    const bool cached = L <= kWCache;
    float gc[kWCache];
    unsigned onm = 0u;
    float p = 1.f;
    if (cached) {
#pragma unroll
        for (int i = 0; i < kWCache; ++i) {
            const int64_t t = s0 + i;
            const bool in = t < s1;
            const float gv = in ? ld_f32(glp + (b * a.T + t) * a.Hv + hv) : 1.f;
            const bool on = in && t < steps && (!a.mask || a.mask[b * a.T + t] != 0u);
            gc[i] = on ? gv : 1.f;
            onm |= on ? 1u << i : 0u;
        }
#pragma unroll
        for (int i = 0; i < kWCache; ++i) p *= gc[i];
    } else {
        for (int64_t t = s0; t < s1; ++t) p *= gfold(t);
    }
    // inclusive suffix product over the lanes of the warp: lanes lane..31
    float inc = p;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_down_sync(0xffffffffu, inc, o);
        if (lane + o < 32) inc *= x;
    }
    float exc = __shfl_down_sync(0xffffffffu, inc, 1);  // lanes lane+1..31
    if (lane == 31) exc = 1.f;
    if (lane == 0) wtot[warp] = inc;
    __syncthreads();
    if (warp == 0) {  // the same over the warps' products
        const float v = lane < NW ? wtot[lane] : 1.f;
        float winc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float x = __shfl_down_sync(0xffffffffu, winc, o);
            if (lane + o < 32) winc *= x;
        }
        float wexc = __shfl_down_sync(0xffffffffu, winc, 1);
        if (lane == 31) wexc = 1.f;
        __syncwarp();
        if (lane < NW) wtot[lane] = wexc;
        if (lane == 0) a.gam[n] = winc;
    }
    __syncthreads();
    float run = exc * wtot[warp];
    float *w = a.w + n * a.T;
    if (cached) {
#pragma unroll
        for (int i = kWCache - 1; i >= 0; --i) {
            const int64_t t = s0 + i;
            if (t < s1) {
                const bool on = (onm >> i) & 1u;
                w[t] = on ? run : 0.f;
                run = on ? run * gc[i] : run;
            }
        }
    } else {
        for (int64_t t = s1 - 1; t >= s0; --t) {
            const bool on = t < steps && (!a.mask || a.mask[b * a.T + t] != 0u);
            const float gv = ld_f32(glp + (b * a.T + t) * a.Hv + hv);
            w[t] = on ? run : 0.f;
            run = on ? run * gv : run;
        }
    }
}

// ------------------------------------------------------------ the contraction
// Steps per pipeline stage, and the depth of the raw ring of cp.async copies
// (stages in flight ahead of the fill).  Up to Dk = 128 two stages keep a
// CTA under half of an SM's shared memory, so two CTAs (sixteen filling
// warps) share an SM: measured 26 % faster on a 4096-step replay than six
// stages at one CTA per SM.  Larger Dk fit one CTA per SM either way.
__host__ __device__ constexpr int tc_kb(int dk) { return kTcSteps; }
__host__ __device__ constexpr int tc_raw_depth(int dk) { return dk <= 128 ? 2 : 4; }
// CTAs per SM the shared-memory budget admits (the split plan aims at this
// many per SM of a 128-SM reference count, independent of the device).
__host__ __device__ constexpr int tc_ctas_per_sm(int dk) { return dk <= 128 ? 2 : 1; }
constexpr int kTcRawPitch = kTcRows + 8;  // elements per staged delta row (bank spread)
__host__ __device__ constexpr int tc_kpitch(int dk) { return dk + 8; }  // per staged k row
// Raw tape rows of one stage as the cp.async copies land them (element type).
__host__ __device__ constexpr size_t tc_raw_bytes(int dk, int esize) {
    return align16((size_t)tc_kb(dk) * kTcRawPitch * esize) + align16((size_t)tc_kb(dk) * tc_kpitch(dk) * esize);
}
__host__ __device__ constexpr size_t tc_canon_bytes(int dk) {
    return (size_t)2 * kTcRows * tc_kb(dk) * 4 + (size_t)2 * dk * tc_kb(dk) * 4;
}
__host__ __device__ constexpr size_t replay_tc_smem_bytes2(int dk, int esize, bool staged) {
    return 2 * tc_canon_bytes(dk) + (staged ? tc_raw_depth(dk) * tc_raw_bytes(dk, esize) : 0) + 128;
}

// STAGED: the tape rows of each stage arrive by cp.async (16-byte pieces from
// every thread, RD stages ahead of the fill) into a raw ring in shared
// memory, and the fill reads them there; the other form loads them from
// global memory in the fill (any alignment).
template <typename TIn, int DK, bool STAGED>
__global__ void __launch_bounds__(kTcThreads, tc_ctas_per_sm(DK)) replay_tc_kernel(const ReplayTcArgs a) {
    constexpr int KB = tc_kb(DK);
    constexpr int NKQ = KB / 4;               // core matrices along the steps
    constexpr size_t CANON = tc_canon_bytes(DK);
    constexpr size_t RAW = tc_raw_bytes(DK, (int)sizeof(TIn));
    constexpr unsigned SBO = NKQ * 128;       // bytes between 8-row core-matrix groups
    constexpr unsigned A_BYTES = kTcRows * KB * 4, B_BYTES = DK * KB * 4;
    constexpr int NCOL = tc_cols(DK);
    constexpr int DP = kTcRawPitch, KP = tc_kpitch(DK);
    constexpr int RD = tc_raw_depth(DK);
    // bf16 / f16 k rows are exact in tf32: their low operand tile would be
    // zero, so it is neither filled nor multiplied
    constexpr bool kBExact = !std::is_same<TIn, float>::value;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *raw0 = smem + 2 * CANON;
    unsigned char *tail = raw0 + (STAGED ? RD * RAW : 0);
    uint64_t *mbar_mma = reinterpret_cast<uint64_t *>(tail);        // [2]
    uint32_t *taddr_s = reinterpret_cast<uint32_t *>(tail + 16);
    uint64_t *mbar_never = reinterpret_cast<uint64_t *>(tail + 24);  // never completed (testing hook)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t tiles_rb = a.B * a.Hv * a.row_blocks;
    const int split = (int)(blockIdx.x / tiles_rb);
    const int64_t item = blockIdx.x - (int64_t)split * tiles_rb;
    const int64_t n = item / a.row_blocks, rb = item - n * a.row_blocks;
    const int64_t b = n / a.Hv, hv = n - b * a.Hv;
    const int64_t row0 = rb * kTcRows;
    const int rows = (int)min((int64_t)kTcRows, a.Dv - row0);
    const int64_t t_begin = (int64_t)split * a.split_steps;
    const int64_t t_end = min(a.T, t_begin + a.split_steps);
    const int nstages = t_end > t_begin ? (int)((t_end - t_begin + KB - 1) / KB) : 0;
    const TIn *dlp = static_cast<const TIn *>(a.delta_log);
    const TIn *klp = static_cast<const TIn *>(a.k_log);
    const float *wn = a.w + n * a.T;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(taddr_s)),
                     "r"(NCOL));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_addr(&mbar_mma[i])));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_addr(mbar_never)));
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    const uint32_t tmem = *taddr_s;
    pdl_trigger();
    pdl_wait();
    const uint32_t idesc = tc_idesc_tf32(DK);

    // cp.async (16-byte pieces, every thread) of stage s's tape rows into raw
    // slot s % RD, one commit group per stage (empty past the end)
    constexpr int VEC = 16 / (int)sizeof(TIn);
    const int dpr = rows / VEC;  // 16-byte pieces per staged delta row
    auto issue_raw = [&](int s) {
        if (STAGED && s < nstages) {
            const int64_t ts = t_begin + (int64_t)s * KB;
            const int cnt = (int)min((int64_t)KB, t_end - ts);
            TIn *rD = reinterpret_cast<TIn *>(raw0 + (s % RD) * RAW);
            TIn *rK = reinterpret_cast<TIn *>(raw0 + (s % RD) * RAW + align16((size_t)KB * DP * sizeof(TIn)));
            for (int i = tid; i < cnt * dpr; i += kTcThreads) {
                const int tt = i / dpr, x = (i - tt * dpr) * VEC;
                cp_async16(rD + tt * DP + x, dlp + ((b * a.T + ts + tt) * a.Hv + hv) * a.Dv + row0 + x);
            }
#pragma unroll 4
            for (int i = tid; i < cnt * (DK / VEC); i += kTcThreads) {
                const int tt = i / (DK / VEC), x = (i - tt * (DK / VEC)) * VEC;
                cp_async16(rK + tt * KP + x, klp + ((b * a.T + ts + tt) * a.Hv + hv) * DK + x);
            }
        }
        if (STAGED) cp_async_commit();
    };
    for (int s = 0; s < RD; ++s) issue_raw(s);
    if (STAGED) cp_async_wait_group<RD - 1>();  // stage 0 landed (this thread's pieces)
    __syncthreads();

    // testing hook (gdn_inject_wait_expiry): one wait that nothing completes,
    // so the pipeline's bound runs out deterministically
    bool ok = !a.inject_expiry || mbar_wait(smem_addr(mbar_never), 0u, a.wait_cycles);
    int last_issued = nstages - 1;  // last stage whose MMAs were issued (-1: none)
    // one core matrix (8 rows x 4 steps) per warp instruction: lane -> (row % 8, step % 4)
    const int cr = lane >> 2, cs = lane & 3;
    // warp w fills core matrices cm = w + 8 j: step quad w % 4, row / column
    // group 2 j + w / 4 -- one step per lane per stage
    const int kq = warp & 3, gq = warp >> 2;
    // the decay weight of this lane's step, from a register ring filled four
    // stages ahead (a global load the fill depends on: issued in its own
    // stage it would stall every stage for a round trip; the ring's register
    // moves still tie each load to the stage after the one that issued it)
    auto weight_of = [&](int s) {
        const int64_t t = t_begin + (int64_t)s * KB + 4 * kq + cs;
        return s < nstages && t < t_end ? wn[t] : 0.f;
    };
    float wq0 = weight_of(0), wq1 = weight_of(1), wq2 = weight_of(2), wq3 = weight_of(3);
    for (int s = 0; s < nstages; ++s) {
        unsigned char *buf = smem + (s & 1) * CANON;
        float *Ah = reinterpret_cast<float *>(buf);
        float *Al = reinterpret_cast<float *>(buf + A_BYTES);
        float *Bh = reinterpret_cast<float *>(buf + 2 * A_BYTES);
        float *Bl = reinterpret_cast<float *>(buf + 2 * A_BYTES + B_BYTES);
        const int64_t ts = t_begin + (int64_t)s * KB;
        const int64_t tq0 = ts + 4 * kq + cs;
        const float w0 = wq0;
        wq0 = wq1;
        wq1 = wq2;
        wq2 = wq3;
        wq3 = weight_of(s + 4);
        if (s >= 2) ok = mbar_wait(smem_addr(&mbar_mma[s & 1]), ((s - 2) >> 1) & 1, a.wait_cycles) && ok;  // buffer free
        const TIn *rD = reinterpret_cast<const TIn *>(raw0 + (s % RD) * RAW);
        const TIn *rK = reinterpret_cast<const TIn *>(raw0 + (s % RD) * RAW + align16((size_t)KB * DP * sizeof(TIn)));
        // Loads first (all independent), then the tf32 splits and the stores:
        // the staged values and the operand tiles live in the same shared
        // memory, so interleaving them would order every load after the
        // previous store.
        constexpr int NA = kTcRows / 16, NB = DK / 16;  // core matrices per lane
        float av[NA], bv[NB];
#pragma unroll
        for (int j = 0; j < NA; ++j) {  // A: delta rows scaled by w (row = lane of D, k = step)
            const int r = 8 * (2 * j + gq) + cr;
            float d = 0.f;
            if (tq0 < t_end && r < rows)
                d = STAGED ? Elem<TIn>::to_f32(rD[(4 * kq + cs) * DP + r])
                         : ld_f32(dlp + ((b * a.T + tq0) * a.Hv + hv) * a.Dv + row0 + r);
            av[j] = d;
        }
#pragma unroll
        for (int j = 0; j < NB; ++j) {  // B: k rows (n = state column, k = step)
            const int c = 8 * (2 * j + gq) + cr;
            float kv = 0.f;
            if (tq0 < t_end)
                kv = STAGED ? Elem<TIn>::to_f32(rK[(4 * kq + cs) * KP + c])
                          : ld_f32(klp + ((b * a.T + tq0) * a.Hv + hv) * DK + c);
            bv[j] = kv;
        }
#pragma unroll
        for (int j = 0; j < NA; ++j) {
            float hi, lo;
            tc_split(w0 != 0.f ? w0 * av[j] : 0.f, hi, lo);
            const int off = ((2 * j + gq) * SBO + kq * 128 + cr * 16 + cs * 4) / 4;
            Ah[off] = hi;
            Al[off] = lo;
        }
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const int off = ((2 * j + gq) * SBO + kq * 128 + cr * 16 + cs * 4) / 4;
            if constexpr (kBExact) {
                Bh[off] = w0 != 0.f ? bv[j] : 0.f;
            } else {
                float hi, lo;
                tc_split(w0 != 0.f ? bv[j] : 0.f, hi, lo);
                Bh[off] = hi;
                Bl[off] = lo;
            }
        }
        if (STAGED) cp_async_wait_group<RD - 2>();  // stage s+1 landed (this thread's pieces)
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        ok = __syncthreads_and(ok);  // stage filled, stage s+1 staged (every wait succeeded)
        if (!ok) {
            last_issued = s - 1;
            break;
        }
        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
            const unsigned ah = smem_addr(Ah), al = smem_addr(Al), bh = smem_addr(Bh), bl = smem_addr(Bl);
#pragma unroll
            for (int k8 = 0; k8 < KB / 8; ++k8) {
                const unsigned koff = k8 * 256;  // two core matrices along K per MMA
                const uint32_t acc0 = (s > 0 || k8 > 0) ? 1u : 0u;
                tc_mma_tf32(tmem, tc_desc(al + koff, 128, SBO), tc_desc(bh + koff, 128, SBO), idesc, acc0);
                if constexpr (!kBExact)
                    tc_mma_tf32(tmem, tc_desc(ah + koff, 128, SBO), tc_desc(bl + koff, 128, SBO), idesc, 1u);
                tc_mma_tf32(tmem, tc_desc(ah + koff, 128, SBO), tc_desc(bh + koff, 128, SBO), idesc, 1u);
            }
            tc_commit(smem_addr(&mbar_mma[s & 1]));
        }
        issue_raw(s + RD);  // raw slot s % RD was consumed before the barrier
    }
    if (last_issued >= 0) {
        // the drain: always up to the default bound, so that no product is in
        // flight when tensor memory is released
        const bool done = mbar_wait(smem_addr(&mbar_mma[last_issued & 1]), (last_issued >> 1) & 1);
        ok = ok && done;
    }
    if (!ok && tid == 0) atomicExch(a.wait_flag, 1u);
    if (STAGED) cp_async_wait_all();  // no copy outlives the CTA
    ok = __syncthreads_and(ok);
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");

    // epilogue: warp w reads accumulator lanes 32 (w % 4) .. + 31 (its state
    // rows) and the columns of half w / 4
    const int64_t row = row0 + 32 * (warp & 3) + lane;
    const int c_begin = (warp >> 2) * (DK / 2), c_end = c_begin + DK / 2;
    const bool live = row < a.Dv;
    const bool direct = a.partial == nullptr;
    float *dst = direct ? a.state_out + (n * a.Dv + row) * DK
                        : a.partial + (((int64_t)split * a.B * a.Hv + n) * a.Dv + row) * DK;
    const float gam = a.gam[n];
#pragma unroll 1
    for (int c0 = c_begin; c0 < c_end; c0 += 16) {
        float v[16];
        if (ok && last_issued >= 0) {
            tc_ld16(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)c0, v);
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = ok ? 0.f : __int_as_float(0x7fc00000);
        }
        if (live) {
            if (direct) {
                const float4 *si = reinterpret_cast<const float4 *>(a.state_in + (n * a.Dv + row) * DK + c0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 x = __ldcs(si + q);
                    v[4 * q + 0] = fmaf(gam, x.x, v[4 * q + 0]);
                    v[4 * q + 1] = fmaf(gam, x.y, v[4 * q + 1]);
                    v[4 * q + 2] = fmaf(gam, x.z, v[4 * q + 2]);
                    v[4 * q + 3] = fmaf(gam, x.w, v[4 * q + 3]);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                __stcs(reinterpret_cast<float4 *>(dst + c0) + q,
                       make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(NCOL));
}

// S_out = Gam S_in + the partial sums of the step splits, in split order.
__global__ void __launch_bounds__(256) replay_reduce_kernel(const ReplayTcArgs a, int dk) {
    pdl_trigger();
    pdl_wait();
    const int64_t per_tile = a.Dv * dk / 4;  // float4 per tile
    const int64_t total = a.B * a.Hv * per_tile;
    const int64_t plane = a.B * a.Hv * a.Dv * dk / 4;
    const float4 *si = reinterpret_cast<const float4 *>(a.state_in);
    const float4 *pp = reinterpret_cast<const float4 *>(a.partial);
    float4 *so = reinterpret_cast<float4 *>(a.state_out);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float gam = a.gam[i / per_tile];
        const float4 x = __ldcs(si + i);
        // the first eight partials are loaded before any is added (one
        // round trip instead of one per split); the sum keeps split order
        constexpr int kBatch = 8;
        float4 pb[kBatch];
#pragma unroll
        for (int s = 0; s < kBatch; ++s)
            if (s < a.splits) pb[s] = __ldcs(pp + s * plane + i);
        float4 r = make_float4(gam * x.x, gam * x.y, gam * x.z, gam * x.w);
#pragma unroll
        for (int s = 0; s < kBatch; ++s)
            if (s < a.splits) {
                r.x += pb[s].x;
                r.y += pb[s].y;
                r.z += pb[s].z;
                r.w += pb[s].w;
            }
        for (int s = kBatch; s < a.splits; ++s) {
            const float4 p = __ldcs(pp + s * plane + i);
            r.x += p.x;
            r.y += p.y;
            r.z += p.z;
            r.w += p.w;
        }
        __stcs(so + i, r);
    }
}

template <typename TIn, int DK>
cudaError_t launch_replay_tc_dk(const ReplayTcArgs &a, cudaStream_t st, int sm_count) {
    auto kern = a.staged ? replay_tc_kernel<TIn, DK, true> : replay_tc_kernel<TIn, DK, false>;
    const size_t sm = replay_tc_smem_bytes2(DK, (int)sizeof(TIn), a.staged);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    e = launch_dependent(replay_weights_kernel<TIn>, (unsigned)(a.B * a.Hv), kTcWeightsThreads, 0, st, a);
    if (e != cudaSuccess) return e;
    e = launch_dependent(kern, (unsigned)(a.splits * a.B * a.Hv * a.row_blocks), kTcThreads, sm, st, a);
    if (e != cudaSuccess || a.partial == nullptr) return e;
    const int64_t total = a.B * a.Hv * a.Dv * DK / 4;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, (int64_t)8 * (sm_count > 0 ? sm_count : 1));
    return launch_dependent(replay_reduce_kernel, (unsigned)blocks, 256, 0, st, a, DK);
}

template <typename TIn>
cudaError_t launch_replay_tc_type(int dk, const ReplayTcArgs &a, cudaStream_t st, int sms) {
    switch (dk) {
    case 32: return launch_replay_tc_dk<TIn, 32>(a, st, sms);
    case 64: return launch_replay_tc_dk<TIn, 64>(a, st, sms);
    case 128: return launch_replay_tc_dk<TIn, 128>(a, st, sms);
    case 192: return launch_replay_tc_dk<TIn, 192>(a, st, sms);
    case 256: return launch_replay_tc_dk<TIn, 256>(a, st, sms);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn
