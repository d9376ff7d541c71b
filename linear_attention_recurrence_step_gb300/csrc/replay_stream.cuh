// replay_stream.cuh -- the replay fold for calls of at most 16 steps with
// Dk = 128 (the decode, speculative-verify and rollback shapes), as a
// persistent stream of 64-row state blocks fed by TMA.
//
// The fold is the one of replay.cuh ("metaltile-std gated_delta_replay.rs",
// kernel state_replay): over the accepted, unmasked steps t,
//     s <- g_t s + delta_t k_t
// with the same scaled state s = G s^, the same scale schedule and the same
// f32 operations in the same order, so a float32 tape still replays the
// record kernel's state_out bit for bit.  What changes is how the work
// reaches the SM.  The short calls are a single pass over the state, and a
// grid of one CTA per 64-row block pays for a launch ramp and a last partial
// wave that are a large part of a pass; here one CTA per SM walks a stream
// of blocks, a fixed first share and then blocks claimed from a per-launch
// counter (so CTAs on faster SMs take more):
//   * a producer warp loads, for each block, its 64 state rows (one 32 KB
//     TMA box) and the k_log and delta_log rows of the call's steps (one box
//     each, as many steps as the call folds) into a ring of stages completing
//     on mbarriers, and runs the block's scale schedule into the stage;
//   * two groups of four compute warps take alternate blocks: each thread
//     reads its 64 state entries from the stage (a half-warp reads 256
//     contiguous bytes of one row, so no bank conflicts), folds the steps in
//     registers, releases the stage and writes its rows with streaming stores
//     while the next blocks arrive.
// Three copies per block: many small copies (one box per step) measured
// 30 % slower, the TMA unit's per-copy cost setting the pace.
// The register layout of a thread is the FP32 replay's (TileLayout<128, 16,
// 8>: 16 lanes per row group, 8 rows per thread).
//
// Every mbarrier wait is bounded.  A compute warp whose wait runs out writes
// NaN to its rows of that block and of all its later blocks; a producer whose
// wait runs out stops issuing, writes NaN to the blocks it claimed but did
// not issue and to every block still unclaimed, and waits for the copies it
// has in flight; both raise the library's wait-expiry flag.
#pragma once

#include "launch.h"
#include "tile.cuh"
#include "tma.cuh"

namespace gdn {

constexpr int kRsRows = 64;        // state rows per block (four warps of 16 rows)
constexpr int kRsDk = 128;
constexpr int kRsSteps = 16;       // most steps a call may fold
constexpr int kRsGroups = 2;       // compute groups per CTA
constexpr int kRsThreads = 32 * (4 * kRsGroups + 1);  // + the producer warp
constexpr int kRsBatch = 4;        // blocks the producer claims, and gathers the scalars of, at once
constexpr long long kRsDrainCycles = 2000000000ll;    // bound on the drain after a failure (~1 s)
constexpr int kRsSchedSlots = 256;  // per-launch block counters, used round robin
constexpr uint32_t kRsEnd = 0xffffffffu;  // block index meaning "no block"
using RsLayout = TileLayout<kRsDk, 16, 8>;

struct ReplayStreamArgs {
    ReplayArgs a;           // row_blocks counts 64-row blocks
    int64_t nblocks;        // B * Hv * row_blocks
    int box_steps;          // steps per k_log / delta_log box: min(steps, 16), at least 1
    unsigned *wait_flag;    // set to 1 when a bounded wait runs out
    long long wait_cycles;  // bound on the ring's waits
    int inject_expiry;      // testing hook: each compute group waits once on a barrier nothing completes
    unsigned *sched;        // this launch's counters: [0] next block to hand out, [1] CTAs finished
};

// One ring stage (bytes from its 1024-byte aligned start).
template <typename TIn>
struct RsStage {
    static constexpr int ES = (int)sizeof(TIn);
    static constexpr int STATE = kRsRows * kRsDk * 4;         // the block's state rows [64][128] f32
    static constexpr int OFF_K = STATE;                       // k_log rows [16][128]
    static constexpr int OFF_D = OFF_K + kRsSteps * kRsDk * ES;  // delta_log rows [16][64]
    static constexpr int OFF_SC = OFF_D + kRsSteps * kRsRows * ES;  // StepScalars[16]
    static constexpr int OFF_INFO = OFF_SC + kRsSteps * (int)sizeof(StepScalars);  // active bits, direct bits, final scale
    static constexpr int BYTES = (OFF_INFO + 16 + 1023) / 1024 * 1024;
    static constexpr int NSG = 2;                             // stages per compute group
    static constexpr int NS = kRsGroups * NSG;                // stages in all
    static constexpr int OFF_BATCH = NS * BYTES;              // the producer's gathered scalars
    static constexpr int OFF_BAR = OFF_BATCH + kRsBatch * kRsSteps * 8 + kRsBatch * 8;
    static constexpr size_t SMEM = 1024 + (size_t)OFF_BAR + (size_t)(2 * NS + 1) * 8;
    static constexpr uint32_t STEP_TX = (uint32_t)((kRsDk + kRsRows) * ES);  // k and delta rows of one step
    static_assert(OFF_D % 16 == 0 && OFF_SC % 16 == 0, "TMA destinations must be 16-byte aligned");
};

// Exact widening of 4 / 8 consecutive tape entries of type T held in shared memory.
template <typename T>
__device__ __forceinline__ float4 rs_widen4(const T *p);
template <>
__device__ __forceinline__ float4 rs_widen4<float>(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
template <>
__device__ __forceinline__ float4 rs_widen4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 r = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u), __uint_as_float(r.y << 16),
                       __uint_as_float(r.y & 0xffff0000u));
}
template <>
__device__ __forceinline__ float4 rs_widen4<__half>(const __half *p) {
    const uint2 r = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

template <typename TIn>
__global__ void __launch_bounds__(kRsThreads, 1)
replay_stream_kernel(const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_d, const ReplayStreamArgs ra) {
    using St = RsStage<TIn>;
    using Lay = RsLayout;
    constexpr int NS = St::NS, NSG = St::NSG;
    const ReplayArgs &a = ra.a;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (sh_addr(smem_raw) & 1023u)) & 1023u);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar0 = sh_addr(smem + St::OFF_BAR);
    auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(NS + s); };
    const uint32_t never = bar0 + 8u * (uint32_t)(2 * NS);
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full(s), 2);   // the producer's expect-tx arrival and its schedule arrival
            mbar_init(empty(s), 4);  // the four warps of the consuming group
        }
        mbar_init(never, 1);
        mbar_init_fence();
    }
    __syncthreads();
    pdl_trigger();
    pdl_wait();

    // Blocks are handed out by this launch's counter in global memory (after
    // a fixed first share, below): the producer claims them kRsBatch at a
    // time, two batches ahead of their use, so CTAs on faster SMs take more
    // blocks and all of them finish within about a batch of one another.
    // The CTA's k-th block goes to compute group k % kRsGroups as that
    // group's i-th block (i = k / kRsGroups), through the group's own stages:
    // stage (group, i % NSG), its (i / NSG)-th use.  Each barrier thus has a single consumer that waits
    // for its phases in order, so no waiter can see a phase of parity p still
    // pending from an earlier use and take it for the one it waits for.  The
    // block index travels in the stage's info words; kRsEnd there tells a
    // group that no block follows.  Block indices fit 32 bits (checked at
    // launch), so the per-block index arithmetic divides in 32 bits.
    const uint32_t nblocks = (uint32_t)ra.nblocks;
    const uint32_t rb32 = (uint32_t)a.row_blocks, hv32 = (uint32_t)a.Hv;
    auto stage_of = [&](int k) { return (k % kRsGroups) * NSG + (k / kRsGroups) % NSG; };
    auto use_of = [&](int k) { return (k / kRsGroups) / NSG; };  // earlier uses of the block's stage
    auto coords = [&](uint32_t u, uint32_t &n, uint32_t &b, uint32_t &hv, uint32_t &row0) {
        n = u / rb32;
        row0 = (u - n * rb32) * kRsRows;
        b = n / hv32;
        hv = n - b * hv32;
    };
    const long long bound = ra.wait_cycles;
    float *sout = static_cast<float *>(a.state_out);
    // The CTA's first two batches are fixed (blocks blockIdx.x + i gridDim.x,
    // i < 2 kRsBatch, as in a static schedule), so no claim delays the first
    // copies; the counter hands out the blocks after those.  When the fixed
    // batches cover every block (short calls) the counter is not used and
    // each group knows its block count: no end markers either.
    const uint32_t dyn0 = 2u * (uint32_t)kRsBatch * gridDim.x;
    const bool dynamic = dyn0 < nblocks;
    const int nfixed = blockIdx.x < nblocks ? (int)((nblocks - 1 - blockIdx.x) / gridDim.x) + 1 : 0;

    if (warp == 4 * kRsGroups) {
        // ==================================================== producer warp
        const TIn *glp = static_cast<const TIn *>(a.g_log);
        // Per-block scalars -- the accepted count of the block's sequence and,
        // per step, the mask word and g -- are gathered a batch ahead: their
        // loads are issued when the batch before starts and their registers
        // are only read (into the shared buffer) when their own batch starts,
        // so their latency under load never stalls the producer.  The claims
        // run one batch further ahead, for the same reason.
        constexpr int NB = kRsBatch;
        constexpr int PER = NB * kRsSteps / 32;  // (block, step) pairs per lane
        static_assert(PER >= 1 && NB <= 32, "a batch is a whole number of (block, step) pairs per lane");
        float *sb_g = reinterpret_cast<float *>(smem + St::OFF_BATCH);  // [NB][16]
        uint32_t *sb_m = reinterpret_cast<uint32_t *>(sb_g + NB * kRsSteps);  // [NB][16]
        int32_t *sb_acc = reinterpret_cast<int32_t *>(sb_m + NB * kRsSteps);  // [NB]
        uint32_t *sb_id = reinterpret_cast<uint32_t *>(sb_acc + NB);  // [NB]
        TIn r_g[PER];
        uint32_t r_m[PER];
        int32_t r_acc = 0;
        uint32_t r_id = kRsEnd;    // lanes 0 .. NB-1: the blocks of the batch being gathered
        uint32_t r_next = kRsEnd;  // lane 0: the counter's answer for the batch after it
        auto claim = [&]() {  // NB consecutive blocks (read only at the next batch)
            if (dynamic && lane == 0) r_next = atomicAdd(ra.sched, (unsigned)NB);
        };
        auto take_claims = [&](int bi) {  // batch bi's blocks, in order (past the last block: kRsEnd)
            uint32_t id = kRsEnd;
            if (bi < 2)
                id = blockIdx.x + (uint32_t)(bi * NB + lane) * gridDim.x;
            else if (dynamic)
                id = dyn0 + __shfl_sync(0xffffffffu, r_next, 0) + (uint32_t)lane;
            r_id = lane < NB && id < nblocks ? id : kRsEnd;
        };
        auto gather = [&]() {  // issue the scalar loads of the blocks in r_id
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int pi = lane + 32 * i;
                const uint32_t u = __shfl_sync(0xffffffffu, r_id, pi >> 4);
                const int tt = pi & 15;
                r_g[i] = Elem<TIn>::from_f32(1.f);
                r_m[i] = 1u;
                if (u != kRsEnd && tt < a.steps) {
                    uint32_t n, b, hv, row0;
                    coords(u, n, b, hv, row0);
                    const int64_t bt = (int64_t)b * a.T + tt;
                    if (a.mask) r_m[i] = __ldg(a.mask + bt);
                    r_g[i] = glp[bt * a.Hv + hv];
                }
            }
            r_acc = (int32_t)a.steps;
            if (lane < NB && r_id != kRsEnd && a.acc_b) {
                uint32_t n, b, hv, row0;
                coords(r_id, n, b, hv, row0);
                r_acc = __ldg(a.acc_b + b);
            }
        };
        auto park = [&]() {  // the gathered batch into the shared buffer
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                sb_g[lane + 32 * i] = Elem<TIn>::to_f32(r_g[i]);
                sb_m[lane + 32 * i] = r_m[i];
            }
            if (lane < NB) {
                sb_acc[lane] = r_acc;
                sb_id[lane] = r_id;
            }
            __syncwarp();
        };
        take_claims(0);
        gather();
        const uint64_t pol = l2_evict_first_policy();  // each state row is read once
        int issued = 0;
        bool pok = true;
        int k = 0;
        for (;; ++k) {
            if (k % NB == 0) {
                __syncwarp();
                park();
                take_claims(k / NB + 1);
                gather();
                claim();
            }
            const uint32_t u = sb_id[k % NB];
            if (u == kRsEnd) break;
            const int s = stage_of(k);
            unsigned char *st = smem + s * St::BYTES;
            if (use_of(k) > 0) {  // the group's block that used this stage before
                pok = __all_sync(0xffffffffu, mbar_wait_bounded(empty(s), (uint32_t)((use_of(k) - 1) & 1), bound));
                if (!pok) break;
            }
            uint32_t n, b, hv, row0;
            coords(u, n, b, hv, row0);
            const int ib = k % NB;
            const int32_t acc = sb_acc[ib];
            const uint32_t mword = lane < kRsSteps ? sb_m[ib * kRsSteps + lane] : 0u;
            const float gval = lane < kRsSteps ? sb_g[ib * kRsSteps + lane] : 1.f;
            const int steps = (int)(acc < 0 ? 0 : ((int64_t)acc < a.steps ? (int64_t)acc : a.steps));
            const bool on = lane < steps && (a.mask == nullptr || mword != 0u);
            const unsigned act = __ballot_sync(0xffffffffu, on);
            if (lane == 0) {
                mbar_arrive_expect_tx(full(s), (uint32_t)St::STATE + (act ? (uint32_t)ra.box_steps * St::STEP_TX : 0u));
                tma_load_3d(sh_addr(st), &tm_s, 0, (int)row0, (int)n, full(s), pol);
                if (act) {  // the rows of steps 0 .. box_steps - 1 (those past T arrive as zeros)
                    tma_load_4d(sh_addr(st + St::OFF_K), &tm_k, 0, (int)hv, 0, (int)b, full(s));
                    tma_load_4d(sh_addr(st + St::OFF_D), &tm_d, (int)row0, (int)hv, 0, (int)b, full(s));
                }
            }
            issued = k + 1;
            // The block's scale schedule: the operations of scale_schedule
            // (tile.cuh) in the same order -- from G = 1, G' = G g per active
            // step, folded when G' leaves range -- with every lane walking the
            // chain on shuffled g values instead of one lane reading them from
            // shared memory; lane tt keeps step tt's G'.
            float Gl = 1.f, gp_mine = 1.f;
            unsigned direct = 0u;
#pragma unroll
            for (int tt = 0; tt < kRsSteps; ++tt) {
                const float gt = __shfl_sync(0xffffffffu, gval, tt);
                if ((act >> tt) & 1u) {
                    const float Gp = __fmul_rn(Gl, gt);
                    const bool dir = !scale_in_range(Gp);
                    if (lane == tt) gp_mine = Gp;
                    direct |= (dir ? 1u : 0u) << tt;
                    Gl = dir ? 1.f : Gp;
                }
            }
            if (on) {
                StepScalars *sc = reinterpret_cast<StepScalars *>(st + St::OFF_SC);
                sc[lane].Gp = gp_mine;
                sc[lane].inv = ((direct >> lane) & 1u) ? 1.f : __frcp_rn(gp_mine);
            }
            if (lane == 0) {
                unsigned *info = reinterpret_cast<unsigned *>(st + St::OFF_INFO);
                info[0] = act;
                info[1] = direct;
                info[2] = __float_as_uint(Gl);
                info[3] = u;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(full(s));
        }
        // The last CTA to finish claiming resets the counters for the launch
        // that next uses this slot (only launches that use the counter).
        auto finish_claims = [&]() {
            if (dynamic && lane == 0) {
                __threadfence();  // this CTA's claims come before its count
                if (atomicAdd(ra.sched + 1, 1u) == gridDim.x - 1) {
                    atomicExch(ra.sched, 0u);
                    atomicExch(ra.sched + 1, 0u);
                }
            }
        };
        if (pok) finish_claims();  // no further claim: counted now, so its latency overlaps the drain
        if (!pok) {
            if (lane == 0) atomicExch(ra.wait_flag, 1u);
            // the blocks this CTA claimed but did not issue, and every block no
            // CTA has claimed yet (taken from the counter here, so the other
            // CTAs stop), are written as NaN
            auto poison = [&](uint32_t u) {
                if (u >= nblocks) return;
                uint32_t n, b, hv, row0;
                coords(u, n, b, hv, row0);
                const float nanv = __int_as_float(0x7fc00000);
                const float4 nan4 = make_float4(nanv, nanv, nanv, nanv);
                for (int e = lane; e < kRsRows * (kRsDk / 4); e += 32) {
                    const int r = e / (kRsDk / 4), c = e - r * (kRsDk / 4);
                    if ((int64_t)row0 + r < a.Dv)
                        reinterpret_cast<float4 *>(sout)[((int64_t)n * a.Dv + row0 + r) * (kRsDk / 4) + c] = nan4;
                }
            };
            for (int i = k % NB; i < NB; ++i) poison(sb_id[i]);
            for (int i = 0; i < NB; ++i) poison(__shfl_sync(0xffffffffu, r_id, i));
            const uint32_t next0 = __shfl_sync(0xffffffffu, r_next, 0);
            for (int i = 0; i < NB; ++i) poison(next0 == kRsEnd ? kRsEnd : dyn0 + next0 + (uint32_t)i);
            while (dynamic) {
                uint32_t u = lane == 0 ? atomicAdd(ra.sched, 1u) : 0u;
                u = dyn0 + __shfl_sync(0xffffffffu, u, 0);
                if (u >= nblocks) break;
                poison(u);
            }
            finish_claims();
        }
        // No copy may land after the CTA exits, whatever the compute warps
        // did: wait for the last block issued into each stage (the blocks
        // before it on that stage completed before it was issued).  This
        // comes before the end markers, whose arrivals complete one more
        // phase on a stage: a wait for the phase before that would see its
        // parity come round again and never succeed.
        for (int g = 0; g < kRsGroups; ++g) {
            const int ng = issued > g ? (issued - 1 - g) / kRsGroups + 1 : 0;  // group g's blocks issued
            for (int i = ng > NSG ? ng - NSG : 0; i < ng; ++i) {
                const int kk = i * kRsGroups + g;
                mbar_wait_bounded(full(stage_of(kk)), (uint32_t)(use_of(kk) & 1), kRsDrainCycles);
            }
        }
        // each group's next stage gets the end marker (once every copy landed)
        for (int e = 0; dynamic && pok && e < kRsGroups; ++e) {
            const int s = stage_of(k + e);
            if (use_of(k + e) > 0)
                pok = __all_sync(0xffffffffu,
                                 mbar_wait_bounded(empty(s), (uint32_t)((use_of(k + e) - 1) & 1), bound));
            if (pok && lane == 0) {
                reinterpret_cast<unsigned *>(smem + s * St::BYTES + St::OFF_INFO)[3] = kRsEnd;
                mbar_arrive(full(s));  // both of the phase's arrivals; no copy
                mbar_arrive(full(s));
            }
            __syncwarp();
        }
        if (!pok && lane == 0) atomicExch(ra.wait_flag, 1u);
        return;
    }

    // ======================================================== compute groups
    const int grp = warp >> 2, w4 = warp & 3;
    const int gi = lane / Lay::L, j = lane % Lay::L;
    const int lr0 = w4 * Lay::RW + gi * Lay::RT;  // first row of this thread within the block
    // After a wait runs out the group goes on taking its blocks from their
    // stages (each wait bounded again) and writes them as NaN.
    bool ok = true;
    for (int k = grp; dynamic || k < nfixed; k += kRsGroups) {
        const int s = stage_of(k);
        const unsigned char *st = smem + s * St::BYTES;
        const uint32_t par = (uint32_t)(use_of(k) & 1);
        // a block of the fixed share is known before its stage is ready
        const uint32_t uf = k < 2 * kRsBatch ? blockIdx.x + (uint32_t)k * gridDim.x : kRsEnd;
        uint32_t n, b, hv, row0;
        if (uf < nblocks) coords(uf, n, b, hv, row0);
        if (ok && !__all_sync(0xffffffffu, mbar_wait_bounded(ra.inject_expiry && k == grp ? never : full(s), par, bound)))
            ok = false;
        if (!ok && !__all_sync(0xffffffffu, mbar_wait_bounded(full(s), par, kRsDrainCycles))) break;
        const unsigned *info = reinterpret_cast<const unsigned *>(st + St::OFF_INFO);
        if (uf >= nblocks) {  // a block from the counter, or the end marker
            const uint32_t u = info[3];
            if (u == kRsEnd) break;
            coords(u, n, b, hv, row0);
        }
        Slice<Lay> sl;
        float G = 1.f;
        if (ok) {
            // this thread's rows: float4 chunk c * 16 + j of rows lr0 .. lr0 + 7
#pragma unroll
            for (int m = 0; m < Lay::RT; ++m)
#pragma unroll
                for (int c = 0; c < Lay::NCH; ++c)
                    sl[m][c] = reinterpret_cast<const float4 *>(st)[(lr0 + m) * (kRsDk / 4) + c * Lay::L + j];
            const unsigned act = info[0], direct = info[1];
            G = __uint_as_float(info[2]);
            const StepScalars *sc = reinterpret_cast<const StepScalars *>(st + St::OFF_SC);
            const TIn *kr = reinterpret_cast<const TIn *>(st + St::OFF_K);
            const TIn *dr = reinterpret_cast<const TIn *>(st + St::OFF_D);
            for (unsigned bits = act; bits; bits &= bits - 1u) {
                const int tt = __ffs(bits) - 1;
                const StepScalars S = sc[tt];
                float4 kk[Lay::NCH];
#pragma unroll
                for (int c = 0; c < Lay::NCH; ++c) kk[c] = rs_widen4<TIn>(kr + tt * kRsDk + 4 * (c * Lay::L + j));
                float d[Lay::RT];
#pragma unroll
                for (int q = 0; q < Lay::RT / 4; ++q) {
                    const float4 x = rs_widen4<TIn>(dr + tt * kRsRows + lr0 + 4 * q);
                    d[4 * q + 0] = __fmul_rn(x.x, S.inv);
                    d[4 * q + 1] = __fmul_rn(x.y, S.inv);
                    d[4 * q + 2] = __fmul_rn(x.z, S.inv);
                    d[4 * q + 3] = __fmul_rn(x.w, S.inv);
                }
                if ((direct >> tt) & 1u) rescale_rows<Lay>(sl, S.Gp);
                rank1_update<Lay>(sl, kk, d);
            }
        } else {
            const float nanv = __int_as_float(0x7fc00000);
#pragma unroll
            for (int m = 0; m < Lay::RT; ++m)
#pragma unroll
                for (int c = 0; c < Lay::NCH; ++c) sl[m][c] = make_float4(nanv, nanv, nanv, nanv);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));  // this warp is done with the stage
        store_rows<Lay>(sl, G, sout, n, a.Dv, row0 + lr0, j);
    }
    if (!ok && lane == 0) atomicExch(ra.wait_flag, 1u);
}

}  // namespace gdn
