// replay.cuh -- the replay kernel: re-fold the accepted prefix of an
// innovation tape onto a state snapshot ("metaltile-std
// gated_delta_replay.rs", module doc and kernel state_replay):
//     do_step = (t < accepted) && mask[b,t]
//     s <- select(do_step, s g_t + k_t delta_t, s)
// The page evaluates both arms for every t < T and selects; here the step
// flag is uniform per CTA, so skipped steps are branched over and their tape
// slots (and every slot at t >= accepted) are never read.  With per-sequence
// accepted counts (one per b) the count is read once per CTA, since a CTA's
// rows all belong to one sequence.
//
// The fold uses the same scaled state s = G s^ and the same f32 operations as
// the record kernel (G' = G g, fold the scale when G' leaves range, else
// s^ <- fma(k, delta * (1/G'), s^)), so replaying a float32 tape reproduces
// the record kernel's state_out bit for bit.  Tape rows are staged through
// the same two-slot cp.async ring as record's inputs.
#pragma once

#include <type_traits>

#include "launch.h"
#include "record.cuh"
#include "tile.cuh"

namespace gdn {

// Shared memory of the replay kernel (bytes), in carve order:
//   raw ring   2 x { K[tc][dk], D[tc][rows] }   element type
//   f32 work   { K, D } (2-byte element types only)
//   scalars    StepScalars[tc], g[tc], {direct bits, final scale}
__host__ __device__ constexpr size_t replay_smem_bytes(int dk, int tc, int rows, int esize) {
    return 2 * align16((size_t)(tc * dk + tc * rows) * esize) +
           (esize == 4 ? 0 : align16((size_t)(tc * dk + tc * rows) * 4)) +
           align16((size_t)tc * sizeof(StepScalars)) + align16((size_t)tc * 4) + 16;
}

// TST: the state is stored in TIn (widened on load, rounded on store);
// otherwise it is float32.
// Register budget: five resident CTAs per SM when a thread holds at most 64
// state floats (measured 3 % faster than four on the rollback shape).
template <class Lay>
__host__ __device__ constexpr int replay_min_blocks() { return Lay::STATE <= 64 ? 5 : 2; }

template <typename TIn, class Lay, bool TST>
__global__ void __launch_bounds__(32 * kMaxWarpsPerCta, replay_min_blocks<Lay>())
replay_kernel(const ReplayArgs a) {
    pdl_trigger();
    pdl_wait();
    using TS = typename std::conditional<TST, TIn, float>::type;
    constexpr int DK = Lay::DK;
    constexpr int RT = Lay::RT, NCH = Lay::NCH, L = Lay::L, RW = Lay::RW;
    constexpr bool kF32 = std::is_same<TIn, float>::value;
    extern __shared__ __align__(16) unsigned char smem[];

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int gi = lane / L, j = lane % L;
    const int R = a.rows_cta, TC = a.tc;
    const int64_t n = blockIdx.x / a.row_blocks;
    const int64_t rb = blockIdx.x - n * a.row_blocks;
    const int64_t b = n / a.Hv, hv = n - b * a.Hv;
    const int64_t row0 = rb * R;
    const int vlim = (int)min((int64_t)R, a.Dv - row0);
    const int lr0 = warp * RW + gi * RT;

    const size_t slot_bytes = align16((size_t)(TC * DK + TC * R) * sizeof(TIn));
    unsigned char *ring = smem;
    auto slotK = [&](int sl) { return reinterpret_cast<TIn *>(ring + sl * slot_bytes); };
    auto slotD = [&](int sl) { return slotK(sl) + TC * DK; };
    unsigned char *p = ring + 2 * slot_bytes;
    float *wK = nullptr, *wD = nullptr;
    if (!kF32) {
        wK = reinterpret_cast<float *>(p);
        wD = wK + TC * DK;
        p += align16((size_t)(TC * DK + TC * R) * 4);
    }
    StepScalars *sc = reinterpret_cast<StepScalars *>(p);
    p += align16((size_t)TC * sizeof(StepScalars));
    float *sg = reinterpret_cast<float *>(p);
    p += align16((size_t)TC * 4);
    unsigned *s_direct = reinterpret_cast<unsigned *>(p);
    float *s_gfinal = reinterpret_cast<float *>(p + 4);

    const TIn *dlp = static_cast<const TIn *>(a.delta_log);
    const TIn *klp = static_cast<const TIn *>(a.k_log);
    const TIn *glp = static_cast<const TIn *>(a.g_log);

    // steps this CTA folds: uniform per CTA (one sequence b per CTA)
    int64_t steps = a.steps;
    if (a.acc_b) {
        const int64_t ab = (int64_t)__ldg(a.acc_b + b);
        steps = ab < 0 ? 0 : (ab < steps ? ab : steps);
    }

    float pre_g = 1.f;
    auto issue = [&](int64_t c) -> unsigned {
        const int64_t t0 = c * TC;
        const int tcnt = (int)min((int64_t)TC, steps - t0);
        const int slot = (int)(c & 1);
        const unsigned bits = chunk_bits(a.mask ? a.mask + b * a.T + t0 : nullptr, tcnt, lane);
        const int64_t row_first = (b * a.T + t0) * a.Hv + hv;  // (b, t0, hv)
        async_rows<TIn>(slotK(slot), klp + row_first * DK, a.Hv * DK, tcnt, DK, DK, bits, tid, nthr);
        const int64_t d_off = row_first * a.Dv + row0;
        if (a.vec_d) {
            async_rows<TIn>(slotD(slot), dlp + d_off, a.Hv * a.Dv, tcnt, R, vlim, bits, tid, nthr);
        } else {
            TIn *dst = slotD(slot);
            for (int i = tid; i < tcnt * R; i += nthr) {
                const int tt = i / R, r = i - tt * R;
                if (((bits >> tt) & 1u) && r < vlim) dst[i] = dlp[d_off + tt * a.Hv * a.Dv + r];
            }
        }
        cp_async_commit();
        if (tid < tcnt && ((bits >> tid) & 1u)) pre_g = ld_f32(glp + row_first + tid * a.Hv);
        return bits;
    };

    Slice<Lay> s;
    const int64_t nchunks = (steps + TC - 1) / TC;
    unsigned next_bits = nchunks > 0 ? issue(0) : 0u;
    load_rows<Lay>(s, static_cast<const TS *>(a.state_in), n, a.Dv, row0 + lr0, j);
    float G_sched = 1.f;

    for (int64_t c = 0; c < nchunks; ++c) {
        const int tcnt = (int)min((int64_t)TC, steps - c * TC);
        const int slot = (int)(c & 1);
        const unsigned bits = next_bits;
        cp_async_wait_all();
        __syncthreads();  // (a)
        const float *cK, *cD;
        if (kF32) {
            cK = reinterpret_cast<const float *>(slotK(slot));
            cD = reinterpret_cast<const float *>(slotD(slot));
            if (vlim < R)
                for (int i = tid; i < tcnt * R; i += nthr)
                    if ((i % R) >= vlim) reinterpret_cast<float *>(slotD(slot))[i] = 0.f;
        } else {
            widen_block<TIn>(wK, slotK(slot), tcnt * DK, DK, DK, tid, nthr);
            widen_block<TIn>(wD, slotD(slot), tcnt * R, R, vlim, tid, nthr);
            cK = wK;
            cD = wD;
        }
        if (tid < tcnt) sg[tid] = pre_g;
        __syncthreads();  // (b)
        if (c + 1 < nchunks) next_bits = issue(c + 1);
        if (warp == (nthr >> 5) - 1) {  // the last warp runs the scale schedule
            const unsigned dbits = scale_schedule(sc, sg, bits, tcnt, G_sched, lane);
            if (lane == 0) {
                *s_direct = dbits;
                *s_gfinal = G_sched;
            }
        }
        __syncthreads();  // (c)
        const unsigned direct = *s_direct;

        for (int tt = 0; tt < tcnt; ++tt) {
            if (!((bits >> tt) & 1u)) continue;  // uniform across the CTA
            const StepScalars S = sc[tt];
            float4 kk[NCH];
            lane_chunks<Lay>(kk, cK + tt * DK, j);
            float d[RT];
            if (RT % 4 == 0) {  // this thread's RT rows are contiguous and 16-byte aligned
                const float4 *d4 = reinterpret_cast<const float4 *>(cD + tt * R + lr0);
#pragma unroll
                for (int q = 0; q < RT / 4; ++q) {
                    const float4 x = d4[q];
                    d[4 * q + 0] = __fmul_rn(x.x, S.inv);
                    d[4 * q + 1] = __fmul_rn(x.y, S.inv);
                    d[4 * q + 2] = __fmul_rn(x.z, S.inv);
                    d[4 * q + 3] = __fmul_rn(x.w, S.inv);
                }
            } else {
#pragma unroll
                for (int m = 0; m < RT; ++m) d[m] = __fmul_rn(cD[tt * R + lr0 + m], S.inv);
            }
            if ((direct >> tt) & 1u) rescale_rows<Lay>(s, S.Gp);
            rank1_update<Lay>(s, kk, d);
        }
    }
    const float G = nchunks > 0 ? *s_gfinal : 1.f;
    store_rows<Lay>(s, G, static_cast<TS *>(a.state_out), n, a.Dv, row0 + lr0, j);
}

template <typename TIn, class Lay>
cudaError_t launch_replay_layout(const ReplayArgs &a, const Geometry &geo, cudaStream_t st) {
    auto kern = replay_kernel<TIn, Lay, false>;
    if constexpr (!std::is_same<TIn, float>::value) {
        if (a.tstate) kern = replay_kernel<TIn, Lay, true>;
    }
    if (geo.smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)geo.smem);
        if (e != cudaSuccess) return e;
    }
    const int64_t blocks = (int64_t)(a.B * a.Hv) * geo.row_blocks;
    return launch_dependent(kern, (unsigned)blocks, geo.threads, geo.smem, st, a);
}

}  // namespace gdn
