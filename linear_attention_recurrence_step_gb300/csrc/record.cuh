// record.cuh -- the record kernel: T gated delta-rule steps with delta-tape
// capture ("metaltile-std gated_delta_replay.rs", kernel
// gated_delta_step_record; tape layout from the module doc).
//
// Per state row s (Dk floats) and active step t, the page computes
//     s <- g s;  kv = s.k;  delta = (v - kv) beta;  tape <- delta;
//     s <- s + k delta;  y = s.q
// with two dot-product reductions per step.  This kernel computes the same
// quantities in one reduction round per step, on the scaled state s = G s^:
//     a = s^.k,  b = s^.q                       (one 2-level shuffle round)
//     G' = G g;  kv = G' a;  delta = (v - kv) beta
//     y = G' b + delta (k.q)                     (k.q computed once per step)
//     s^ <- fma(k, delta / G', s^),  G <- G'     (3 FMAs per entry per step)
// and writes s = G s^ at the end.  When G' leaves [2^-32, 2^32] the scale is
// folded into s^ first and the step is the page's direct form (see
// scale_in_range).  Masked-off steps are skipped entirely, uniformly per CTA
// (the mask is per (b, t)).
//
// Timesteps are staged in chunks of tc through a two-slot cp.async ring (the
// next chunk's k / q / v rows are in flight while this chunk is computed);
// bf16 / f16 rows are widened to f32 once per chunk.
#pragma once

#include <type_traits>

#include "launch.h"
#include "tile.cuh"

namespace gdn {


// Shared memory of the record kernel (bytes), in carve order:
//   raw ring   2 x { K[tc][dk], Q[tc][dk], V[tc][rows] }   element type
//   f32 work   { K, Q, V } (only for 2-byte element types; f32 reads the ring)
//   scalars    StepScalars[tc], g[tc], {direct bits, final scale}
__host__ __device__ constexpr size_t record_smem_bytes(int dk, int tc, int rows, int esize) {
    return 2 * align16((size_t)(2 * tc * dk + tc * rows) * esize) +
           (esize == 4 ? 0 : align16((size_t)(2 * tc * dk + tc * rows) * 4)) +
           align16((size_t)tc * sizeof(StepScalars)) + align16((size_t)tc * 4) + 16;
}

// TST: the state is stored in TIn (widened on load, rounded on store);
// otherwise it is float32.
template <typename TIn, class Lay, bool TST>
__global__ void __launch_bounds__(Lay::MAX_THREADS, Lay::MIN_BLOCKS)
record_kernel(const RecordArgs a) {
    pdl_trigger();
    pdl_wait();
    using TS = typename std::conditional<TST, TIn, float>::type;
    constexpr int DK = Lay::DK;
    constexpr int RT = Lay::RT, NCH = Lay::NCH, L = Lay::L, RW = Lay::RW, REDV = Lay::REDV;
    constexpr bool kF32 = std::is_same<TIn, float>::value;
    constexpr int VEC = 16 / sizeof(TIn);
    extern __shared__ __align__(16) unsigned char smem[];

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int gi = lane / L, j = lane % L;
    const int R = a.rows_cta, TC = a.tc;
    const int64_t n = blockIdx.x / a.row_blocks;
    const int64_t rb = blockIdx.x - n * a.row_blocks;
    const int64_t b = n / a.Hv, hv = n - b * a.Hv;
    const int64_t hk = a.tiled_gqa ? hv % a.Hk : hv / (a.Hv / a.Hk);  // key head of hv
    const int64_t row0 = rb * R;
    const int vlim = (int)min((int64_t)R, a.Dv - row0);  // live rows of this block
    const int lr0 = warp * RW + gi * RT;                 // this thread's first local row
    const int my_m = REDV == 2 ? j : (j >> 1);           // row finished by this lane
    const int my_lr = lr0 + my_m;
    const bool my_store = (REDV == 2 || (j & 1) == 0) && my_lr < vlim;
    const int src0 = lane & ~(L - 1);                    // first lane of the row group

    // ---- carve shared memory (ring slots addressed arithmetically: no
    // dynamically indexed pointer arrays, which would live in local memory)
    const size_t slot_bytes = align16((size_t)(2 * TC * DK + TC * R) * sizeof(TIn));
    unsigned char *ring = smem;
    auto slotK = [&](int sl) { return reinterpret_cast<TIn *>(ring + sl * slot_bytes); };
    auto slotQ = [&](int sl) { return slotK(sl) + TC * DK; };
    auto slotV = [&](int sl) { return slotK(sl) + 2 * TC * DK; };
    unsigned char *p = ring + 2 * slot_bytes;
    float *wK = nullptr, *wQ = nullptr, *wV = nullptr;
    if (!kF32) {
        wK = reinterpret_cast<float *>(p);
        wQ = wK + TC * DK;
        wV = wQ + TC * DK;
        p += align16((size_t)(2 * TC * DK + TC * R) * 4);
    }
    StepScalars *sc = reinterpret_cast<StepScalars *>(p);
    p += align16((size_t)TC * sizeof(StepScalars));
    float *sg = reinterpret_cast<float *>(p);
    p += align16((size_t)TC * 4);
    unsigned *s_direct = reinterpret_cast<unsigned *>(p);
    float *s_gfinal = reinterpret_cast<float *>(p + 4);

    const TIn *qp = static_cast<const TIn *>(a.q);
    const TIn *kp = static_cast<const TIn *>(a.k);
    const TIn *vp = static_cast<const TIn *>(a.v);
    const TIn *gp = static_cast<const TIn *>(a.g);
    const TIn *bp = static_cast<const TIn *>(a.beta);
    TIn *yp = static_cast<TIn *>(a.y);
    TIn *dp = static_cast<TIn *>(a.delta_log);
    TIn *klp = static_cast<TIn *>(a.k_log);
    TIn *glp = static_cast<TIn *>(a.g_log);
    const bool capture = (rb == 0);  // one CTA per tile writes k_log / g_log

    // ---- issue the copies of chunk c into ring slot c & 1; scalars to registers
    float pre_g = 1.f, pre_b = 0.f;
    auto issue = [&](int64_t c) -> unsigned {
        const int64_t t0 = c * TC;
        const int tcnt = (int)min((int64_t)TC, a.T - t0);
        const int slot = (int)(c & 1);
        const unsigned bits = chunk_bits(a.mask ? a.mask + b * a.T + t0 : nullptr, tcnt, lane);
        const int64_t kq_off = ((b * a.T + t0) * a.Hk + hk) * DK;
        async_rows<TIn>(slotK(slot), kp + kq_off, a.Hk * DK, tcnt, DK, DK, bits, tid, nthr);
        async_rows<TIn>(slotQ(slot), qp + kq_off, a.Hk * DK, tcnt, DK, DK, bits, tid, nthr);
        const int64_t v_off = ((b * a.T + t0) * a.Hv + hv) * a.Dv + row0;
        if (a.vec_v) {
            async_rows<TIn>(slotV(slot), vp + v_off, a.Hv * a.Dv, tcnt, R, vlim, bits, tid, nthr);
        } else {
            TIn *dst = slotV(slot);
            for (int i = tid; i < tcnt * R; i += nthr) {
                const int tt = i / R, r = i - tt * R;
                if (((bits >> tt) & 1u) && r < vlim) dst[i] = vp[v_off + tt * a.Hv * a.Dv + r];
            }
        }
        cp_async_commit();
        if (tid < tcnt && ((bits >> tid) & 1u)) {
            const int64_t gb = (b * a.T + t0 + tid) * a.Hv + hv;
            pre_g = ld_f32(gp + gb);
            pre_b = ld_f32(bp + gb);
        }
        return bits;
    };

    // The state slice stays in registers for the whole launch.
    Slice<Lay> s;
    unsigned next_bits = issue(0);
    load_rows<Lay>(s, static_cast<const TS *>(a.state_in), n, a.Dv, row0 + lr0, j);
    float G_sched = 1.f;  // the scale schedule's running G (kept by the last warp)

    const int64_t nchunks = (a.T + TC - 1) / TC;
    for (int64_t c = 0; c < nchunks; ++c) {
        const int64_t t0 = c * TC;
        const int tcnt = (int)min((int64_t)TC, a.T - t0);
        const int slot = (int)(c & 1);
        const unsigned bits = next_bits;
        cp_async_wait_all();
        __syncthreads();  // (a) chunk c visible to all; chunk c-1 fully consumed
        const float *cK, *cQ, *cV;
        if (kF32) {
            cK = reinterpret_cast<const float *>(slotK(slot));
            cQ = reinterpret_cast<const float *>(slotQ(slot));
            cV = reinterpret_cast<const float *>(slotV(slot));
            if (vlim < R)
                for (int i = tid; i < tcnt * R; i += nthr)
                    if ((i % R) >= vlim) reinterpret_cast<float *>(slotV(slot))[i] = 0.f;
        } else {
            widen_block<TIn>(wK, slotK(slot), tcnt * DK, DK, DK, tid, nthr);
            widen_block<TIn>(wQ, slotQ(slot), tcnt * DK, DK, DK, tid, nthr);
            widen_block<TIn>(wV, slotV(slot), tcnt * R, R, vlim, tid, nthr);
            cK = wK;
            cQ = wQ;
            cV = wV;
        }
        if (tid < tcnt) {
            sg[tid] = pre_g;
            sc[tid].beta = pre_b;
        }
        if (capture) {  // tape capture: k_log / g_log rows of the active steps
            const int64_t gb0 = (b * a.T + t0) * a.Hv + hv;
            if (klp) {
                const TIn *src = slotK(slot);
                for (int i = tid; i < tcnt * (DK / VEC); i += nthr) {
                    const int tt = i / (DK / VEC), x = (i - tt * (DK / VEC)) * VEC;
                    if ((bits >> tt) & 1u)
                        *reinterpret_cast<uint4 *>(klp + (gb0 + tt * a.Hv) * DK + x) =
                            *reinterpret_cast<const uint4 *>(src + tt * DK + x);
                }
            }
            if (glp && tid < tcnt && ((bits >> tid) & 1u)) st_from_f32(glp + gb0 + tid * a.Hv, pre_g);
        }
        __syncthreads();  // (b) chunk c staged; its ring slot may be refilled
        if (c + 1 < nchunks) next_bits = issue(c + 1);
        // k.q of every active step, one warp per step
        for (int tt = warp; tt < tcnt; tt += nthr >> 5) {
            float acc = 0.f;
            if ((bits >> tt) & 1u)
                for (int i = lane; i < DK; i += 32) acc = fmaf(cK[tt * DK + i], cQ[tt * DK + i], acc);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) sc[tt].kq = acc;
        }
        if (warp == (nthr >> 5) - 1) {  // the last warp runs the scale schedule
            const unsigned dbits = scale_schedule(sc, sg, bits, tcnt, G_sched, lane);
            if (lane == 0) {
                *s_direct = dbits;
                *s_gfinal = G_sched;
            }
        }
        __syncthreads();  // (c) per-step scalars ready
        const unsigned direct = *s_direct;

        // ---- the recurrence over the chunk
        const int64_t orow0 = ((b * a.T + t0) * a.Hv + hv) * a.Dv + row0 + my_lr;
        for (int tt = 0; tt < tcnt; ++tt) {
            if (!((bits >> tt) & 1u)) continue;  // uniform across the CTA
            const StepScalars S = sc[tt];
            float4 kk[NCH], qq[NCH];
            lane_chunks<Lay>(kk, cK + tt * DK, j);
            lane_chunks<Lay>(qq, cQ + tt * DK, j);

            // a = s^.k and b = s^.q partials over this lane's chunks
            float2 pa[RT], pb[RT];
#pragma unroll
            for (int m = 0; m < RT; ++m) pa[m] = pb[m] = make_float2(0.f, 0.f);
#pragma unroll
            for (int cc = 0; cc < NCH; ++cc) {
#pragma unroll
                for (int m = 0; m < RT; ++m) {
                    pa[m] = ffma2(lo2(s[m][cc]), lo2(kk[cc]), pa[m]);
                    pb[m] = ffma2(lo2(s[m][cc]), lo2(qq[cc]), pb[m]);
                }
#pragma unroll
                for (int m = 0; m < RT; ++m) {
                    pa[m] = ffma2(hi2(s[m][cc]), hi2(kk[cc]), pa[m]);
                    pb[m] = ffma2(hi2(s[m][cc]), hi2(qq[cc]), pb[m]);
                }
            }
            float red[2 * RT];
#pragma unroll
            for (int m = 0; m < RT; ++m) {
                red[2 * m] = pa[m].x + pa[m].y;
                red[2 * m + 1] = pb[m].x + pb[m].y;
            }
            transpose_reduce<Lay>(red, j);
            float A, Bq;  // s^.k and s^.q of this lane's row
            if (REDV == 2) {
                A = red[0];
                Bq = red[1];
            } else {
                const float other = __shfl_xor_sync(0xffffffffu, red[0], 1);
                A = (j & 1) ? other : red[0];
                Bq = (j & 1) ? red[0] : other;
            }

            // this lane's row: delta, y, the tape, and delta / G'
            const float kv = S.Gp * A;
            const float delta = (cV[tt * R + my_lr] - kv) * S.beta;
            const float yv = fmaf(S.Gp, Bq, delta * S.kq);
            const float dmine = __fmul_rn(delta, S.inv);
            if (my_store) {
                const int64_t o = orow0 + (int64_t)tt * a.Hv * a.Dv;
                st_from_f32(yp + o, yv);
                st_from_f32(dp + o, delta);
            }
            float d[RT];
#pragma unroll
            for (int m = 0; m < RT; ++m)
                d[m] = __shfl_sync(0xffffffffu, dmine, src0 + (REDV == 2 ? m : 2 * m));
            if ((direct >> tt) & 1u) rescale_rows<Lay>(s, S.Gp);
            rank1_update<Lay>(s, kk, d);
        }
    }
    const float G = nchunks > 0 ? *s_gfinal : 1.f;
    store_rows<Lay>(s, G, static_cast<TS *>(a.state_out), n, a.Dv, row0 + lr0, j);
}

template <typename TIn, class Lay>
cudaError_t launch_record_layout(const RecordArgs &a, const Geometry &geo, cudaStream_t st) {
    auto kern = record_kernel<TIn, Lay, false>;
    if constexpr (!std::is_same<TIn, float>::value) {
        if (a.tstate) kern = record_kernel<TIn, Lay, true>;
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
