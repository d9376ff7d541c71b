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
//     y = G' b + delta (k.q)                     (k.q precomputed per step)
//     s^ <- fma(k, delta / G', s^),  G <- G'     (3 FMAs per entry per step)
// and writes s = G s^ at the end.  When G' leaves [2^-32, 2^32] the scale is
// folded into s^ first and the step is the page's direct form (see
// scale_in_range).  Masked-off steps are skipped entirely, uniformly per CTA
// (the mask is per (b, t)).
#pragma once

#include "launch.h"
#include "tile.cuh"

namespace gdn {

// Shared memory of one staged chunk of tc timesteps (floats unless noted):
//   sK[tc][DK]  sQ[tc][DK]  sV[tc][rows_cta]  sG[tc]  sB[tc]  sKQ[tc]  sAct[tc] (int)
__host__ __device__ constexpr size_t record_smem_bytes(int dk, int tc, int rows_cta) {
    return sizeof(float) * ((size_t)2 * tc * dk + (size_t)tc * rows_cta + 3 * (size_t)tc) +
           sizeof(int) * (size_t)tc;
}

template <typename TIn, int DK>
__global__ void __launch_bounds__(kMaxThreads, MinBlocks<DK>::value)
record_kernel(const RecordArgs a) {
    using Lay = TileLayout<DK>;
    constexpr int RT = Lay::RT, NCH = Lay::NCH, L = Lay::L, GPW = Lay::GPW, RW = Lay::RW;
    extern __shared__ __align__(16) float smem[];

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int gi = lane / L, j = lane % L;
    const int rows_cta = a.rows_cta, TC = a.tc;
    const int64_t n = blockIdx.x / a.row_blocks;
    const int64_t rb = blockIdx.x - n * a.row_blocks;
    const int64_t b = n / a.Hv, hv = n - b * a.Hv;
    const int64_t hk = hv / (a.Hv / a.Hk);
    const int64_t row0 = rb * rows_cta;

    float *sK = smem;
    float *sQ = sK + TC * DK;
    float *sV = sQ + TC * DK;
    float *sG = sV + TC * rows_cta;
    float *sB = sG + TC;
    float *sKQ = sB + TC;
    int *sAct = reinterpret_cast<int *>(sKQ + TC);

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

    // The state slice stays in registers for the whole launch.
    float4 s[RT][NCH];
    load_rows<DK>(s, a.state_in, n, a.Dv, row0, warp, gi, j);
    float G = 1.f;

    for (int64_t t0 = 0; t0 < a.T; t0 += TC) {
        const int tcnt = (int)min((int64_t)TC, a.T - t0);
        const uint32_t *mrow = a.mask ? a.mask + b * a.T + t0 : nullptr;
        if (t0 > 0) __syncthreads();  // previous chunk fully consumed

        // ---- stage the chunk: k, q rows of head hk; v entries of this CTA's rows; g, beta
        const int64_t kq_off = ((b * a.T + t0) * a.Hk + hk) * DK;
        stage_key_rows<TIn, DK>(sK, kp, kq_off, a.Hk * DK, tcnt, mrow, tid, nthr);
        stage_key_rows<TIn, DK>(sQ, qp, kq_off, a.Hk * DK, tcnt, mrow, tid, nthr);
        for (int i = tid; i < tcnt * rows_cta; i += nthr) {
            const int tt = i / rows_cta;
            const int64_t dv = row0 + (i - tt * rows_cta);
            float val = 0.f;
            if (dv < a.Dv && (!mrow || __ldg(mrow + tt) != 0u))
                val = ld_f32(vp + ((b * a.T + t0 + tt) * a.Hv + hv) * a.Dv + dv);
            sV[i] = val;
        }
        for (int i = tid; i < tcnt; i += nthr) {
            const int on = mrow ? (__ldg(mrow + i) != 0u) : 1;
            const int64_t gb = (b * a.T + t0 + i) * a.Hv + hv;
            sAct[i] = on;
            sG[i] = on ? ld_f32(gp + gb) : 1.f;
            sB[i] = on ? ld_f32(bp + gb) : 0.f;
        }
        __syncthreads();
        // k.q of every staged step, one warp per step
        for (int tt = warp; tt < tcnt; tt += nthr >> 5) {
            float acc = 0.f;
            if (sAct[tt])
                for (int i = lane; i < DK; i += 32) acc = fmaf(sK[tt * DK + i], sQ[tt * DK + i], acc);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) sKQ[tt] = acc;
        }
        __syncthreads();

        // ---- the recurrence over the chunk
        for (int tt = 0; tt < tcnt; ++tt) {
            if (!sAct[tt]) continue;  // uniform across the CTA
            const float *krow = sK + tt * DK;
            const float4 *k4 = reinterpret_cast<const float4 *>(krow);
            const float4 *q4 = reinterpret_cast<const float4 *>(sQ + tt * DK);

            // a = s^.k and b = s^.q partials over this lane's chunks
            float2 pa[RT], pb[RT];
#pragma unroll
            for (int m = 0; m < RT; ++m) pa[m] = pb[m] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const float4 kk = k4[c * L + j];
                const float4 qq = q4[c * L + j];
#pragma unroll
                for (int m = 0; m < RT; ++m) {
                    pa[m] = ffma2(lo2(s[m][c]), lo2(kk), pa[m]);
                    pa[m] = ffma2(hi2(s[m][c]), hi2(kk), pa[m]);
                    pb[m] = ffma2(lo2(s[m][c]), lo2(qq), pb[m]);
                    pb[m] = ffma2(hi2(s[m][c]), hi2(qq), pb[m]);
                }
            }
            float red[2 * RT];
#pragma unroll
            for (int m = 0; m < RT; ++m) {
                red[2 * m] = pa[m].x + pa[m].y;
                red[2 * m + 1] = pb[m].x + pb[m].y;
            }
#pragma unroll
            for (int off = 1; off < L; off <<= 1)
#pragma unroll
                for (int i = 0; i < 2 * RT; ++i) red[i] += __shfl_xor_sync(0xffffffffu, red[i], off);

            const float gt = sG[tt], bt = sB[tt], kq = sKQ[tt];
            const float Gp = __fmul_rn(G, gt);
            const bool direct = !scale_in_range(Gp);
            const float inv = direct ? 1.f : __frcp_rn(Gp);
            const int64_t orow = ((b * a.T + t0 + tt) * a.Hv + hv) * a.Dv;
            float d[RT];
#pragma unroll
            for (int m = 0; m < RT; ++m) {
                const int lr = warp * RW + gi + m * GPW;
                const float kv = Gp * red[2 * m];
                const float delta = (sV[tt * rows_cta + lr] - kv) * bt;
                const float yv = fmaf(Gp, red[2 * m + 1], delta * kq);
                d[m] = __fmul_rn(delta, inv);
                if ((m % L) == j) {
                    const int64_t dv = row0 + lr;
                    if (dv < a.Dv) {
                        st_from_f32(yp + orow + dv, yv);
                        st_from_f32(dp + orow + dv, delta);
                    }
                }
            }
            if (direct) {
                rescale_rows<DK>(s, Gp);
                G = 1.f;
            } else {
                G = Gp;
            }
            rank1_update<DK>(s, krow, d, j);

            if (capture) {
                const int64_t gb = (b * a.T + t0 + tt) * a.Hv + hv;
                if (klp)
                    for (int i = tid; i < DK; i += nthr) st_from_f32(klp + gb * DK + i, krow[i]);
                if (glp && tid == 0) st_from_f32(glp + gb, gt);
            }
        }
    }

    store_rows<DK>(s, G, a.state_out, n, a.Dv, row0, warp, gi, j);
}

template <typename TIn, int DK>
cudaError_t launch_record_t(const RecordArgs &a, const Geometry &geo, cudaStream_t st) {
    auto kern = record_kernel<TIn, DK>;
    if (geo.smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)geo.smem);
        if (e != cudaSuccess) return e;
    }
    const int64_t blocks = (int64_t)(a.B * a.Hv) * geo.row_blocks;
    kern<<<(unsigned)blocks, geo.threads, geo.smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
