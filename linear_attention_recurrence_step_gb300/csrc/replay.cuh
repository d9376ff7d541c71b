// replay.cuh -- the replay kernel: re-fold the accepted prefix of an
// innovation tape onto a state snapshot ("metaltile-std
// gated_delta_replay.rs", module doc and kernel state_replay):
//     do_step = (t < accepted) && mask[b,t]
//     s <- select(do_step, s g_t + k_t delta_t, s)
// The page evaluates both arms for every t < T and selects; here the step
// flag is uniform per CTA, so skipped steps are branched over and their tape
// slots (and every slot at t >= accepted) are never read.
//
// The fold uses the same scaled state s = G s^ and the same f32 operations as
// the record kernel (G' = G g, fold the scale when G' leaves range, else
// s^ <- fma(k, delta * (1/G'), s^)), so replaying a float32 tape reproduces
// the record kernel's state_out bit for bit.
#pragma once

#include "launch.h"
#include "tile.cuh"

namespace gdn {

// Shared memory of one staged chunk: sK[tc][DK] sD[tc][rows_cta] sG[tc] sAct[tc] (int)
__host__ __device__ constexpr size_t replay_smem_bytes(int dk, int tc, int rows_cta) {
    return sizeof(float) * ((size_t)tc * dk + (size_t)tc * rows_cta + (size_t)tc) +
           sizeof(int) * (size_t)tc;
}

template <typename TIn, int DK>
__global__ void __launch_bounds__(kMaxThreads, MinBlocks<DK>::value)
replay_kernel(const ReplayArgs a) {
    using Lay = TileLayout<DK>;
    constexpr int RT = Lay::RT, L = Lay::L, GPW = Lay::GPW, RW = Lay::RW;
    (void)L;
    extern __shared__ __align__(16) float smem[];

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int gi = lane / Lay::L, j = lane % Lay::L;
    const int rows_cta = a.rows_cta, TC = a.tc;
    const int64_t n = blockIdx.x / a.row_blocks;
    const int64_t rb = blockIdx.x - n * a.row_blocks;
    const int64_t b = n / a.Hv, hv = n - b * a.Hv;
    const int64_t row0 = rb * rows_cta;

    float *sK = smem;
    float *sD = sK + TC * DK;
    float *sG = sD + TC * rows_cta;
    int *sAct = reinterpret_cast<int *>(sG + TC);

    const TIn *dlp = static_cast<const TIn *>(a.delta_log);
    const TIn *klp = static_cast<const TIn *>(a.k_log);
    const TIn *glp = static_cast<const TIn *>(a.g_log);

    float4 s[RT][Lay::NCH];
    load_rows<DK>(s, a.state_in, n, a.Dv, row0, warp, gi, j);
    float G = 1.f;

    for (int64_t t0 = 0; t0 < a.steps; t0 += TC) {
        const int tcnt = (int)min((int64_t)TC, a.steps - t0);
        const uint32_t *mrow = a.mask ? a.mask + b * a.T + t0 : nullptr;
        if (t0 > 0) __syncthreads();

        const int64_t row_first = (b * a.T + t0) * a.Hv + hv;  // (b, t0, hv)
        stage_key_rows<TIn, DK>(sK, klp, row_first * DK, a.Hv * DK, tcnt, mrow, tid, nthr);
        for (int i = tid; i < tcnt * rows_cta; i += nthr) {
            const int tt = i / rows_cta;
            const int64_t dv = row0 + (i - tt * rows_cta);
            float val = 0.f;
            if (dv < a.Dv && (!mrow || __ldg(mrow + tt) != 0u))
                val = ld_f32(dlp + (row_first + tt * a.Hv) * a.Dv + dv);
            sD[i] = val;
        }
        for (int i = tid; i < tcnt; i += nthr) {
            const int on = mrow ? (__ldg(mrow + i) != 0u) : 1;
            sAct[i] = on;
            sG[i] = on ? ld_f32(glp + row_first + i * a.Hv) : 1.f;
        }
        __syncthreads();

        for (int tt = 0; tt < tcnt; ++tt) {
            if (!sAct[tt]) continue;  // uniform across the CTA
            const float Gp = __fmul_rn(G, sG[tt]);
            const bool direct = !scale_in_range(Gp);
            const float inv = direct ? 1.f : __frcp_rn(Gp);
            float d[RT];
#pragma unroll
            for (int m = 0; m < RT; ++m)
                d[m] = __fmul_rn(sD[tt * rows_cta + warp * RW + gi + m * GPW], inv);
            if (direct) {
                rescale_rows<DK>(s, Gp);
                G = 1.f;
            } else {
                G = Gp;
            }
            rank1_update<DK>(s, sK + tt * DK, d, j);
        }
    }

    store_rows<DK>(s, G, a.state_out, n, a.Dv, row0, warp, gi, j);
}

template <typename TIn, int DK>
cudaError_t launch_replay_t(const ReplayArgs &a, const Geometry &geo, cudaStream_t st) {
    auto kern = replay_kernel<TIn, DK>;
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
