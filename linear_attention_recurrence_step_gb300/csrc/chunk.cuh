// chunk.cuh -- chunked prefill: the record recurrence of "metaltile-std
// gated_delta_replay.rs" (kernel gated_delta_step_record) regrouped over
// chunks of C = 16 steps so that long calls run as dense products on the
// tensor cores (warp-level mma.sync, tf32 operands, f32 accumulate), in
// float32 accuracy.
//
// Within a chunk (steps 0..C-1 after the chunk's first step, state s_in at
// entry, inactive steps given g = 1 and beta = 0) the step
//     s <- g s;  delta = beta (v - s.k);  s <- s + k delta;  y = s.q
// unrolls, with Gam_t = prod_{x<=t} g_x and A[t][u] = prod_{u<x<=t} g_x, to
//     (I + N) delta = r,   N[t][u] = beta_t A[t][u] (k_u.k_t)   (u < t)
//     r_t   = beta_t (v_t - Gam_t s_in.k_t)
//     y_t   = Gam_t s_in.q_t + sum_{u<=t} A[t][u] (k_u.q_t) delta_u
//     s_out = Gam_{C-1} s_in + sum_u A[C-1][u] delta_u k_u
// No step divides by a decay, so g = 0 or long products of small g need no
// special case.  Everything that does not depend on the state -- W = (I+N)^-1
// with beta folded in (Wb[t][u] = W[t][u] beta_u), Mq[t][u] = A[t][u]
// (k_u.q_t), Gam, aC[u] = A[C-1][u] -- is computed for every (b, hv, chunk)
// at once by chunk_local_kernel into a caller-provided workspace.  The
// sequential part, chunk_scan_kernel, then walks the chunks of one tile's row
// block with four MMA products per chunk:
//     P  = S_in [Gam K ; Gam Q]^T     (rows x 2C, contraction over Dk)
//     D  = (V^T - P_k) Wb^T           (the deltas, contraction over C)
//     Y  = P_q + D Mq^T               (contraction over C)
//     S  = Gam_{C-1} S_in + D (aC K)  (rows x Dk, contraction over C)
//
// Accuracy: every product runs as three tf32 MMAs (a_hi b_lo + a_lo b_hi +
// a_hi b_hi, each operand split x = hi + lo with hi = tf32(x)), which keeps
// about 21 significant bits per product and f32 accumulation; the state stays
// f32 in the accumulator fragments for the whole launch.
//
// Work split: a CTA owns 16 state rows of one (b, hv) tile and four warps
// split the Dk columns (each holds 16 rows x Dk/4 of the state).  The partial
// products P of the four warps are summed through shared memory once per
// chunk; that exchange is the kernel's only CTA barrier per chunk.  Inputs of
// chunk c+2 are copied with cp.async into a three-slot ring while chunk c is
// computed, so the barrier of chunk c also publishes chunk c+1.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"
#include "tile.cuh"

namespace gdn {

constexpr int kCkC = 16;           // timesteps per chunk
constexpr int kCkWarps = 4;        // warps per scan CTA (Dk split four ways)
constexpr int kCkRows = 16;        // state rows per scan CTA
constexpr int kCkLocalThreads = 256;
constexpr int kCkWsFloats = 2 * kCkC * kCkC + 2 * kCkC;  // Wb, Mq, Gam, aC per (b, hv, chunk)
constexpr int kCkPartStride = 40;  // floats per row of a partial-product block (32 + pad)

__host__ __device__ constexpr int ck_kstride(int dk) { return dk + 8; }  // padded k / q row (elements)
__host__ __device__ constexpr int ck_vstride(int esize) { return kCkRows + 16 / esize; }

__host__ __device__ constexpr size_t ck_slot_bytes(int dk, int esize) {
    return align16((size_t)2 * kCkC * ck_kstride(dk) * esize) +
           align16((size_t)kCkC * ck_vstride(esize) * esize) + (size_t)kCkWsFloats * 4;
}
__host__ __device__ constexpr size_t chunk_scan_smem_bytes(int dk, int esize) {
    return 3 * ck_slot_bytes(dk, esize) +
           (size_t)2 * kCkWarps * kCkRows * kCkPartStride * 4;
}
__host__ __device__ constexpr size_t chunk_local_smem_bytes(int dk) {
    return (size_t)2 * kCkC * (dk + 1) * 4 + (size_t)4 * kCkC * (kCkC + 1) * 4 +
           (size_t)3 * kCkC * 4;
}

// ------------------------------------------------------------ tf32 products
__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
    return r;
}
// x ~ hi + lo, both tf32; x - hi is exact in f32.
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    hi = tf32_rna(x);
    lo = tf32_rna(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// d += a b in three tf32 products, small terms first.
__device__ __forceinline__ void mma3_tf32(float (&d)[4], const uint32_t (&ah)[4],
                                          const uint32_t (&al)[4], uint32_t bh0, uint32_t bh1,
                                          uint32_t bl0, uint32_t bl1) {
    mma_tf32_1688(d, al, bh0, bh1);
    mma_tf32_1688(d, ah, bl0, bl1);
    mma_tf32_1688(d, ah, bh0, bh1);
}

// An m16n8 accumulator fragment (lane = 4 g + t holds rows g, g+8 and columns
// 2t, 2t+1) reused as an m16n8k8 A fragment.  The contraction index is
// permuted -- logical k = t is column 2t, logical k = t + 4 is column 2t + 1 --
// and every B fragment below uses the same permutation, so the product is
// unchanged and no value moves between lanes.
__device__ __forceinline__ void acc_as_a(const float (&c)[4], uint32_t (&hi)[4], uint32_t (&lo)[4]) {
    split_tf32(c[0], hi[0], lo[0]);  // row g,   k = t
    split_tf32(c[2], hi[1], lo[1]);  // row g+8, k = t
    split_tf32(c[1], hi[2], lo[2]);  // row g,   k = t + 4
    split_tf32(c[3], hi[3], lo[3]);  // row g+8, k = t + 4
}

template <typename T>
__device__ __forceinline__ float2 ld2f(const T *p);
template <>
__device__ __forceinline__ float2 ld2f<float>(const float *p) {
    return *reinterpret_cast<const float2 *>(p);
}
template <>
__device__ __forceinline__ float2 ld2f<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}
template <>
__device__ __forceinline__ float2 ld2f<__half>(const __half *p) {
    return __half22float2(*reinterpret_cast<const __half2 *>(p));
}

// ------------------------------------------------------------ chunk-local part
// One CTA per (b, hv, chunk): Gram products, decay products, the unit
// lower-triangular inverse, and the tape capture of k_log / g_log.
template <typename TIn, int DK>
__global__ void __launch_bounds__(kCkLocalThreads)
chunk_local_kernel(const ChunkArgs a) {
    constexpr int C = kCkC;
    constexpr int KS = DK + 1;   // f32 row stride: row u of a warp lands on bank u
    constexpr int CS = C + 1;
    extern __shared__ __align__(16) unsigned char smem[];
    float *sk = reinterpret_cast<float *>(smem);
    float *sq = sk + C * KS;
    float *sA = sq + C * KS;     // A[t][u], u <= t
    float *sKK = sA + C * CS;    // k_t . k_u
    float *sKQ = sKK + C * CS;   // k_u . q_t
    float *sW = sKQ + C * CS;    // W = (I + N)^-1
    float *sg = sW + C * CS;     // effective g (1 on inactive steps)
    float *sb = sg + C;          // effective beta (0 on inactive steps)
    float *sG = sb + C;          // Gam_t

    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t nch = a.nchunks;
    const int64_t n = blockIdx.x / nch;
    const int64_t c = blockIdx.x - n * nch;
    const int64_t b = n / a.Hv, hv = n - b * a.Hv;
    const int64_t hk = a.tiled_gqa ? hv % a.Hk : hv / (a.Hv / a.Hk);
    const int64_t t0 = c * C;
    const int tcnt = (int)min((int64_t)C, a.T - t0);
    const unsigned bits = chunk_bits(a.mask ? a.mask + b * a.T + t0 : nullptr, tcnt, lane);

    const TIn *kp = static_cast<const TIn *>(a.k);
    const TIn *qp = static_cast<const TIn *>(a.q);
    const TIn *gp = static_cast<const TIn *>(a.g);
    const TIn *bp = static_cast<const TIn *>(a.beta);

    // k / q rows of active steps, widened; rows of inactive steps are zero
    for (int i = tid; i < C * DK; i += kCkLocalThreads) {
        const int tt = i / DK, x = i - tt * DK;
        float kv = 0.f, qv = 0.f;
        if ((bits >> tt) & 1u) {
            const int64_t off = ((b * a.T + t0 + tt) * a.Hk + hk) * DK + x;
            kv = ld_f32(kp + off);
            qv = ld_f32(qp + off);
        }
        sk[tt * KS + x] = kv;
        sq[tt * KS + x] = qv;
    }
    if (tid < C) {
        const bool on = (bits >> tid) & 1u;
        const int64_t gi = (b * a.T + t0 + tid) * a.Hv + hv;
        sg[tid] = on ? ld_f32(gp + gi) : 1.f;
        sb[tid] = on ? ld_f32(bp + gi) : 0.f;
    }
    __syncthreads();

    // one (t, u) pair per thread: Gram entries and the decay product A[t][u]
    {
        const int t = tid >> 4, u = tid & 15;
        float kk = 0.f, kq = 0.f;
#pragma unroll 8
        for (int x = 0; x < DK; ++x) {
            const float ku = sk[u * KS + x];
            kk = fmaf(sk[t * KS + x], ku, kk);
            kq = fmaf(sq[t * KS + x], ku, kq);
        }
        sKK[t * CS + u] = kk;
        sKQ[t * CS + u] = kq;
        float p = 1.f;
        for (int x = u + 1; x <= t; ++x) p *= sg[x];
        sA[t * CS + u] = u <= t ? p : 0.f;
        if (u == 0) {
            float G = 1.f;
            for (int x = 0; x <= t; ++x) G *= sg[x];
            sG[t] = G;
        }
    }
    __syncthreads();

    // W = (I + N)^-1 by forward substitution, one column u per thread:
    // W[t][u] = -sum_{u <= x < t} N[t][x] W[x][u],  N[t][x] = beta_t A[t][x] KK[t][x]
    if (tid < C) {
        const int u = tid;
        for (int t = 0; t < C; ++t) {
            float w;
            if (t < u) {
                w = 0.f;
            } else if (t == u) {
                w = 1.f;
            } else {
                float acc = 0.f;
                for (int x = u; x < t; ++x)
                    acc = fmaf(sb[t] * sA[t * CS + x] * sKK[t * CS + x], sW[x * CS + u], acc);
                w = -acc;
            }
            sW[t * CS + u] = w;
        }
    }
    __syncthreads();

    float *ws = a.workspace + (n * nch + c) * kCkWsFloats;
    {
        const int t = tid >> 4, u = tid & 15;
        ws[t * C + u] = u <= t ? sW[t * CS + u] * sb[u] : 0.f;            // Wb
        ws[C * C + t * C + u] = u <= t ? sA[t * CS + u] * sKQ[t * CS + u] : 0.f;  // Mq
        if (tid < C) ws[2 * C * C + tid] = sG[tid];                        // Gam
        if (tid < C) ws[2 * C * C + C + tid] = sA[(C - 1) * CS + tid];     // aC
    }

    // tape capture: k_log rows and g_log of the active steps
    if (a.k_log) {
        TIn *klp = static_cast<TIn *>(a.k_log);
        for (int i = tid; i < C * DK; i += kCkLocalThreads) {
            const int tt = i / DK, x = i - tt * DK;
            if ((bits >> tt) & 1u)
                klp[((b * a.T + t0 + tt) * a.Hv + hv) * DK + x] =
                    kp[((b * a.T + t0 + tt) * a.Hk + hk) * DK + x];
        }
    }
    if (a.g_log && tid < tcnt && ((bits >> tid) & 1u)) {
        const int64_t gi = (b * a.T + t0 + tid) * a.Hv + hv;
        static_cast<TIn *>(a.g_log)[gi] = gp[gi];
    }
}

// ------------------------------------------------------------ sequential part
template <typename TIn, int DK>
__global__ void __launch_bounds__(32 * kCkWarps)
chunk_scan_kernel(const ChunkArgs a) {
    constexpr int C = kCkC;
    constexpr int KPW = DK / kCkWarps;   // state columns per warp
    constexpr int NJ = KPW / 8;          // 8-column blocks per warp
    constexpr int KS = ck_kstride(DK);
    constexpr int ES = (int)sizeof(TIn);
    constexpr int VS = ck_vstride(ES);
    constexpr int PS = kCkPartStride;
    extern __shared__ __align__(16) unsigned char smem[];

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int64_t n = blockIdx.x / a.row_blocks;
    const int64_t rb = blockIdx.x - n * a.row_blocks;
    const int64_t b = n / a.Hv, hv = n - b * a.Hv;
    const int64_t hk = a.tiled_gqa ? hv % a.Hk : hv / (a.Hv / a.Hk);
    const int64_t row0 = rb * kCkRows;
    const int vlim = (int)min((int64_t)kCkRows, a.Dv - row0);
    const int cw = warp * KPW;           // first state column of this warp
    const int64_t nch = a.nchunks;

    const size_t slot_bytes = ck_slot_bytes(DK, ES);
    auto slotK = [&](int sl) { return reinterpret_cast<TIn *>(smem + sl * slot_bytes); };
    auto slotQ = [&](int sl) { return slotK(sl) + C * KS; };
    auto slotV = [&](int sl) {
        return reinterpret_cast<TIn *>(smem + sl * slot_bytes + align16((size_t)2 * C * KS * ES));
    };
    auto slotW = [&](int sl) {
        return reinterpret_cast<float *>(smem + sl * slot_bytes + align16((size_t)2 * C * KS * ES) +
                                         align16((size_t)C * VS * ES));
    };
    float *part = reinterpret_cast<float *>(smem + 3 * slot_bytes);  // [2][warps][16][PS]

    const TIn *qp = static_cast<const TIn *>(a.q);
    const TIn *kp = static_cast<const TIn *>(a.k);
    const TIn *vp = static_cast<const TIn *>(a.v);

    // ---- issue chunk cc into ring slot cc % 3 (an empty group past the end).
    // Rows of inactive steps are zeroed, never copied: every product of the
    // chunk multiplies them (by zero coefficients, which must not meet NaN).
    auto issue = [&](int64_t cc) {
        if (cc < nch) {
            const int sl = (int)(cc % 3);
            const int64_t t0 = cc * C;
            const int tcnt = (int)min((int64_t)C, a.T - t0);
            const unsigned bits = chunk_bits(a.mask ? a.mask + b * a.T + t0 : nullptr, tcnt, lane);
            if (bits != 0xffffu) {
                for (int i = tid; i < C * (DK / 4); i += nthr) {
                    const int tt = i / (DK / 4), x = (i - tt * (DK / 4)) * 4;
                    if (!((bits >> tt) & 1u)) {
                        TIn *kr = slotK(sl) + tt * KS + x;
                        TIn *qr = slotQ(sl) + tt * KS + x;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            kr[e] = Elem<TIn>::from_f32(0.f);
                            qr[e] = Elem<TIn>::from_f32(0.f);
                        }
                    }
                }
                for (int i = tid; i < C * kCkRows; i += nthr) {
                    const int tt = i / kCkRows, r = i - tt * kCkRows;
                    if (!((bits >> tt) & 1u)) slotV(sl)[tt * VS + r] = Elem<TIn>::from_f32(0.f);
                }
            }
            const int64_t kq_off = ((b * a.T + t0) * a.Hk + hk) * DK;
            async_rows_to<TIn>(slotK(sl), KS, kp + kq_off, a.Hk * DK, tcnt, DK, DK, bits, tid, nthr);
            async_rows_to<TIn>(slotQ(sl), KS, qp + kq_off, a.Hk * DK, tcnt, DK, DK, bits, tid, nthr);
            const int64_t v_off = ((b * a.T + t0) * a.Hv + hv) * a.Dv + row0;
            if (a.vec_v && vlim == kCkRows) {
                async_rows_to<TIn>(slotV(sl), VS, vp + v_off, a.Hv * a.Dv, tcnt, kCkRows, kCkRows,
                                   bits, tid, nthr);
            } else {
                for (int i = tid; i < tcnt * kCkRows; i += nthr) {
                    const int tt = i / kCkRows, r = i - tt * kCkRows;
                    if ((bits >> tt) & 1u)
                        slotV(sl)[tt * VS + r] =
                            r < vlim ? vp[v_off + tt * a.Hv * a.Dv + r] : Elem<TIn>::from_f32(0.f);
                }
            }
            const float *wsrc = a.workspace + (n * nch + cc) * kCkWsFloats;
            for (int i = tid; i < kCkWsFloats / 4; i += nthr) cp_async16(slotW(sl) + 4 * i, wsrc + 4 * i);
        }
        cp_async_commit();
    };

    // ---- the state slice of this warp: rows g, g+8; columns cw + 8j + 2t, +1
    float S[NJ][4];
    {
        const float *s_in = a.state_in + (n * a.Dv + row0) * DK;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int col = cw + 8 * j + 2 * t;
            float2 lo = make_float2(0.f, 0.f), hi = make_float2(0.f, 0.f);
            if (g < vlim) lo = __ldcs(reinterpret_cast<const float2 *>(s_in + g * DK + col));
            if (g + 8 < vlim) hi = __ldcs(reinterpret_cast<const float2 *>(s_in + (g + 8) * DK + col));
            S[j][0] = lo.x;
            S[j][1] = lo.y;
            S[j][2] = hi.x;
            S[j][3] = hi.y;
        }
    }

    issue(0);
    issue(1);
    cp_async_wait_group<1>();
    __syncthreads();

    TIn *yp = static_cast<TIn *>(a.y);
    TIn *dp = static_cast<TIn *>(a.delta_log);

    for (int64_t c = 0; c < nch; ++c) {
        const int sl = (int)(c % 3);
        const int64_t t0 = c * C;
        const int tcnt = (int)min((int64_t)C, a.T - t0);
        const TIn *cK = slotK(sl);
        const TIn *cQ = slotQ(sl);
        const TIn *cV = slotV(sl);
        const float *cW = slotW(sl);
        const float *Wb = cW, *Mq = cW + C * C, *Gam = cW + 2 * C * C, *aC = cW + 2 * C * C + C;

        // ---- P (this warp's columns): [Gam K ; Gam Q] rows as B (n = step),
        // the state as A (k = column)
        float P[4][4] = {};  // n-tiles: K steps 0-7, K 8-15, Q 0-7, Q 8-15
        {
            const float gam0 = Gam[g], gam1 = Gam[8 + g];
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                uint32_t ah[4], al[4];
                acc_as_a(S[j], ah, al);
                const int col = cw + 8 * j + 2 * t;
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const TIn *X = nt < 2 ? cK : cQ;
                    const int step = 8 * (nt & 1) + g;
                    const float gm = (nt & 1) ? gam1 : gam0;
                    const float2 x = ld2f<TIn>(X + step * KS + col);
                    uint32_t bh0, bl0, bh1, bl1;
                    split_tf32(gm * x.x, bh0, bl0);
                    split_tf32(gm * x.y, bh1, bl1);
                    mma3_tf32(P[nt], ah, al, bh0, bh1, bl0, bl1);
                }
            }
        }
        float *mypart = part + ((c & 1) * kCkWarps + warp) * kCkRows * PS;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            *reinterpret_cast<float2 *>(mypart + g * PS + 8 * nt + 2 * t) = make_float2(P[nt][0], P[nt][1]);
            *reinterpret_cast<float2 *>(mypart + (g + 8) * PS + 8 * nt + 2 * t) =
                make_float2(P[nt][2], P[nt][3]);
        }
        cp_async_wait_group<0>();
        __syncthreads();  // partials of chunk c and the inputs of chunk c+1 are visible
        issue(c + 2);

        // ---- sum the four partials (P_k for everyone, P_q for the y warp)
        const float *pc = part + (c & 1) * kCkWarps * kCkRows * PS;
        const bool ywarp = warp == 0;
        float Pk[2][4] = {}, Pq[2][4] = {};
#pragma unroll
        for (int w = 0; w < kCkWarps; ++w) {
            const float *pw = pc + w * kCkRows * PS;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float2 u0 = *reinterpret_cast<const float2 *>(pw + g * PS + 8 * nt + 2 * t);
                const float2 u1 = *reinterpret_cast<const float2 *>(pw + (g + 8) * PS + 8 * nt + 2 * t);
                Pk[nt][0] += u0.x;
                Pk[nt][1] += u0.y;
                Pk[nt][2] += u1.x;
                Pk[nt][3] += u1.y;
                if (ywarp) {
                    const float2 w0 = *reinterpret_cast<const float2 *>(pw + g * PS + 16 + 8 * nt + 2 * t);
                    const float2 w1 =
                        *reinterpret_cast<const float2 *>(pw + (g + 8) * PS + 16 + 8 * nt + 2 * t);
                    Pq[nt][0] += w0.x;
                    Pq[nt][1] += w0.y;
                    Pq[nt][2] += w1.x;
                    Pq[nt][3] += w1.y;
                }
            }
        }

        // ---- R = V^T - P_k;  D = R Wb^T (every warp: D is MMA-2's A operand)
        float D[2][4] = {};
        {
            uint32_t rh[2][4], rl[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int s0 = 8 * i + 2 * t;
                float r[4];
                r[0] = Elem<TIn>::to_f32(cV[s0 * VS + g]) - Pk[i][0];
                r[1] = Elem<TIn>::to_f32(cV[(s0 + 1) * VS + g]) - Pk[i][1];
                r[2] = Elem<TIn>::to_f32(cV[s0 * VS + g + 8]) - Pk[i][2];
                r[3] = Elem<TIn>::to_f32(cV[(s0 + 1) * VS + g + 8]) - Pk[i][3];
                acc_as_a(r, rh[i], rl[i]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float2 w = *reinterpret_cast<const float2 *>(Wb + (8 * nt + g) * C + 8 * i + 2 * t);
                    uint32_t bh0, bl0, bh1, bl1;
                    split_tf32(w.x, bh0, bl0);
                    split_tf32(w.y, bh1, bl1);
                    mma3_tf32(D[nt], rh[i], rl[i], bh0, bh1, bl0, bl1);
                }
            }
        }
        uint32_t dh[2][4], dl[2][4];
        acc_as_a(D[0], dh[0], dl[0]);
        acc_as_a(D[1], dh[1], dl[1]);

        const unsigned bits = chunk_bits(a.mask ? a.mask + b * a.T + t0 : nullptr, tcnt, lane);
        if (ywarp) {
            // ---- Y = P_q + D Mq^T, stored for active steps of live rows
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float2 m = *reinterpret_cast<const float2 *>(Mq + (8 * nt + g) * C + 8 * i + 2 * t);
                    uint32_t bh0, bl0, bh1, bl1;
                    split_tf32(m.x, bh0, bl0);
                    split_tf32(m.y, bh1, bl1);
                    mma3_tf32(Pq[nt], dh[i], dl[i], bh0, bh1, bl0, bl1);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s = 8 * nt + 2 * t + (e & 1), r = g + 8 * (e >> 1);
                    if (s < tcnt && ((bits >> s) & 1u) && r < vlim)
                        yp[((b * a.T + t0 + s) * a.Hv + hv) * a.Dv + row0 + r] = Elem<TIn>::from_f32(Pq[nt][e]);
                }
        } else if (warp == 1 && dp) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s = 8 * nt + 2 * t + (e & 1), r = g + 8 * (e >> 1);
                    if (s < tcnt && ((bits >> s) & 1u) && r < vlim)
                        dp[((b * a.T + t0 + s) * a.Hv + hv) * a.Dv + row0 + r] = Elem<TIn>::from_f32(D[nt][e]);
                }
        }

        // ---- S = Gam_{C-1} S + D (aC K): B = aC-scaled k rows (k = step, n = column)
        {
            const float gl = Gam[C - 1];
            float ac[2][2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                ac[i][0] = aC[8 * i + 2 * t];
                ac[i][1] = aC[8 * i + 2 * t + 1];
            }
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) S[j][e] *= gl;
                const int col = cw + 8 * j + g;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int s0 = 8 * i + 2 * t;
                    uint32_t bh0, bl0, bh1, bl1;
                    split_tf32(ac[i][0] * Elem<TIn>::to_f32(cK[s0 * KS + col]), bh0, bl0);
                    split_tf32(ac[i][1] * Elem<TIn>::to_f32(cK[(s0 + 1) * KS + col]), bh1, bl1);
                    mma3_tf32(S[j], dh[i], dl[i], bh0, bh1, bl0, bl1);
                }
            }
        }
    }
    cp_async_wait_group<0>();

    {
        float *s_out = a.state_out + (n * a.Dv + row0) * DK;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int col = cw + 8 * j + 2 * t;
            if (g < vlim) __stcs(reinterpret_cast<float2 *>(s_out + g * DK + col), make_float2(S[j][0], S[j][1]));
            if (g + 8 < vlim)
                __stcs(reinterpret_cast<float2 *>(s_out + (g + 8) * DK + col), make_float2(S[j][2], S[j][3]));
        }
    }
}

template <typename TIn, int DK>
cudaError_t launch_chunk_dk(const ChunkArgs &a, cudaStream_t st) {
    auto local = chunk_local_kernel<TIn, DK>;
    auto scan = chunk_scan_kernel<TIn, DK>;
    const size_t lsm = chunk_local_smem_bytes(DK);
    const size_t ssm = chunk_scan_smem_bytes(DK, (int)sizeof(TIn));
    cudaError_t e;
    if (lsm > 48 * 1024) {
        e = cudaFuncSetAttribute(local, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lsm);
        if (e != cudaSuccess) return e;
    }
    if (ssm > 48 * 1024) {
        e = cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssm);
        if (e != cudaSuccess) return e;
    }
    const int64_t tiles = a.B * a.Hv;
    local<<<(unsigned)(tiles * a.nchunks), kCkLocalThreads, lsm, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    scan<<<(unsigned)(tiles * a.row_blocks), 32 * kCkWarps, ssm, st>>>(a);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_chunk_type(int dk, const ChunkArgs &a, cudaStream_t st) {
    switch (dk) {
    case 32: return launch_chunk_dk<TIn, 32>(a, st);
    case 64: return launch_chunk_dk<TIn, 64>(a, st);
    case 128: return launch_chunk_dk<TIn, 128>(a, st);
    case 192: return launch_chunk_dk<TIn, 192>(a, st);
    case 256: return launch_chunk_dk<TIn, 256>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn
