// chunk.cuh -- chunked prefill: the record recurrence of "metaltile-std
// gated_delta_replay.rs" (kernel gated_delta_step_record) regrouped over
// chunks of C = 16 steps so that long calls run as dense products on the
// tensor cores (warp-level mma.sync, tf32 operands, f32 accumulate), in
// float32 accuracy.
//
// Within a chunk (steps 0..C-1, state s_in at entry, inactive steps given
// g = 1 and beta = 0) the step
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
// sequential part, chunk_scan_kernel, walks the chunks of one tile's row
// block with four MMA products per chunk:
//     P  = S_in [K ; Q]^T, then scaled by Gam per step (rows x 2C, over Dk)
//     D  = (V^T - P_k) Wb^T           (the deltas, contraction over C)
//     Y  = P_q + D Mq^T               (contraction over C)
//     S  = Gam_{C-1} S_in + (D aC) K  (rows x Dk, contraction over C)
//
// Accuracy: every product runs as three tf32 MMAs (a_hi b_lo + a_lo b_hi +
// a_hi b_hi, each operand split x = hi + lo with hi = x truncated to tf32 and
// lo = x - hi exact in f32), about 20 significant bits per product with f32
// accumulation; bf16 / f16 k and q are exact in tf32, so with those inputs
// the products with a k / q operand take two.  The state stays f32 in the
// accumulator fragments for the whole launch.
//
// Work split: a CTA owns 16 state rows of one (b, hv) tile and four warps
// split the Dk columns (each holds 16 rows x Dk/4 of the state).  The partial
// products P of the four warps are summed through shared memory once per
// chunk; that exchange is the kernel's only CTA barrier per chunk.  The
// outputs are spread over the warps: two write the delta_log rows and two
// the y rows, eight steps each.  Inputs of chunk c+2 are copied with
// cp.async into a three-slot ring while chunk c is computed, so the barrier
// of chunk c also publishes chunk c+1.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tile.cuh"

namespace gdn {

constexpr int kCkC = 16;           // timesteps per chunk
constexpr int kCkWarps = 4;        // warps per scan CTA (Dk split four ways)
constexpr int kCkThreads = 32 * kCkWarps;
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
    return 3 * ck_slot_bytes(dk, esize) + (size_t)2 * kCkWarps * kCkRows * kCkPartStride * 4;
}
constexpr int kCkHeadsPerPass = 4;  // value heads of one key head processed side by side
__host__ __device__ constexpr size_t chunk_local_smem_bytes(int dk) {
    return (size_t)2 * kCkC * (dk + 4) * 4 + (size_t)(4 + 2 * kCkHeadsPerPass) * kCkC * (kCkC + 1) * 4 +
           (size_t)3 * kCkHeadsPerPass * kCkC * 4;
}

// ------------------------------------------------------------ tf32 products
// x ~ hi + lo: the tensor core reads an f32 register as tf32 by dropping its
// 13 low mantissa bits (truncation, checked on the GPU for m16n8k8 tf32), so
// hi is x itself (read as trunc(x)) and lo = x - trunc(x), exact in f32 and
// below 2^-10 |x|; the tensor core reads lo's tf32 part in turn, which leaves
// |error| < 2^-20 |x|.
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    hi = __float_as_uint(x);
    lo = __float_as_uint(x - __uint_as_float(hi & 0xffffe000u));
}
__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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

// One 16-byte piece of T widened to f32 (exact).
template <typename T>
__device__ __forceinline__ void widen_piece(uint4 raw, float (&out)[16 / sizeof(T)]);
template <>
__device__ __forceinline__ void widen_piece<float>(uint4 raw, float (&out)[4]) {
    out[0] = __uint_as_float(raw.x);
    out[1] = __uint_as_float(raw.y);
    out[2] = __uint_as_float(raw.z);
    out[3] = __uint_as_float(raw.w);
}
template <>
__device__ __forceinline__ void widen_piece<__nv_bfloat16>(uint4 raw, float (&out)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
template <>
__device__ __forceinline__ void widen_piece<__half>(uint4 raw, float (&out)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        out[2 * i] = f.x;
        out[2 * i + 1] = f.y;
    }
}

// ------------------------------------------------------------ chunk-local part
// One CTA per (b, hk, chunk): the Gram products of key head hk (shared by the
// G value heads that read it), then for each of those value heads the decay
// products, the unit lower-triangular inverse, the workspace block and the
// tape capture of k_log / g_log.
template <typename TIn, int DK>
__global__ void __launch_bounds__(kCkLocalThreads)
chunk_local_kernel(const ChunkArgs a) {
    pdl_trigger();
    pdl_wait();
    constexpr int C = kCkC;
    constexpr int KS = DK + 4;   // f32 row stride: float4 rows u land 4 banks apart
    constexpr int CS = C + 1;
    constexpr int VEC = 16 / (int)sizeof(TIn);
    // bf16 / f16 values are exact in tf32: their Gram products take one MMA
    constexpr bool kTf32Exact = !std::is_same<TIn, float>::value;
    extern __shared__ __align__(16) unsigned char smem[];
    float *sk = reinterpret_cast<float *>(smem);
    float *sq = sk + C * KS;
    float *sGr = sq + C * KS;    // [half of Dk][KK, KQ][C][CS]
    constexpr int HP = kCkHeadsPerPass;
    float *sA = sGr + 4 * C * CS;  // [HP][C][CS] A[t][u], u <= t (zero above)
    float *sN = sA + HP * C * CS;  // [HP][C][CS] N[t][u], u < t (zero elsewhere)
    float *sg = sN + HP * C * CS;  // [HP][C] effective g (1 on inactive steps)
    float *sb = sg + HP * C;       // [HP][C] effective beta (0 on inactive steps)
    float *sG = sb + HP * C;       // [HP][C] Gam_t

    // k_t . k_u and k_u . q_t: the two halves of the contraction, summed in a
    // fixed order
    auto KK = [&](int t, int u) { return sGr[t * CS + u] + sGr[(2 * C + t) * CS + u]; };
    auto KQ = [&](int t, int u) { return sGr[(C + t) * CS + u] + sGr[(3 * C + t) * CS + u]; };

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t nch = a.nchunks;
    const int64_t m = blockIdx.x / nch;          // b * Hk + hk
    const int64_t c = blockIdx.x - m * nch;
    const int64_t b = m / a.Hk, hk = m - b * a.Hk;
    const int64_t G = a.Hv / a.Hk;
    const int64_t t0 = c * C;
    const int tcnt = (int)min((int64_t)C, a.T - t0);
    auto hv_at = [&](int64_t h) { return a.tiled_gqa ? hk + h * a.Hk : hk * G + h; };

    const TIn *kp = static_cast<const TIn *>(a.k);
    const TIn *qp = static_cast<const TIn *>(a.q);
    const TIn *gp = static_cast<const TIn *>(a.g);
    const TIn *bp = static_cast<const TIn *>(a.beta);

    // ---- every load of the chunk is issued before any of them is waited
    // for: the k / q pieces of the steps inside the call, g and beta of the
    // first pass of value heads, then the mask words.
    constexpr int NPIECE = C * DK / VEC;  // 16-byte pieces of a chunk's k (or q) rows
    constexpr int NPC = (NPIECE + kCkLocalThreads - 1) / kCkLocalThreads;
    uint4 kraw[NPC], qraw[NPC];
#pragma unroll
    for (int j = 0; j < NPC; ++j) {
        const int i = tid + j * kCkLocalThreads;
        kraw[j] = qraw[j] = make_uint4(0u, 0u, 0u, 0u);
        const int tt = i / (DK / VEC), x = (i - tt * (DK / VEC)) * VEC;
        if (i < NPIECE && tt < tcnt) {
            const int64_t off = ((b * a.T + t0 + tt) * a.Hk + hk) * DK + x;
            kraw[j] = *reinterpret_cast<const uint4 *>(kp + off);
            qraw[j] = *reinterpret_cast<const uint4 *>(qp + off);
        }
    }
    const int nh0 = (int)min((int64_t)kCkHeadsPerPass, G);
    TIn g0 = Elem<TIn>::from_f32(1.f), b0 = Elem<TIn>::from_f32(0.f);
    if (tid < nh0 * C && tid % C < tcnt) {
        const int64_t gi = (b * a.T + t0 + tid % C) * a.Hv + hv_at(tid / C);
        g0 = gp[gi];
        b0 = bp[gi];
    }
    const unsigned bits = chunk_bits(a.mask ? a.mask + b * a.T + t0 : nullptr, tcnt, lane);

    // k / q rows widened into shared memory (rows of inactive steps zero);
    // k_log rows of the active steps copied bit for bit from the same pieces
#pragma unroll
    for (int j = 0; j < NPC; ++j) {
        const int i = tid + j * kCkLocalThreads;
        if (i >= NPIECE) break;
        const int tt = i / (DK / VEC), x = (i - tt * (DK / VEC)) * VEC;
        const bool on = (bits >> tt) & 1u;
        float kv[VEC], qv[VEC];
        widen_piece<TIn>(kraw[j], kv);
        widen_piece<TIn>(qraw[j], qv);
#pragma unroll
        for (int e = 0; e < VEC; e += 4) {
            *reinterpret_cast<float4 *>(sk + tt * KS + x + e) =
                on ? make_float4(kv[e], kv[e + 1], kv[e + 2], kv[e + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4 *>(sq + tt * KS + x + e) =
                on ? make_float4(qv[e], qv[e + 1], qv[e + 2], qv[e + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (a.k_log && on) {
            TIn *klp = static_cast<TIn *>(a.k_log);
            for (int64_t h = 0; h < G; ++h)
                *reinterpret_cast<uint4 *>(klp + ((b * a.T + t0 + tt) * a.Hv + hv_at(h)) * DK + x) = kraw[j];
        }
    }
    __syncthreads();

    // ---- Gram blocks on the tensor cores: per product (KK, KQ) two m16n8
    // tiles (steps t 0-15 x u 0-7, 8-15), each contracted over the two halves
    // of Dk: eight tile-halves, one per warp.  A = k or q rows (m = step t),
    // B = k rows (n = step u), both read straight from the f32 rows; f32 rows
    // take three tf32 products (hi / lo split), about 20 significant bits.
    static_assert(kCkLocalThreads == 256 && kCkC == 16, "one tile-half per warp");
    {
        constexpr int KH = DK / 2;
        const int g8 = lane >> 2, t4 = lane & 3;
        const int h = warp >> 2, which = (warp >> 1) & 1, nt = warp & 1;
        const float *Ar = (which ? sq : sk) + g8 * KS + h * KH + t4;
        const float *Br = sk + (8 * nt + g8) * KS + h * KH + t4;
        float dm[4] = {0.f, 0.f, 0.f, 0.f}, ds[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KH / 8; ++ks) {
            const float av[4] = {Ar[8 * ks], Ar[8 * KS + 8 * ks], Ar[8 * ks + 4], Ar[8 * KS + 8 * ks + 4]};
            uint32_t ah[4], al[4], bh0, bl0, bh1, bl1;
#pragma unroll
            for (int e = 0; e < 4; ++e) split_tf32(av[e], ah[e], al[e]);
            split_tf32(Br[8 * ks], bh0, bl0);
            split_tf32(Br[8 * ks + 4], bh1, bl1);
            if constexpr (!kTf32Exact) {
                mma_tf32_1688(ds, al, bh0, bh1);
                mma_tf32_1688(ds, ah, bl0, bl1);
            }
            mma_tf32_1688(dm, ah, bh0, bh1);
        }
        float *dst = sGr + ((2 * h + which) * C + g8) * CS + 8 * nt + 2 * t4;
        dst[0] = dm[0] + ds[0];
        dst[1] = dm[1] + ds[1];
        dst[8 * CS] = dm[2] + ds[2];
        dst[8 * CS + 1] = dm[3] + ds[3];
    }

    // the value heads that read key head hk, up to kCkHeadsPerPass at a time:
    // decay products, the inverse and the workspace block of each head run
    // side by side (one 16-thread group per head for the inverse)
    for (int64_t i0 = 0; i0 < G; i0 += kCkHeadsPerPass) {
        const int nh = (int)min((int64_t)kCkHeadsPerPass, G - i0);
        auto hv_of = [&](int i) { return hv_at(i0 + i); };
        if (tid < nh * C) {
            // g and beta of the pass (the first pass's were loaded up front);
            // g_log of the active steps
            const int i = tid / C, tt = tid - i * C;
            const bool on = (bits >> tt) & 1u;
            const int64_t gi = (b * a.T + t0 + tt) * a.Hv + hv_of(i);
            const TIn gr = i0 == 0 ? g0 : (on ? gp[gi] : g0);
            const TIn br = i0 == 0 ? b0 : (on ? bp[gi] : b0);
            sg[i * C + tt] = on ? Elem<TIn>::to_f32(gr) : 1.f;
            sb[i * C + tt] = on ? Elem<TIn>::to_f32(br) : 0.f;
            if (a.g_log && on) static_cast<TIn *>(a.g_log)[gi] = gr;
        }
        __syncthreads();  // g, beta of these heads; Gram entries (first pass)
        if (tid < nh * C) {
            // column u of head i, walked down the steps: A[t][u] = A[t-1][u] g_t
            // from A[u][u] = 1 (the products in the same order as a walk from
            // g_{u+1} to g_t), N below the diagonal, Gam_t = g_0 ... g_t
            const int i = tid / C, u = tid - i * C;
            const float *gh = sg + i * C, *bh = sb + i * C;
            float p = 1.f, gm = 1.f;
#pragma unroll
            for (int t = 0; t < C; ++t) {
                const float gt = gh[t];
                if (t > u) p *= gt;
                sA[(i * C + t) * CS + u] = t >= u ? p : 0.f;
                sN[(i * C + t) * CS + u] = t > u ? bh[t] * p * KK(t, u) : 0.f;
                gm *= gt;
                if (u == 0) sG[i * C + t] = gm;
            }
        }
        __syncthreads();

        // workspace block of the pass's head i: a base for (b, chunk) and a
        // stride per value head
        float *const ws_b = a.workspace + (b * a.Hv * nch + c) * kCkWsFloats;
        auto ws_of = [&](int i) { return ws_b + hv_of(i) * (nch * kCkWsFloats); };
        if (tid < nh * C) {
            // W = (I + N)^-1 of head i, one column u per thread, held in registers:
            // W[t][u] = -sum_{x < t} N[t][x] W[x][u]  (W[x][u] = 0 for x < u)
            const int i = tid / C, u = tid - i * C;
            const float *Nh = sN + i * C * CS;
            float w[C];
#pragma unroll
            for (int t = 0; t < C; ++t) {
                float acc = 0.f;
#pragma unroll
                for (int x = 0; x < t; ++x) acc = fmaf(Nh[t * CS + x], w[x], acc);
                w[t] = t < u ? 0.f : (t == u ? 1.f : -acc);
            }
            const float bu = sb[i * C + u];
            float *ws = ws_of(i);
#pragma unroll
            for (int t = 0; t < C; ++t) ws[t * C + u] = w[t] * bu;  // Wb
        }
        const int ft = tid - nh * C;  // the other threads: Mq, Gam, aC
        if (ft >= 0) {
            const int nf = kCkLocalThreads - nh * C;
            for (int e = ft; e < nh * C * C; e += nf) {
                const int i = e / (C * C), j = e - i * C * C, t = j >> 4, u = j & 15;
                float *ws = ws_of(i);
                ws[C * C + j] = u <= t ? sA[(i * C + t) * CS + u] * KQ(t, u) : 0.f;  // Mq
            }
            for (int e = ft; e < nh * 2 * C; e += nf) {
                const int i = e / (2 * C), j = e - i * 2 * C;
                float *ws = ws_of(i);
                ws[2 * C * C + j] = j < C ? sG[i * C + j] : sA[(i * C + C - 1) * CS + (j - C)];  // Gam, aC
            }
        }
        __syncthreads();  // sg / sb / sA / sN are rewritten for the next heads
    }
}

// ------------------------------------------------------------ sequential part
template <typename TIn, int DK>
__global__ void __launch_bounds__(kCkThreads)
chunk_scan_kernel(const ChunkArgs a) {
    pdl_trigger();
    pdl_wait();
    constexpr int C = kCkC;
    constexpr int KPW = DK / kCkWarps;   // state columns per warp
    // bf16 / f16 values are exact in tf32: the low terms of k / q operands
    // are zero, and their products are skipped
    constexpr bool kTf32Exact = !std::is_same<TIn, float>::value;
    constexpr int NJ = KPW / 8;          // 8-column blocks per warp
    constexpr int KS = ck_kstride(DK);
    constexpr int ES = (int)sizeof(TIn);
    constexpr int VEC = 16 / ES;         // elements per 16-byte piece
    constexpr int VPR = DK / VEC;        // 16-byte pieces per k / q row
    constexpr int VS = ck_vstride(ES);
    constexpr int VVR = kCkRows / VEC;   // 16-byte pieces per staged v row
    constexpr int PS = kCkPartStride;
    extern __shared__ __align__(16) unsigned char smem[];

    const int tid = threadIdx.x;
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

    constexpr size_t kSlot = ck_slot_bytes(DK, ES);
    constexpr size_t kOffV = align16((size_t)2 * C * KS * ES);
    constexpr size_t kOffW = kOffV + align16((size_t)C * VS * ES);
    auto slotK = [&](int sl) { return reinterpret_cast<TIn *>(smem + sl * kSlot); };
    auto slotQ = [&](int sl) { return slotK(sl) + C * KS; };
    auto slotV = [&](int sl) { return reinterpret_cast<TIn *>(smem + sl * kSlot + kOffV); };
    auto slotW = [&](int sl) { return reinterpret_cast<float *>(smem + sl * kSlot + kOffW); };
    float *part = reinterpret_cast<float *>(smem + 3 * kSlot);         // [2][warps][16][PS]

    const TIn *qp = static_cast<const TIn *>(a.q);
    const TIn *kp = static_cast<const TIn *>(a.k);
    const TIn *vp = static_cast<const TIn *>(a.v);
    const bool vec_v = a.vec_v && vlim == kCkRows;

    // ---- mask bits of a chunk: lane tt's mask word, loaded a chunk before
    // its bits are formed, so no step of the loop waits on a mask load
    auto mask_word = [&](int64_t cc) {
        const int64_t t = cc * C + lane;
        return a.mask && cc < nch && lane < C && t < a.T ? __ldg(a.mask + b * a.T + t) : 1u;
    };
    auto bits_of = [&](int64_t cc, uint32_t word) {  // the same answer on every lane
        if (cc >= nch) return 0u;
        const int tcnt = (int)min((int64_t)C, a.T - cc * C);
        if (!a.mask) return tcnt >= 32 ? 0xffffffffu : ((1u << tcnt) - 1u);
        return __ballot_sync(0xffffffffu, lane < tcnt && word != 0u);
    };

    // ---- issue chunk cc into ring slot sl (an empty group past the end).
    // Rows of inactive steps are zeroed, never copied: every product of the
    // chunk multiplies them (by zero coefficients, which must not meet NaN).
    auto issue = [&](int64_t cc, int sl, unsigned bits) {
        if (cc < nch) {
            const int64_t t0 = cc * C;
            const int tcnt = (int)min((int64_t)C, a.T - t0);
            const TIn *ksrc = kp + ((b * a.T + t0) * a.Hk + hk) * DK;
            const TIn *qsrc = qp + ((b * a.T + t0) * a.Hk + hk) * DK;
            const int64_t kq_stride = a.Hk * DK;
            TIn *kd = slotK(sl), *qd = slotQ(sl);
#pragma unroll
            for (int ii = 0; ii < (C * VPR + kCkThreads - 1) / kCkThreads; ++ii) {
                const int i = tid + ii * kCkThreads;
                if ((C * VPR) % kCkThreads != 0 && i >= C * VPR) break;
                const int tt = i / VPR, x = (i - tt * VPR) * VEC;
                if ((bits >> tt) & 1u) {
                    cp_async16(kd + tt * KS + x, ksrc + tt * kq_stride + x);
                    cp_async16(qd + tt * KS + x, qsrc + tt * kq_stride + x);
                } else {
                    *reinterpret_cast<uint4 *>(kd + tt * KS + x) = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4 *>(qd + tt * KS + x) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            const TIn *vsrc = vp + ((b * a.T + t0) * a.Hv + hv) * a.Dv + row0;
            const int64_t v_stride = a.Hv * a.Dv;
            TIn *vd = slotV(sl);
            if (vec_v) {
                if (tid < C * VVR) {
                    const int tt = tid / VVR, x = (tid - tt * VVR) * VEC;
                    if ((bits >> tt) & 1u)
                        cp_async16(vd + tt * VS + x, vsrc + tt * v_stride + x);
                    else
                        *reinterpret_cast<uint4 *>(vd + tt * VS + x) = make_uint4(0u, 0u, 0u, 0u);
                }
            } else {
                for (int i = tid; i < C * kCkRows; i += kCkThreads) {
                    const int tt = i / kCkRows, r = i - tt * kCkRows;
                    vd[tt * VS + r] = ((bits >> tt) & 1u) && r < vlim ? vsrc[tt * v_stride + r]
                                                                      : Elem<TIn>::from_f32(0.f);
                }
            }
            const float *wsrc = a.workspace + (n * nch + cc) * kCkWsFloats;
            float *wd = slotW(sl);
#pragma unroll
            for (int ii = 0; ii < (kCkWsFloats / 4 + kCkThreads - 1) / kCkThreads; ++ii) {
                const int i = tid + ii * kCkThreads;
                if (i < kCkWsFloats / 4) cp_async16(wd + 4 * i, wsrc + 4 * i);
            }
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

    // bits of chunks c and c + 1, and the mask word of chunk c + 2
    unsigned bits_c = bits_of(0, mask_word(0)), bits_c1 = bits_of(1, mask_word(1));
    uint32_t word_c2 = mask_word(2);
    issue(0, 0, bits_c);
    issue(1, 1, bits_c1);
    cp_async_wait_group<1>();
    __syncthreads();

    // Outputs of a chunk, spread over the four warps: warp w writes the
    // delta_log (w < 2) or y (w >= 2) rows of steps 8 (w & 1) .. 8 (w & 1) + 7.
    static_assert(kCkWarps == 4, "the output roles assume four warps");
    TIn *yp = static_cast<TIn *>(a.y);
    TIn *dp = static_cast<TIn *>(a.delta_log);
    const bool ywarp = warp >= 2;
    const int oh = warp & 1;  // this warp's n-tile: steps 8 oh .. 8 oh + 7
    const bool out_warp = ywarp || dp != nullptr;
    TIn *const outp = ywarp ? yp : dp;

    int sl = 0, sl2 = 2;  // ring slots of chunks c and c + 2
    for (int64_t c = 0; c < nch; ++c) {
        const int64_t t0 = c * C;
        const int tcnt = (int)min((int64_t)C, a.T - t0);
        const TIn *cK = slotK(sl);
        const TIn *cQ = slotQ(sl);
        const TIn *cV = slotV(sl);
        const float *cW = slotW(sl);
        const float *Wb = cW, *Mq = cW + C * C, *Gam = cW + 2 * C * C, *aC = cW + 2 * C * C + C;

        // ---- P (this warp's columns, unscaled): [K ; Q] rows as B (n = step),
        // the state as A (k = column).  Main and small tf32 terms accumulate
        // in separate registers (two shorter dependency chains).
        // n-tiles: K steps 0-7, K 8-15, Q 0-7, Q 8-15.  The three tf32 terms
        // accumulate separately: twelve independent chains of NJ products.
        float Pm[4][4] = {}, Pa[4][4] = {}, Pb[4][4] = {};
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            uint32_t ah[4], al[4];
            acc_as_a(S[j], ah, al);
            const int col = cw + 8 * j + 2 * t;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const TIn *X = nt < 2 ? cK : cQ;
                const float2 x = ld2f<TIn>(X + (8 * (nt & 1) + g) * KS + col);
                uint32_t bh0, bl0, bh1, bl1;
                split_tf32(x.x, bh0, bl0);
                split_tf32(x.y, bh1, bl1);
                mma_tf32_1688(Pa[nt], al, bh0, bh1);
                if constexpr (!kTf32Exact) mma_tf32_1688(Pb[nt], ah, bl0, bl1);
                mma_tf32_1688(Pm[nt], ah, bh0, bh1);
            }
        }
        float *mypart = part + ((c & 1) * kCkWarps + warp) * kCkRows * PS;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) p[e] = Pm[nt][e] + (Pa[nt][e] + Pb[nt][e]);
            *reinterpret_cast<float2 *>(mypart + g * PS + 8 * nt + 2 * t) = make_float2(p[0], p[1]);
            *reinterpret_cast<float2 *>(mypart + (g + 8) * PS + 8 * nt + 2 * t) = make_float2(p[2], p[3]);
        }
        cp_async_wait_group<0>();
        __syncthreads();  // partials of chunk c and the inputs of chunk c+1 are visible
        const unsigned bits_c2 = bits_of(c + 2, word_c2);
        word_c2 = mask_word(c + 3);  // used one chunk from now
        issue(c + 2, sl2, bits_c2);

        // ---- sum the four partials and scale by Gam (P_k for every warp; the
        // y warps also P_q of their n-tile)
        const float *pc = part + (c & 1) * kCkWarps * kCkRows * PS;
        float Pk[2][4] = {}, Pq[4] = {};
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
            }
            if (ywarp) {
                const float2 w0 = *reinterpret_cast<const float2 *>(pw + g * PS + 16 + 8 * oh + 2 * t);
                const float2 w1 = *reinterpret_cast<const float2 *>(pw + (g + 8) * PS + 16 + 8 * oh + 2 * t);
                Pq[0] += w0.x;
                Pq[1] += w0.y;
                Pq[2] += w1.x;
                Pq[3] += w1.y;
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float2 gm = *reinterpret_cast<const float2 *>(Gam + 8 * nt + 2 * t);
            Pk[nt][0] *= gm.x;
            Pk[nt][1] *= gm.y;
            Pk[nt][2] *= gm.x;
            Pk[nt][3] *= gm.y;
        }
        {
            const float2 gm = *reinterpret_cast<const float2 *>(Gam + 8 * oh + 2 * t);
            Pq[0] *= gm.x;
            Pq[1] *= gm.y;
            Pq[2] *= gm.x;
            Pq[3] *= gm.y;
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
            float Da[2][4] = {}, Db[2][4] = {};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float2 w = *reinterpret_cast<const float2 *>(Wb + (8 * nt + g) * C + 8 * i + 2 * t);
                    uint32_t bh0, bl0, bh1, bl1;
                    split_tf32(w.x, bh0, bl0);
                    split_tf32(w.y, bh1, bl1);
                    mma_tf32_1688(Da[nt], rl[i], bh0, bh1);
                    mma_tf32_1688(Db[nt], rh[i], bl0, bl1);
                    mma_tf32_1688(D[nt], rh[i], bh0, bh1);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) D[nt][e] += Da[nt][e] + Db[nt][e];
        }

        const unsigned bits = bits_c;
        if (out_warp) {
            float o[4];
            if (ywarp) {
                // ---- Y = P_q + D Mq^T for this warp's n-tile
                uint32_t dh[2][4], dl[2][4];
                acc_as_a(D[0], dh[0], dl[0]);
                acc_as_a(D[1], dh[1], dl[1]);
                // the three tf32 terms in separate accumulators (two-deep chains)
                float Ym[4] = {}, Ya[4] = {}, Yb[4] = {};
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float2 mq = *reinterpret_cast<const float2 *>(Mq + (8 * oh + g) * C + 8 * i + 2 * t);
                    uint32_t bh0, bl0, bh1, bl1;
                    split_tf32(mq.x, bh0, bl0);
                    split_tf32(mq.y, bh1, bl1);
                    mma_tf32_1688(Ya, dl[i], bh0, bh1);
                    mma_tf32_1688(Yb, dh[i], bl0, bl1);
                    mma_tf32_1688(Ym, dh[i], bh0, bh1);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] = Pq[e] + (Ym[e] + (Ya[e] + Yb[e]));
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] = oh ? D[1][e] : D[0][e];
            }
            // straight from the fragments: lane (g, t) holds rows g, g + 8 of
            // steps 2t, 2t + 1, so each store writes four runs of 8 rows
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int s = 8 * oh + 2 * t + (e & 1), r = g + 8 * (e >> 1);
                if (s < tcnt && ((bits >> s) & 1u) && r < vlim)
                    outp[((b * a.T + t0 + s) * a.Hv + hv) * a.Dv + row0 + r] = Elem<TIn>::from_f32(o[e]);
            }
        }

        // ---- S = Gam_{C-1} S + (D aC) K: B = raw k rows (k = step, n = column)
        {
            uint32_t eh[2][4], el[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float2 ac = *reinterpret_cast<const float2 *>(aC + 8 * i + 2 * t);
                const float de[4] = {D[i][0] * ac.x, D[i][1] * ac.y, D[i][2] * ac.x, D[i][3] * ac.y};
                acc_as_a(de, eh[i], el[i]);
            }
            const float gl = Gam[C - 1];
            float Ua[NJ][4] = {}, Ub[NJ][4] = {};  // small tf32 terms, separate chains
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) S[j][e] *= gl;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int s0 = 8 * i + 2 * t;
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int col = cw + 8 * j + g;
                    uint32_t bh0, bl0, bh1, bl1;
                    split_tf32(Elem<TIn>::to_f32(cK[s0 * KS + col]), bh0, bl0);
                    split_tf32(Elem<TIn>::to_f32(cK[(s0 + 1) * KS + col]), bh1, bl1);
                    mma_tf32_1688(Ua[j], el[i], bh0, bh1);
                    if constexpr (!kTf32Exact) mma_tf32_1688(Ub[j], eh[i], bl0, bl1);
                    mma_tf32_1688(S[j], eh[i], bh0, bh1);
                }
            }
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) S[j][e] += Ua[j][e] + Ub[j][e];
        }
        sl = sl == 2 ? 0 : sl + 1;
        sl2 = sl2 == 2 ? 0 : sl2 + 1;
        bits_c = bits_c1;
        bits_c1 = bits_c2;
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
    e = launch_dependent(local, (unsigned)(a.B * a.Hk * a.nchunks), kCkLocalThreads, lsm, st, a);
    if (e != cudaSuccess) return e;
    return launch_dependent(scan, (unsigned)(a.B * a.Hv * a.row_blocks), kCkThreads, ssm, st, a);
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
