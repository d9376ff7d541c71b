// tile.cuh -- how a CTA holds its slice of one (b, hv) state tile in registers.
//
// The page kernels give every state row s[Dk] its own 32-lane simdgroup
// ("metaltile-std gated_delta_replay.rs", DISPATCH INVARIANTS: grid
// [1, Dv, B*Hv], threadgroup [32,1,1], Dk/32 entries per lane) and reduce
// each dot product across all 32 lanes.  Here a group of L lanes shares a
// block of RT = 8 consecutive rows:
//
//   lane = gi * L + j        (gi: row group of the warp, j: 0..L-1)
//   local rows of (warp, gi) = warp * RW + gi * RT + m,  m in [0, RT)
//   lane j holds the float4 chunks j, j+L, j+2L, ... of each of its rows
//
// (L = 8 for Dk <= 128, L = 16 above).  A warp-wide 16-byte load of one chunk
// index touches whole 128-byte lines; a 16-byte shared-memory load of k or q
// serves L distinct chunks per quarter-warp; and a transposed butterfly
// reduction over the L lanes leaves each lane the two dot products (s.k, s.q)
// of exactly one row (RT == L) or one of the two (RT == L/2), so the scalar
// part of a step runs once per row instead of once per lane.  Rows are
// independent (the recurrence never mixes value rows), so a tile may be split
// across CTAs by rows.
#pragma once

#include "common.cuh"

namespace gdn {

// A thread layout: Dk columns per row, L lanes per row group, RT rows per
// thread.  DefaultLayout<DK> is the one the library launches.
template <int DK_, int L_, int RT_>
struct TileLayout {
    static constexpr int DK = DK_;
    static constexpr int L = L_;                        // lanes per row group
    static constexpr int RT = RT_;                      // rows per thread
    static constexpr int NCH = DK / (4 * L);            // float4 chunks per lane per row
    static constexpr int GPW = 32 / L;                  // row groups per warp
    static constexpr int RW = GPW * RT;                 // rows per warp
    static constexpr int MAX_WARPS = (128 / RW) < 1 ? 1 : (128 / RW);  // a CTA covers <= 128 rows
    static constexpr int LOG2L = L == 4 ? 2 : (L == 8 ? 3 : (L == 16 ? 4 : 5));
    static constexpr int REDV = 2 * RT / L;             // dot values a lane keeps after the reduce
    static constexpr int STATE = RT * DK / L;           // state floats per thread
    static constexpr int MAX_THREADS = 32 * MAX_WARPS;
    // resident CTAs per SM the register budget is sized for
    static constexpr int MIN_BLOCKS =
        STATE <= 32 ? 4 : (STATE <= 64 ? (MAX_THREADS >= 256 ? 2 : 3) : (MAX_THREADS >= 256 ? 1 : 2));
    static_assert(DK % (4 * L) == 0, "Dk must be a multiple of 4 L");
    static_assert(RT == L || 2 * RT == L, "one or two lanes per row after the reduce");
};

// lanes per row group: 8 for Dk <= 64, 16 above (64, 96 or 128 state floats
// per thread at Dk = 128, 192, 256)
template <int DK>
struct DefaultLayout {
    using type = TileLayout<DK, (DK <= 64 ? 8 : 16), 8>;
};

template <class Lay>
using Slice = float4[Lay::RT][Lay::NCH];

// Index of the first float4 of state row (n, dv).
__device__ __forceinline__ int64_t row_base4(int64_t n, int64_t Dv, int64_t dv, int dk) {
    return ((n * Dv + dv) * dk) >> 2;
}

// Four consecutive state entries of type TS as f32 (exact), and back
// (rounded to nearest-even for 2-byte types): 16-byte pieces for f32, 8-byte
// pieces otherwise, at the same entry positions.
template <typename TS>
__device__ __forceinline__ float4 ld_state4(const TS *p, int64_t i4) {
    if constexpr (sizeof(TS) == 4) {
        return __ldcs(reinterpret_cast<const float4 *>(p) + i4);
    } else {
        const uint2 raw = __ldcs(reinterpret_cast<const uint2 *>(p) + i4);
        const TS *e = reinterpret_cast<const TS *>(&raw);
        return make_float4(Elem<TS>::to_f32(e[0]), Elem<TS>::to_f32(e[1]), Elem<TS>::to_f32(e[2]),
                           Elem<TS>::to_f32(e[3]));
    }
}
template <typename TS>
__device__ __forceinline__ void st_state4(TS *p, int64_t i4, float4 x) {
    if constexpr (sizeof(TS) == 4) {
        __stcs(reinterpret_cast<float4 *>(p) + i4, x);
    } else {
        uint2 raw;
        TS *e = reinterpret_cast<TS *>(&raw);
        e[0] = Elem<TS>::from_f32(x.x);
        e[1] = Elem<TS>::from_f32(x.y);
        e[2] = Elem<TS>::from_f32(x.z);
        e[3] = Elem<TS>::from_f32(x.w);
        __stcs(reinterpret_cast<uint2 *>(p) + i4, raw);
    }
}

// Load this thread's rows of the tile (zeros for rows past Dv).
template <class Lay, typename TS>
__device__ __forceinline__ void load_rows(Slice<Lay> &s, const TS *state, int64_t n, int64_t Dv,
                                          int64_t row_first, int j) {
#pragma unroll
    for (int m = 0; m < Lay::RT; ++m) {
        const int64_t dv = row_first + m;
        const bool live = dv < Dv;
        const int64_t base = live ? row_base4(n, Dv, dv, Lay::DK) : 0;
#pragma unroll
        for (int c = 0; c < Lay::NCH; ++c)
            s[m][c] = live ? ld_state4(state, base + c * Lay::L + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// s <- s * G for the whole slice, then store rows < Dv (streaming stores).
template <class Lay, typename TS>
__device__ __forceinline__ void store_rows(Slice<Lay> &s, float G, TS *state, int64_t n,
                                           int64_t Dv, int64_t row_first, int j) {
    const float2 g2 = make_float2(G, G);
    const bool scale = G != 1.f;
#pragma unroll
    for (int m = 0; m < Lay::RT; ++m) {
        const int64_t dv = row_first + m;
        if (dv >= Dv) continue;
        const int64_t base = row_base4(n, Dv, dv, Lay::DK);
#pragma unroll
        for (int c = 0; c < Lay::NCH; ++c) {
            float4 x = s[m][c];
            if (scale) x = cat4(fmul2(lo2(x), g2), fmul2(hi2(x), g2));
            st_state4(state, base + c * Lay::L + j, x);
        }
    }
}

// Fold the scale into the slice: s <- s * G (the direct-form fallback).
template <class Lay>
__device__ __forceinline__ void rescale_rows(Slice<Lay> &s, float G) {
    const float2 g2 = make_float2(G, G);
#pragma unroll
    for (int m = 0; m < Lay::RT; ++m)
#pragma unroll
        for (int c = 0; c < Lay::NCH; ++c)
            s[m][c] = cat4(fmul2(lo2(s[m][c]), g2), fmul2(hi2(s[m][c]), g2));
}

// Rank-1 update of the slice: s[m] <- fma(k, d[m], s[m]) (one rounding per entry).
template <class Lay>
__device__ __forceinline__ void rank1_update(Slice<Lay> &s, const float4 (&kk)[Lay::NCH],
                                             const float (&d)[Lay::RT]) {
#pragma unroll
    for (int c = 0; c < Lay::NCH; ++c) {
#pragma unroll
        for (int m = 0; m < Lay::RT; ++m) {
            const float2 dd = make_float2(d[m], d[m]);
            s[m][c] = cat4(ffma2(lo2(kk[c]), dd, lo2(s[m][c])), ffma2(hi2(kk[c]), dd, hi2(s[m][c])));
        }
    }
}

// This lane's chunks of a staged f32 row (k, q or k_log).
template <class Lay>
__device__ __forceinline__ void lane_chunks(float4 (&out)[Lay::NCH], const float *row, int j) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
#pragma unroll
    for (int c = 0; c < Lay::NCH; ++c) out[c] = r4[c * Lay::L + j];
}

// Transposed butterfly over the L lanes of a row group: on entry v[2m],
// v[2m+1] are this lane's partial (s.k, s.q) of row m; on exit v[0 .. REDV)
// holds the group sums of entries [REDV * j, REDV * j + REDV) of that list.
// Each level halves the list: lanes with the level's bit set keep the upper
// half.  (Keeping the rows in natural order keeps the one-time state
// load / store coalesced; a per-lane row permutation would remove the
// selects but splits every 128-byte line across eight rows.)
template <class Lay>
__device__ __forceinline__ void transpose_reduce(float (&v)[2 * Lay::RT], int j) {
#pragma unroll
    for (int lvl = 0; lvl < Lay::LOG2L; ++lvl) {
        const int o = Lay::L >> (lvl + 1);
        const int half = (2 * Lay::RT) >> (lvl + 1);
        const bool upper = (j & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
}

// ----------------------------------------------------- the decay-scale schedule
// Per-step scalars of a chunk, computed once (serially, by one thread) and
// read by every thread: the new scale G' = G * g, 1 / G' (1 on direct steps),
// and whether the step folds the scale into the state (bit tt of `direct`).
// Record and replay both call this function, so they see identical values.
struct StepScalars {
    float Gp, inv, beta, kq;
};

// Run by one whole warp.  Lane 0 walks the chunk's active steps in order
// (G' = G g; fold when G' leaves range) and the lanes then take the
// correctly rounded reciprocals of their own step in parallel.  Returns the
// direct-step bits on every lane; G is updated on every lane.
__device__ __forceinline__ unsigned scale_schedule(StepScalars *sc, const float *g, unsigned act,
                                                   int tcnt, float &G, int lane) {
    unsigned direct = 0u;
    float Gl = G;
    if (lane == 0) {
        for (int tt = 0; tt < tcnt; ++tt) {
            if (!((act >> tt) & 1u)) continue;
            const float Gp = __fmul_rn(Gl, g[tt]);
            const bool dir = !scale_in_range(Gp);
            sc[tt].Gp = Gp;
            direct |= (dir ? 1u : 0u) << tt;
            Gl = dir ? 1.f : Gp;
        }
    }
    __syncwarp();
    direct = __shfl_sync(0xffffffffu, direct, 0);
    G = __shfl_sync(0xffffffffu, Gl, 0);
    if (lane < tcnt && ((act >> lane) & 1u))
        sc[lane].inv = ((direct >> lane) & 1u) ? 1.f : __frcp_rn(sc[lane].Gp);
    return direct;
}

// ------------------------------------------------------------ async staging
// Chunks of timesteps are copied global -> shared with cp.async (16-byte
// pieces, L2 only), two slots deep: the copies of chunk c+1 are in flight
// while chunk c is computed.  The waits are the hardware's cp.async group
// waits on this thread's own copies.

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
// Wait until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Bit tt set when step t0+tt (tt < tcnt <= 32) is on: every lane of every
// warp evaluates the same ballot (mask NULL: all on).
__device__ __forceinline__ unsigned chunk_bits(const uint32_t *mask_row, int tcnt, int lane) {
    if (!mask_row) return tcnt >= 32 ? 0xffffffffu : ((1u << tcnt) - 1u);
    const bool on = lane < tcnt && __ldg(mask_row + lane) != 0u;
    return __ballot_sync(0xffffffffu, on);
}

// Copy rows tt < tcnt with bit tt set: row tt of `row_elems` T elements from
// src + tt * stride to dst + tt * row_elems.  row_elems * sizeof(T) and the
// addresses are multiples of 16 bytes; pieces at or past `limit` elements of
// a row are skipped (the ragged end of a row block).
template <typename T>
__device__ __forceinline__ void async_rows(T *dst, const T *src, int64_t stride, int tcnt,
                                           int row_elems, int limit, unsigned bits, int tid,
                                           int nthr) {
    constexpr int VEC = 16 / sizeof(T);
    const int vpr = row_elems / VEC;
    for (int i = tid; i < tcnt * vpr; i += nthr) {
        const int tt = i / vpr;
        const int x = (i - tt * vpr) * VEC;
        if (((bits >> tt) & 1u) && x < limit) cp_async16(dst + tt * row_elems + x, src + tt * stride + x);
    }
}

// As async_rows, with a destination row stride (elements) that may differ
// from the row length (padded shared-memory rows).
template <typename T>
__device__ __forceinline__ void async_rows_to(T *dst, int dst_stride, const T *src, int64_t stride,
                                              int tcnt, int row_elems, int limit, unsigned bits,
                                              int tid, int nthr) {
    constexpr int VEC = 16 / sizeof(T);
    const int vpr = row_elems / VEC;
    for (int i = tid; i < tcnt * vpr; i += nthr) {
        const int tt = i / vpr;
        const int x = (i - tt * vpr) * VEC;
        if (((bits >> tt) & 1u) && x < limit) cp_async16(dst + tt * dst_stride + x, src + tt * stride + x);
    }
}

// Widen n (a multiple of 16 bytes of T) raw elements to f32, zeroing
// elements whose index within a row of `row_elems` is at or past `limit`.
template <typename T>
__device__ __forceinline__ void widen_block(float *dst, const T *src, int n, int row_elems,
                                            int limit, int tid, int nthr) {
    constexpr int VEC = 16 / sizeof(T);
    for (int i = tid * VEC; i < n; i += nthr * VEC) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(src + i);
        widen16<T>(dst + i, raw);
        if (limit < row_elems) {
            const int col = i % row_elems;
            for (int e = 0; e < VEC; ++e)
                if (col + e >= limit) dst[i + e] = 0.f;
        }
    }
}

}  // namespace gdn
