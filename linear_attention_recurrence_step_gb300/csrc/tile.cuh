// tile.cuh -- how a CTA holds its slice of one (b, hv) state tile in registers.
//
// The page kernels give every state row s[Dk] its own 32-lane simdgroup
// ("metaltile-std gated_delta_replay.rs", DISPATCH INVARIANTS: grid
// [1, Dv, B*Hv], threadgroup [32,1,1], Dk/32 entries per lane) and reduce
// each dot product across all 32 lanes.  Here a row is shared by only L = 4
// lanes, and a thread holds RT rows:
//
//   lane = gi * L + j        (gi: row group 0..7 of the warp, j: 0..L-1)
//   local row of (warp, gi, m) = warp * RW + gi + m * GPW,  m in [0, RT)
//   lane j holds the float4 chunks j, j+L, j+2L, ... of each of its rows
//
// so a dot product is a 2-level xor-shuffle over 4 lanes, the k / q chunks a
// thread reads from shared memory serve RT rows, and a warp-wide 16-byte
// load of one chunk index touches 8 rows x 64 contiguous bytes (whole
// 32-byte sectors).  Rows are independent (the recurrence never mixes
// value rows), so a tile may be split across CTAs by rows.
#pragma once

#include "common.cuh"

namespace gdn {

template <int DK> struct RowsPerThread;  // RT * DK / 4 state floats per thread
template <> struct RowsPerThread<32> { static constexpr int value = 4; };
template <> struct RowsPerThread<64> { static constexpr int value = 4; };
template <> struct RowsPerThread<128> { static constexpr int value = 4; };
template <> struct RowsPerThread<192> { static constexpr int value = 2; };
template <> struct RowsPerThread<256> { static constexpr int value = 2; };

template <int DK>
struct TileLayout {
    static constexpr int L = 4;                       // lanes per row
    static constexpr int RT = RowsPerThread<DK>::value;
    static constexpr int NCH = DK / (4 * L);          // float4 chunks per lane per row
    static constexpr int GPW = 32 / L;                // row groups per warp
    static constexpr int RW = GPW * RT;               // rows per warp
    static constexpr int MAX_WARPS = 4;               // CTA size cap (launch bounds)
    static_assert(DK % (4 * L) == 0, "Dk must be a multiple of 16");
};

constexpr int kMaxThreads = 128;

// Resident CTAs per SM the register budget is sized for: a thread holding
// 128 state floats needs more than the 168 registers that 3 CTAs of 128
// threads allow, so those layouts run 2 CTAs per SM.
template <int DK>
struct MinBlocks {
    static constexpr int value = (TileLayout<DK>::RT * DK / 4 >= 128) ? 2 : 3;
};

// Index of the first float4 of state row (n, dv).
__device__ __forceinline__ int64_t row_base4(int64_t n, int64_t Dv, int64_t dv, int dk) {
    return ((n * Dv + dv) * dk) >> 2;
}

// Load this thread's rows of the tile (zeros for rows past Dv).
template <int DK>
__device__ __forceinline__ void load_rows(float4 (&s)[TileLayout<DK>::RT][TileLayout<DK>::NCH],
                                          const float *state, int64_t n, int64_t Dv,
                                          int64_t row0, int warp, int gi, int j) {
    using Lay = TileLayout<DK>;
    const float4 *p = reinterpret_cast<const float4 *>(state);
#pragma unroll
    for (int m = 0; m < Lay::RT; ++m) {
        const int64_t dv = row0 + warp * Lay::RW + gi + m * Lay::GPW;
        const bool live = dv < Dv;
        const int64_t base = live ? row_base4(n, Dv, dv, DK) : 0;
#pragma unroll
        for (int c = 0; c < Lay::NCH; ++c)
            s[m][c] = live ? __ldcs(p + base + c * Lay::L + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// s <- s * G for the whole slice, then store rows < Dv (streaming stores).
template <int DK>
__device__ __forceinline__ void store_rows(float4 (&s)[TileLayout<DK>::RT][TileLayout<DK>::NCH],
                                           float G, float *state, int64_t n, int64_t Dv,
                                           int64_t row0, int warp, int gi, int j) {
    using Lay = TileLayout<DK>;
    float4 *p = reinterpret_cast<float4 *>(state);
    const float2 g2 = make_float2(G, G);
    const bool scale = G != 1.f;
#pragma unroll
    for (int m = 0; m < Lay::RT; ++m) {
        const int64_t dv = row0 + warp * Lay::RW + gi + m * Lay::GPW;
        if (dv >= Dv) continue;
        const int64_t base = row_base4(n, Dv, dv, DK);
#pragma unroll
        for (int c = 0; c < Lay::NCH; ++c) {
            float4 x = s[m][c];
            if (scale) x = cat4(fmul2(lo2(x), g2), fmul2(hi2(x), g2));
            __stcs(p + base + c * Lay::L + j, x);
        }
    }
}

// Fold the scale into the slice: s <- s * G (the direct-form fallback).
template <int DK>
__device__ __forceinline__ void rescale_rows(float4 (&s)[TileLayout<DK>::RT][TileLayout<DK>::NCH],
                                             float G) {
    using Lay = TileLayout<DK>;
    const float2 g2 = make_float2(G, G);
#pragma unroll
    for (int m = 0; m < Lay::RT; ++m)
#pragma unroll
        for (int c = 0; c < Lay::NCH; ++c)
            s[m][c] = cat4(fmul2(lo2(s[m][c]), g2), fmul2(hi2(s[m][c]), g2));
}

// Rank-1 update of the slice: s[m] <- fma(k, d[m], s[m]) (one rounding per entry).
template <int DK>
__device__ __forceinline__ void rank1_update(float4 (&s)[TileLayout<DK>::RT][TileLayout<DK>::NCH],
                                             const float *k_row, const float (&d)[TileLayout<DK>::RT],
                                             int j) {
    using Lay = TileLayout<DK>;
    const float4 *k4 = reinterpret_cast<const float4 *>(k_row);
#pragma unroll
    for (int c = 0; c < Lay::NCH; ++c) {
        const float4 kk = k4[c * Lay::L + j];
#pragma unroll
        for (int m = 0; m < Lay::RT; ++m) {
            const float2 dd = make_float2(d[m], d[m]);
            s[m][c] = cat4(ffma2(lo2(kk), dd, lo2(s[m][c])), ffma2(hi2(kk), dd, hi2(s[m][c])));
        }
    }
}

// Stage the key rows (k, q or k_log) of a chunk into shared memory as f32:
// row tt of the chunk is src[first_off + tt * step_stride .. + DK).  Rows of
// masked-off steps (mask_row[tt] == 0) are skipped; mask_row may be NULL.
template <typename T, int DK>
__device__ __forceinline__ void stage_key_rows(float *dst, const T *src, int64_t first_off,
                                               int64_t step_stride, int tcnt,
                                               const uint32_t *mask_row, int tid, int nthr) {
    constexpr int VEC = 16 / sizeof(T);
    constexpr int VPR = DK / VEC;
    for (int i = tid; i < tcnt * VPR; i += nthr) {
        const int tt = i / VPR;
        const int x = i - tt * VPR;
        if (mask_row && __ldg(mask_row + tt) == 0u) continue;
        const uint4 raw =
            __ldg(reinterpret_cast<const uint4 *>(src + first_off + tt * step_stride + x * VEC));
        widen16<T>(dst + tt * DK + x * VEC, raw);
    }
}

}  // namespace gdn
