// record_tc.cuh -- the record kernel for calls of at most one 16-step chunk
// on the fifth-generation tensor cores (tcgen05.mma, accumulators in tensor
// memory), fed by TMA.  bf16 inputs, f32 state, Dk = 128, Dv a multiple of
// 128.
//
// The recurrence is the page's ("metaltile-std gated_delta_replay.rs",
// kernel gated_delta_step_record) regrouped over a chunk of C <= 16 steps
// exactly as in record_mma.cuh.  With the chunk-initial state S (rows = value
// rows dv, columns = Dk), per-step scales G'_t (the decay products, see
// scale_schedule) and d_t = delta_t / G'_t:
//     P   = S [K; Q]^T                         (128 rows x 32 step dots)
//     r_t = beta_t (v_t / G'_t - P_k[t]),      d = W r,   W = (I + N)^-1,
//           N[t][u] = beta_t (k_u . k_t) for u < t (both steps active)
//     b_t = P_q[t] + sum_{u<t} d_u (k_u . q_t),
//     delta_t = G'_t d_t,   y_t = G'_t b_t + delta_t (k_t . q_t)
//     S_out = G (S + D K)                       (G: the chunk's final scale)
//
// One work unit is a 128-row block of one (b, hv) state tile.  A persistent
// CTA per SM runs two warpgroups, each on its own sequence of units, and one
// preparation warp:
//   * the warpgroup's thread 0 issues TMA loads: the unit's f32 state rows
//     (four boxes of 32 columns, 128-byte swizzle) into the warpgroup's slot,
//     and the next unit's k / q rows (128-byte swizzle) and v rows into the
//     other of two input buffers;
//   * each thread owns one state row (= one tensor-memory lane): it copies
//     its row into the tensor-memory accumulator S (tcgen05.st) and rewrites
//     the slot in place as the bf16 hi + lo terms of the row (64-byte
//     swizzled K-major operand tiles), so that the f32 state enters the
//     products with 16 significant bits while S itself stays exact;
//   * thread 0 issues MMA1, 16 tcgen05.mma (kind::f16, M = 128, N = 32,
//     K = 16: the hi and lo terms against the k / q rows) into P in tensor
//     memory; the slot is then free for the next unit's state;
//   * the preparation warp computes, one unit ahead, the chunk's Gram
//     matrices k_u . k_t and k_u . q_t (mma.sync), W by forward substitution,
//     the step scales, and writes the k_log / g_log tape;
//   * each thread reads its row of P (tcgen05.ld), solves its row in FP32,
//     writes y and delta (coalesced: a step's 128 rows are contiguous), and
//     stores its d_t as bf16 hi + lo terms (the A operand of MMA2);
//   * thread 0 issues MMA2 (two tcgen05.mma, N = 128, K = 16) accumulating
//     D K onto S, and each thread reads back its final row, scales it by G
//     and writes it.
// Steps past T (zero-filled boxes) and masked steps are inactive: their rows
// of K enter MMA2 as zeros, their r and d are zero, and nothing of theirs is
// written, so whatever the caller left in masked slots never reaches an
// output.  A fold of the scale (G' out of range) takes the per-row serial
// solve, with S rescaled in tensor memory before MMA2.
// Every mbarrier wait is bounded; a warpgroup whose wait runs out writes NaN
// to its unit's state rows, raises the wait-expiry flag and stops.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "launch.h"
#include "record_mma.cuh"
#include "tma.cuh"

namespace gdn {

constexpr int kRtRows = 128;       // state rows per unit (tensor-memory lanes)
constexpr int kRtDk = 128;         // key dimension of this kernel
constexpr int kRtGroups = 2;       // warpgroups (units in flight) per CTA
constexpr int kRtThreads = 192 * kRtGroups;  // per warpgroup: four row warps, a preparation warp, an issuer warp
constexpr uint32_t kRtTmemCols = 512;   // S (128) + P (32) per warpgroup, 256 apart
constexpr long long kRtWaitCycles = 2000000000ll;  // default bound on an mbarrier wait (~1 s)

// per-warpgroup shared memory (bytes)
constexpr uint32_t kRtSlot = kRtRows * kRtDk * 4;           // f32 state rows; then A hi / lo
constexpr uint32_t kRtKq = 2 * kMmaChunk * kRtDk * 2;       // k and q rows (16 steps each)
constexpr uint32_t kRtV = kMmaChunk * kRtRows * 2;          // v rows of the unit
constexpr uint32_t kRtA2 = 2 * kRtRows * kMmaChunk * 2;     // d hi | d lo
constexpr uint32_t kRtB2 = kRtDk * kMmaChunk * 2;           // K^T (K-major)
// preparation block: W, KQ^T, KK, KQ (f32 16x16 each), step scalars, bits
constexpr uint32_t kRtPrep = 4 * 1024 + 16 * (uint32_t)sizeof(StepScalars) + 64 + 16;
constexpr uint32_t kRtPrepAl = 4608;
constexpr uint32_t kRtOffKq = kRtSlot;
constexpr uint32_t kRtOffV = kRtOffKq + 2 * kRtKq;
constexpr uint32_t kRtOffA2 = kRtOffV + 2 * kRtV;
constexpr uint32_t kRtOffB2 = kRtOffA2 + kRtA2;
constexpr uint32_t kRtOffPrep = kRtOffB2 + kRtB2;
constexpr uint32_t kRtGroupBytes = kRtOffPrep + 2 * kRtPrepAl;
// mbarriers per warpgroup: 0 state landed, 1-2 inputs landed [buf], 3 MMA1
// done, 4 MMA2 done, 5-6 preparation ready [buf], 7-8 unit finished [buf],
// 9 operand tiles written (pass), 10 d tiles written (solve), 11 never
// completed (the testing hook gdn_inject_wait_expiry waits on it)
constexpr int kRtBars = 12;
constexpr int kRtBarState = 0, kRtBarIn = 1, kRtBarMma1 = 3, kRtBarMma2 = 4, kRtBarPrep = 5,
              kRtBarDone = 7, kRtBarPass = 9, kRtBarSolve = 10, kRtBarNever = 11;
constexpr uint32_t kRtSmem = kRtGroups * kRtGroupBytes + kRtGroups * kRtBars * 8 + 16 + 1024;
static_assert(kRtPrep <= kRtPrepAl, "preparation block");
static_assert(kRtGroupBytes % 1024 == 0, "warpgroup region alignment");

// Preparation block layout (f32 indices).
struct RtPrep {
    float W[16 * 16];    // W[t][u], unit lower triangular
    float KQT[16 * 16];  // KQT[t][u] = k_u . q_t for u < t (both active), else 0
    float KK[16 * 16];   // KK[u][t] = k_u . k_t for u < t (both active), else 0
    float KQ[16 * 16];   // KQ[u][t] = k_u . q_t for u < t (both active), else 0
    StepScalars sc[16];
    float gv[16];        // the decays of the chunk's steps
    unsigned bits, direct;
    float gfinal;
};

// ------------------------------------------------------------ tcgen05 wrappers
// Shared-memory matrix descriptor: start, leading / stride byte offsets,
// version 1 (bits 46-48) and the swizzle layout (bits 61-63: 0 none,
// 2 128-byte, 4 64-byte).
__device__ __forceinline__ uint64_t rt_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return (uint64_t)((addr >> 4) & 0x3fffu) | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}
// Instruction descriptor of kind::f16 with bf16 A and B (both K-major), f32
// accumulator, M = 128, N = n.
__device__ __forceinline__ uint32_t rt_idesc_bf16(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kRtRows >> 4) << 24);
}
__device__ __forceinline__ void rt_mma(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(da), "l"(db), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void rt_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void rt_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void rt_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void rt_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void rt_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// 32 consecutive columns of this thread's tensor-memory lane.
__device__ __forceinline__ void rt_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// 16 lanes x 256 bits, four 8-column blocks: thread t receives (lane t/4:
// columns 2(t%4), 2(t%4)+1) and (lane 8 + t/4: the same columns) of each block.
__device__ __forceinline__ void rt_ld16x256_x4(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// 16 lanes x 256 bits, sixteen 8-column blocks (the layout of rt_ld16x256_x4).
__device__ __forceinline__ void rt_ld16x256_x16(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
                 : "r"(taddr));
}
__device__ __forceinline__ void rt_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// k / q tile of a unit: boxes of 16 steps x 64 columns (128-byte rows,
// 128-byte swizzle) at [k cols 0-63 | q cols 0-63 | k cols 64-127 | q cols
// 64-127], so that the 32 rows [k; q] of each 64-column half are one
// K-major operand with 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint32_t rt_kq_addr(uint32_t kq, bool isq, int s, int x) {
    return kq + (uint32_t)(x >> 6) * 4096u + (isq ? 2048u : 0u) + (uint32_t)s * 128u +
           ((uint32_t)(((x & 63) >> 3) ^ (s & 7)) << 4);
}

struct RecordTcArgs {
    RecordArgs a;
    int64_t nunits;         // B * Hv * (Dv / 128)
    unsigned *wait_flag;    // set to 1 when a bounded wait runs out
    long long wait_cycles;  // bound on the pipeline's waits (the drain after a
                            // failure always waits up to kRtWaitCycles)
    int inject_expiry;      // testing hook: one wait that nothing completes
};

__global__ void __launch_bounds__(kRtThreads, 1)
record_tc_kernel(const __grid_constant__ CUtensorMap tm_state, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_v,
                 const RecordTcArgs ta) {
    using T = __nv_bfloat16;
    constexpr int C = kMmaChunk;
    const RecordArgs &a = ta.a;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = sh_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *const gbase = smem_raw + (base - raw);
    auto gptr = [&](uint32_t s) { return gbase + (s - base); };  // generic pointer of a shared address

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // warps 0-3 / 4-7: the row warps of warpgroups 0 / 1; then one preparation
    // warp and one issuer warp per warpgroup
    const bool prep_warp = warp >= 4 * kRtGroups && warp < 5 * kRtGroups;
    const bool issuer_warp = warp >= 5 * kRtGroups;
    const int wg = issuer_warp ? warp - 5 * kRtGroups : prep_warp ? warp - 4 * kRtGroups : warp >> 2;
    const int r = tid & 127;  // state row / tensor-memory lane of this thread in its unit
    const uint32_t barbase = base + kRtGroups * kRtGroupBytes;
    auto bar = [&](int g, int i) { return barbase + (uint32_t)(g * kRtBars + i) * 8u; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gptr(barbase + kRtGroups * kRtBars * 8));

    const int tcnt = (int)a.T;  // <= C
    const uint32_t u_rb = (uint32_t)a.row_blocks, u_hv = (uint32_t)a.Hv, u_hk = (uint32_t)a.Hk,
                   u_g = (uint32_t)(a.Hv / a.Hk);
    struct Unit {
        uint32_t n, b, hv, hk, row0;
        bool valid;
    };
    auto unit_of = [&](int g, int64_t j) {
        const int64_t u = (int64_t)blockIdx.x + (2 * j + g) * (int64_t)gridDim.x;
        Unit d;
        d.valid = u < ta.nunits;
        const uint32_t uu = d.valid ? (uint32_t)u : 0u;
        d.n = uu / u_rb;
        d.row0 = (uu - d.n * u_rb) * kRtRows;
        d.b = d.n / u_hv;
        d.hv = d.n - d.b * u_hv;
        d.hk = a.tiled_gqa ? d.hv % u_hk : d.hv / u_g;
        return d;
    };

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         sh_addr(tmem_slot)),
                     "r"(kRtTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    if (tid == 0) {
        for (int g = 0; g < kRtGroups; ++g)
            for (int i = 0; i < kRtBars; ++i) {
                // arrivals: one from the thread that issues (or prepares), or one
                // per row warp
                const bool per_warp = i == kRtBarDone || i == kRtBarDone + 1 || i == kRtBarPass || i == kRtBarSolve;
                mbar_init(bar(g, i), per_warp ? 4u : 1u);
            }
        mbar_init_fence();
    }
    rt_fence_before();
    __syncthreads();
    rt_fence_after();
    const uint32_t tmem0 = *tmem_slot;
    // every CTA of the grid is resident and holds its tensor memory: the next
    // kernel may be scheduled; this one reads nothing the previous kernel
    // wrote before that kernel has completed
    pdl_trigger();
    pdl_wait();

    if (prep_warp) {
        // ================================================ preparation warp
        const T *gp = static_cast<const T *>(a.g);
        const T *bp = static_cast<const T *>(a.beta);
        T *klp = static_cast<T *>(a.k_log);
        T *glp = static_cast<T *>(a.g_log);
        const int g8 = lane >> 2, t4 = lane & 3, lm = lane >> 3, lr8 = lane & 7;
        bool ok = true;
        const int g = wg;
        // the step scalars of a unit (mask entry, decay, beta of step `lane`),
        // loaded one unit ahead
        uint32_t pre_m = 0u;
        float pre_g = 1.f, pre_b = 0.f;
        auto prefetch = [&](const Unit &d) {
            if (!d.valid) return;
            const int64_t bt0 = (int64_t)d.b * a.T;
            const bool lin = lane < tcnt;
            pre_m = lin ? (a.mask ? __ldg(a.mask + bt0 + lane) : 1u) : 0u;
            pre_g = lin ? ld_f32(gp + (bt0 + lane) * a.Hv + d.hv) : 1.f;
            pre_b = lin ? ld_f32(bp + (bt0 + lane) * a.Hv + d.hv) : 0.f;
        };
        Unit d = unit_of(g, 0);
        prefetch(d);
        for (int64_t j = 0; ok && d.valid; ++j) {
            const int buf = (int)(j & 1);
            const uint32_t gb = base + (uint32_t)g * kRtGroupBytes;
            const uint32_t kq = gb + kRtOffKq + buf * kRtKq;
            RtPrep *pp = reinterpret_cast<RtPrep *>(gptr(gb + kRtOffPrep + buf * kRtPrepAl));
            const int64_t bt0 = (int64_t)d.b * a.T;
            const bool lin = lane < tcnt;
            const float gv = pre_g, bv = pre_b;
            const unsigned bits = __ballot_sync(0xffffffffu, pre_m != 0u);
            const Unit dn = unit_of(g, j + 1);
            prefetch(dn);
            // this buffer's previous unit (j - 2) is finished; the k / q rows landed
            if (j >= 2) ok = mbar_wait_bounded(bar(g, kRtBarDone + buf), (uint32_t)(((j >> 1) - 1) & 1), ta.wait_cycles);
            ok = ok && mbar_wait_bounded(bar(g, kRtBarIn + buf), (uint32_t)((j >> 1) & 1), ta.wait_cycles);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            // Gram matrices KK[u][s] = k_u . k_s and KQ[u][s] = k_u . q_s (mma.sync)
            float kk[2][4] = {}, kqm[2][4] = {};
#pragma unroll
            for (int kt = 0; kt < kRtDk / 16; ++kt) {
                uint32_t ka[4], qa[4];
                // matrices: (steps 0-7, k lo), (steps 8-15, k lo), (0-7, k hi), (8-15, k hi)
                ldsm_x4_a(ka, rt_kq_addr(kq, false, lr8 + 8 * (lm & 1), 16 * kt + 8 * (lm >> 1)));
                ldsm_x4_a(qa, rt_kq_addr(kq, true, lr8 + 8 * (lm & 1), 16 * kt + 8 * (lm >> 1)));
                mma_bf16_16816(kk[0], ka, ka[0], ka[2]);
                mma_bf16_16816(kk[1], ka, ka[1], ka[3]);
                mma_bf16_16816(kqm[0], ka, qa[0], qa[2]);
                mma_bf16_16816(kqm[1], ka, qa[1], qa[3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int u = g8 + 8 * (e >> 1), s2 = 8 * nt + 2 * t4 + (e & 1);
                    // entries that involve a masked / absent step are exact zeros
                    const bool on = s2 > u && ((bits >> u) & 1u) && ((bits >> s2) & 1u);
                    pp->KK[u * C + s2] = on ? kk[nt][e] : 0.f;
                    pp->KQ[u * C + s2] = on ? kqm[nt][e] : 0.f;
                    pp->KQT[s2 * C + u] = on ? kqm[nt][e] : 0.f;
                    if (s2 == u) pp->sc[u].kq = kqm[nt][e];
                }
            if (lane < C) {
                pp->sc[lane].beta = bv;
                pp->gv[lane] = gv;
            }
            __syncwarp();
            if (lane < C) {
                // column u = lane of W = (I + N)^-1, N[t][s] = beta_t KK[s][t]:
                // w_t = -beta_t sum_{s<t} KK[s][t] w_s, accumulated row by row as
                // each w_s becomes known (a short dependent chain per step)
                const int u = lane;
                float acc[C], wv[C];
#pragma unroll
                for (int t2 = 0; t2 < C; ++t2) acc[t2] = 0.f;
#pragma unroll
                for (int s2 = 0; s2 < C; ++s2) {
                    const float bt = ((bits >> s2) & 1u) ? pp->sc[s2].beta : 0.f;
                    wv[s2] = s2 < u ? 0.f : (s2 == u ? 1.f : -bt * acc[s2]);
                    const float4 *kr = reinterpret_cast<const float4 *>(pp->KK + s2 * C);
#pragma unroll
                    for (int q4 = (s2 + 1) / 4; q4 < C / 4; ++q4) {
                        const float4 k4 = kr[q4];
                        const float kv4[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (4 * q4 + e > s2) acc[4 * q4 + e] = fmaf(kv4[e], wv[s2], acc[4 * q4 + e]);
                    }
                }
#pragma unroll
                for (int t2 = 0; t2 < C; ++t2) pp->W[t2 * C + u] = wv[t2];
            }
            float G = 1.f;  // the state arrives unscaled
            const unsigned dbits = scale_schedule(pp->sc, pp->gv, bits, tcnt, G, lane);
            if (lane == 0) {
                pp->bits = bits;
                pp->direct = dbits;
                pp->gfinal = G;
            }
            // tape capture: k_log / g_log rows of the active steps
            if (d.row0 == 0) {
                if (klp) {
#pragma unroll
                    for (int it = 0; it < C * (kRtDk / 8) / 32; ++it) {
                        const int q = it * 32 + lane, s = q >> 4, x = (q & 15) * 8;
                        if (s < tcnt && ((bits >> s) & 1u))
                            *reinterpret_cast<uint4 *>(klp + ((bt0 + s) * a.Hv + d.hv) * kRtDk + x) =
                                *reinterpret_cast<const uint4 *>(gptr(rt_kq_addr(kq, false, s, x)));
                    }
                }
                if (glp && lin && ((bits >> lane) & 1u)) st_from_f32(glp + (bt0 + lane) * a.Hv + d.hv, gv);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(g, kRtBarPrep + buf));  // the unit's preparation block is ready
            d = dn;
        }
        if (!ok && lane == 0) atomicExch(ta.wait_flag, 1u);
    } else if (issuer_warp) {
        // ================================================ issuer warp (lane 0)
        // TMA loads of the warpgroup's units and its tcgen05.mma products
        const uint32_t gb = base + (uint32_t)wg * kRtGroupBytes;
        const uint32_t slot = gb;
        const uint32_t tm_s = tmem0 + (uint32_t)(wg * 256);  // S: columns [0, 128)
        const uint32_t tm_p = tm_s + 128;                    // P: columns [128, 160)
        if (lane == 0) {
            const uint64_t pol_state = l2_evict_first_policy();
            auto issue_state = [&](const Unit &d) {
                mbar_arrive_expect_tx(bar(wg, kRtBarState), kRtSlot);
#pragma unroll
                for (int bx = 0; bx < kRtDk / 32; ++bx)
                    tma_load_3d(slot + bx * 16384, &tm_state, bx * 32, (int)d.row0, (int)d.n, bar(wg, kRtBarState),
                                pol_state);
            };
            auto issue_in = [&](const Unit &d, int buf) {
                const uint32_t kq = gb + kRtOffKq + buf * kRtKq, vb = gb + kRtOffV + buf * kRtV;
                const uint32_t bb = bar(wg, kRtBarIn + buf);
                mbar_arrive_expect_tx(bb, kRtKq + kRtV);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    tma_load_4d(kq + h * 4096, &tm_k, h * 64, (int)d.hk, 0, (int)d.b, bb);
                    tma_load_4d(kq + h * 4096 + 2048, &tm_q, h * 64, (int)d.hk, 0, (int)d.b, bb);
                }
                tma_load_4d(vb, &tm_v, (int)d.row0, (int)d.hv, 0, (int)d.b, bb);
            };
            const uint32_t id1 = rt_idesc_bf16(2 * C), id2 = rt_idesc_bf16(kRtDk);
            // the last unit whose copies / products were issued, to drain them if
            // a wait runs out
            int64_t last_s = -1, last_in[2] = {-1, -1}, last_m1 = -1, last_m2 = -1;
            bool ok = true;
            Unit d = unit_of(wg, 0);
            if (d.valid) {
                issue_state(d);
                issue_in(d, 0);
                last_s = 0;
                last_in[0] = 0;
            }
            for (int64_t j = 0; ok && d.valid; ++j) {
                const int buf = (int)(j & 1);
                const uint32_t kq = gb + kRtOffKq + buf * kRtKq;
                const Unit dn = unit_of(wg, j + 1);
                if (dn.valid) {  // the next unit's inputs, once their buffer's last unit (j - 1) is done
                    if (j >= 1)
                        ok = mbar_wait_bounded(bar(wg, kRtBarDone + (buf ^ 1)), (uint32_t)(((j - 1) >> 1) & 1),
                                               ta.wait_cycles);
                    if (!ok) break;
                    issue_in(dn, buf ^ 1);
                    last_in[buf ^ 1] = j + 1;
                }
                // MMA1: P = [S hi; S lo] [K; Q]^T, once the row warps wrote the operand tiles
                ok = mbar_wait_bounded(bar(wg, kRtBarPass), (uint32_t)(j & 1), ta.wait_cycles) &&
                     mbar_wait_bounded(bar(wg, kRtBarIn + buf), (uint32_t)((j >> 1) & 1), ta.wait_cycles);
                if (!ok) break;
                rt_fence_after();
#pragma unroll
                for (int kk = 0; kk < kRtDk / 16; ++kk) {
                    const uint32_t abase = slot + (uint32_t)(kk >> 1) * 16384u + (uint32_t)(kk & 1) * 32u;
                    const uint64_t db =
                        rt_desc(kq + (uint32_t)(kk >> 2) * 4096u + (uint32_t)(kk & 3) * 32u, 16, 1024, 2);
                    rt_mma(tm_p, rt_desc(abase, 16, 512, 4), db, id1, kk > 0 ? 1u : 0u);
                    rt_mma(tm_p, rt_desc(abase + 8192u, 16, 512, 4), db, id1, 1u);
                }
                rt_commit(bar(wg, kRtBarMma1));
                last_m1 = j;
                // the slot is free once MMA1 has read it: the next unit's state rows
                ok = mbar_wait_bounded(bar(wg, kRtBarMma1), (uint32_t)(j & 1), ta.wait_cycles);
                if (!ok) break;
                if (dn.valid) {
                    issue_state(dn);
                    last_s = j + 1;
                }
                // MMA2: S += [D hi; D lo] K, once the row warps wrote D and K^T
                ok = mbar_wait_bounded(bar(wg, kRtBarSolve), (uint32_t)(j & 1), ta.wait_cycles);
                if (!ok) break;
                rt_fence_after();
                const uint64_t db = rt_desc(gb + kRtOffB2, 128, 256, 0);
                rt_mma(tm_s, rt_desc(gb + kRtOffA2, 128, 256, 0), db, id2, 1u);
                rt_mma(tm_s, rt_desc(gb + kRtOffA2 + 4096u, 128, 256, 0), db, id2, 1u);
                rt_commit(bar(wg, kRtBarMma2));
                last_m2 = j;
                d = dn;
            }
            if (!ok) {
                atomicExch(ta.wait_flag, 1u);
                // let every copy and product this warp issued land before the CTA
                // releases its shared and tensor memory (bounded again)
                if (last_s >= 0) mbar_wait_bounded(bar(wg, kRtBarState), (uint32_t)(last_s & 1), kRtWaitCycles);
                for (int b2 = 0; b2 < 2; ++b2)
                    if (last_in[b2] >= 0)
                        mbar_wait_bounded(bar(wg, kRtBarIn + b2), (uint32_t)((last_in[b2] >> 1) & 1), kRtWaitCycles);
                if (last_m1 >= 0) mbar_wait_bounded(bar(wg, kRtBarMma1), (uint32_t)(last_m1 & 1), kRtWaitCycles);
                if (last_m2 >= 0) mbar_wait_bounded(bar(wg, kRtBarMma2), (uint32_t)(last_m2 & 1), kRtWaitCycles);
            }
        }
    } else {
        // ================================================ the row warps of a warpgroup
        const uint32_t gb = base + (uint32_t)wg * kRtGroupBytes;
        const uint32_t slot = gb;
        const uint32_t tm_s = tmem0 + (uint32_t)(wg * 256);  // S: columns [0, 128)
        const uint32_t tm_p = tm_s + 128;                    // P: columns [128, 160)
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        const int barid = 1 + wg;
        T *yp = static_cast<T *>(a.y);
        T *dp = static_cast<T *>(a.delta_log);
        float *sout = static_cast<float *>(a.state_out);
        // a wait that runs out raises the flag at once; the warpgroup stops at
        // its next shared barrier
        // After a failed wait the rest of the unit still arrives on every
        // barrier (so nothing else waits in vain) but skips the tensor-memory
        // reads that the missing product would have fed, and writes NaN as the
        // unit's state rows.  The decision is taken per warp (tensor-memory
        // loads are warp-wide).
        auto wait = [&](uint32_t b, int64_t phase, bool &okv) {
            if (okv && !mbar_wait_bounded(b, (uint32_t)(phase & 1), ta.wait_cycles)) {
                okv = false;
                atomicExch(ta.wait_flag, 1u);
            }
            okv = __all_sync(0xffffffffu, okv);
        };
        bool ok = true;
        if (ta.inject_expiry) wait(bar(wg, kRtBarNever), 0, ok);  // testing hook: runs out
        for (int64_t j = 0;; ++j) {
            const Unit d = unit_of(wg, j);
            if (!d.valid) break;
            const int buf = (int)(j & 1);
            const uint32_t kq = gb + kRtOffKq + buf * kRtKq;
            const T *vs = reinterpret_cast<const T *>(gptr(gb + kRtOffV + buf * kRtV));
            const RtPrep *pp = reinterpret_cast<const RtPrep *>(gptr(gb + kRtOffPrep + buf * kRtPrepAl));

            // ---- the state rows: into S (tensor memory) and, in place, into the
            // bf16 hi / lo operand tiles of MMA1 (two boxes of 32 columns at a time)
            wait(bar(wg, kRtBarState), j, ok);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t x[2][32];
#pragma unroll
                for (int bb2 = 0; bb2 < 2; ++bb2) {
                    const int bx = 2 * half + bb2;
                    const unsigned char *row = gptr(slot + bx * 16384 + r * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 v4 = *reinterpret_cast<const uint4 *>(row + ((c ^ (r & 7)) << 4));
                        x[bb2][4 * c] = v4.x;
                        x[bb2][4 * c + 1] = v4.y;
                        x[bb2][4 * c + 2] = v4.z;
                        x[bb2][4 * c + 3] = v4.w;
                    }
                    rt_st32(tm_s + lane_off + (uint32_t)(32 * bx), x[bb2]);
                }
                // both boxes read by every row before they are rewritten; the
                // first of these barriers also stops the warpgroup after a failed wait
                if (half == 0) {
                    if (named_bar_or(barid, 128, !ok)) {
                        ok = false;
                        break;
                    }
                } else {
                    named_bar_sync(barid, 128);
                }
#pragma unroll
                for (int bb2 = 0; bb2 < 2; ++bb2) {
                    const int bx = 2 * half + bb2;
                    unsigned char *hrow = gptr(slot + bx * 16384 + r * 64);
                    unsigned char *lrow = hrow + 8192;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t h4[4], l4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            split_bf16x2(__uint_as_float(x[bb2][8 * c + 2 * e]),
                                         __uint_as_float(x[bb2][8 * c + 2 * e + 1]), h4[e], l4[e]);
                        const int pc = (c ^ ((r >> 1) & 3)) << 4;
                        *reinterpret_cast<uint4 *>(hrow + pc) = make_uint4(h4[0], h4[1], h4[2], h4[3]);
                        *reinterpret_cast<uint4 *>(lrow + pc) = make_uint4(l4[0], l4[1], l4[2], l4[3]);
                    }
                }
            }
            if (!ok) {
                // poison this unit's state rows
                float *orow = sout + ((int64_t)d.n * a.Dv + d.row0 + r) * kRtDk;
                const float nan = __int_as_float(0x7fc00000);
                for (int c = 0; c < kRtDk / 4; ++c)
                    __stcs(reinterpret_cast<float4 *>(orow) + c, make_float4(nan, nan, nan, nan));
                break;
            }
            rt_wait_st();
            fence_async_smem();
            rt_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(wg, kRtBarPass));

            // ---- while MMA1 runs: the step scalars, K^T (inactive steps zero)
            // and this row's v entries
            wait(bar(wg, kRtBarPrep + buf), j >> 1, ok);
            wait(bar(wg, kRtBarIn + buf), j >> 1, ok);
            const unsigned bits = pp->bits;
            {
                // K^T (the B operand of MMA2, K-major core matrices of 8 columns x
                // 8 steps): warp q transposes columns 32q .. 32q+31, an 8 x 8 block
                // at a time (ldmatrix.trans from the swizzled k rows, stmatrix into
                // the core matrix); the halves of inactive steps are cleared
                const int q = warp & 3, lm = lane >> 3, l8 = lane & 7, t4 = lane & 3;
                const uint32_t mlo = (((bits >> (2 * t4)) & 1u) ? 0x0000ffffu : 0u) |
                                     (((bits >> (2 * t4 + 1)) & 1u) ? 0xffff0000u : 0u);
                const uint32_t mhi = (((bits >> (8 + 2 * t4)) & 1u) ? 0x0000ffffu : 0u) |
                                     (((bits >> (9 + 2 * t4)) & 1u) ? 0xffff0000u : 0u);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    // matrices: (steps 0-7 | 8-15) x (column groups 2hh, 2hh+1 of this warp)
                    const int sg = lm & 1, cg = 4 * q + 2 * hh + (lm >> 1);
                    uint32_t f[4];
                    ldsm_x4_t_a(f, rt_kq_addr(kq, false, 8 * sg + l8, 8 * cg));
                    f[0] &= mlo;
                    f[1] &= mhi;
                    f[2] &= mlo;
                    f[3] &= mhi;
                    const uint32_t dst = gb + kRtOffB2 + (uint32_t)cg * 256u + (uint32_t)sg * 128u + (uint32_t)l8 * 16u;
                    stsm_x4_a(dst, f);
                }
            }
            float vv[C];
#pragma unroll
            for (int s2 = 0; s2 < C; ++s2) vv[s2] = __bfloat162float(vs[s2 * kRtRows + r]);

            wait(bar(wg, kRtBarMma1), j, ok);
            rt_fence_after();

            // ---- this row's step dots, and the FP32 solve
            uint32_t pr[32];
            if (ok) {
                rt_ld32(tm_p + lane_off, pr);
                rt_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) pr[e] = 0u;
            }
            const unsigned direct = pp->direct;
            float dd[C];
            float phi_all = 1.f;
            const int64_t obase = (((int64_t)d.b * a.T) * a.Hv + d.hv) * a.Dv + d.row0 + r;
            const int64_t ostep = a.Hv * a.Dv;
            if (direct == 0u) {
                float rr[C];
#pragma unroll
                for (int s = 0; s < C; ++s) {
                    const StepScalars S = pp->sc[s];
                    rr[s] = ((bits >> s) & 1u) ? S.beta * (vv[s] * S.inv - __uint_as_float(pr[s])) : 0.f;
                }
#pragma unroll
                for (int s = 0; s < C; ++s) {  // d = W r (W unit lower triangular)
                    float acc = rr[s];
                    const float4 *wr = reinterpret_cast<const float4 *>(pp->W + s * C);
#pragma unroll
                    for (int q4 = 0; 4 * q4 < s; ++q4) {
                        const float4 w4 = wr[q4];
                        const float wv4[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (4 * q4 + e < s) acc = fmaf(wv4[e], rr[4 * q4 + e], acc);
                    }
                    dd[s] = acc;
                }
                // y and delta follow MMA2's issue (below): nothing of theirs feeds it
            } else {
                // a fold of the scale inside the chunk: the serial solve of this row
                float pa[C], pb[C];
#pragma unroll
                for (int s = 0; s < C; ++s) {
                    pa[s] = __uint_as_float(pr[s]);
                    pb[s] = __uint_as_float(pr[C + s]);
                    dd[s] = 0.f;
                }
#pragma unroll
                for (int tau = 0; tau < C; ++tau) {
                    if (!((bits >> tau) & 1u)) continue;
                    const StepScalars S = pp->sc[tau];
                    const bool fold = (direct >> tau) & 1u;
                    if (fold) {  // s^ <- G' s^ before this step
                        const float phi = S.Gp;
                        phi_all *= phi;
#pragma unroll
                        for (int s = 0; s < C; ++s) {
                            pa[s] *= phi;
                            pb[s] *= phi;
                            dd[s] *= phi;
                        }
                    }
                    const float Gp = fold ? 1.f : S.Gp;
                    const float kv = Gp * pa[tau];
                    const float delta = (vv[tau] - kv) * S.beta;
                    const float yv = fmaf(Gp, pb[tau], delta * S.kq);
                    const float dval = delta * S.inv;
                    dd[tau] = dval;
                    st_from_f32(yp + obase + tau * ostep, yv);
                    st_from_f32(dp + obase + tau * ostep, delta);
#pragma unroll
                    for (int s = tau + 1; s < C; ++s) {
                        pa[s] = fmaf(dval, pp->KK[tau * C + s], pa[s]);
                        pb[s] = fmaf(dval, pp->KQ[tau * C + s], pb[s]);
                    }
                }
            }
            // d as bf16 hi + lo (the A operand of MMA2: K-major core matrices,
            // 8 rows x 16 bytes, 128 bytes apart along the steps, 256 along rows)
            {
                uint32_t h8[8], l8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) split_bf16x2(dd[2 * e], dd[2 * e + 1], h8[e], l8[e]);
                unsigned char *a2 = gptr(gb + kRtOffA2 + (uint32_t)(r >> 3) * 256u + (uint32_t)(r & 7) * 16u);
                *reinterpret_cast<uint4 *>(a2) = make_uint4(h8[0], h8[1], h8[2], h8[3]);
                *reinterpret_cast<uint4 *>(a2 + 128) = make_uint4(h8[4], h8[5], h8[6], h8[7]);
                *reinterpret_cast<uint4 *>(a2 + 4096) = make_uint4(l8[0], l8[1], l8[2], l8[3]);
                *reinterpret_cast<uint4 *>(a2 + 4096 + 128) = make_uint4(l8[4], l8[5], l8[6], l8[7]);
            }
            if (phi_all != 1.f && ok) {
                // folds in this chunk (the same in every row): S <- phi S before adding D K
#pragma unroll 1
                for (int c = 0; c < kRtDk / 32; ++c) {
                    uint32_t sv[32];
                    rt_ld32(tm_s + lane_off + (uint32_t)(32 * c), sv);
                    rt_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) sv[e] = __float_as_uint(__uint_as_float(sv[e]) * phi_all);
                    rt_st32(tm_s + lane_off + (uint32_t)(32 * c), sv);
                }
                rt_wait_st();
            }
            fence_async_smem();
            rt_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(wg, kRtBarSolve));
            if (direct == 0u) {
                // y_t = G'_t b_t + delta_t (k_t . q_t), b_t = P_q[t] + sum_{u<t} d_u (k_u . q_t),
                // while MMA2 runs
#pragma unroll
                for (int s = 0; s < C; ++s) {
                    if (!((bits >> s) & 1u)) continue;
                    float bq = __uint_as_float(pr[C + s]);
                    const float4 *kr = reinterpret_cast<const float4 *>(pp->KQT + s * C);
#pragma unroll
                    for (int q4 = 0; 4 * q4 < s; ++q4) {
                        const float4 k4 = kr[q4];
                        const float kv4[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (4 * q4 + e < s) bq = fmaf(dd[4 * q4 + e], kv4[e], bq);
                    }
                    const StepScalars S = pp->sc[s];
                    const float delta = S.Gp * dd[s];
                    const float yv = fmaf(S.Gp, bq, delta * S.kq);
                    st_from_f32(yp + obase + s * ostep, yv);
                    st_from_f32(dp + obase + s * ostep, delta);
                }
            }

            // ---- s = G s^, streaming stores.  The accumulator is read in the
            // m16n8 fragment shape (16x256b): thread t holds rows t/4 and 8 + t/4
            // of a 16-lane half and columns 2(t%4), 2(t%4)+1 of every 8-column
            // block, so every store instruction writes 8 rows x 32 contiguous bytes.
            wait(bar(wg, kRtBarMma2), j, ok);
            rt_fence_after();
            const float Gf = ok ? pp->gfinal : __int_as_float(0x7fc00000);  // NaN after a failed wait
            const int q = warp & 3;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const int rbase = 32 * q + 16 * h + (lane >> 2);
                float *o0 = sout + ((int64_t)d.n * a.Dv + d.row0 + rbase) * kRtDk + 2 * (lane & 3);
                float *o1 = o0 + 8 * kRtDk;
                uint32_t sv[64];
                if (ok) {
                    rt_ld16x256_x16(tm_s + ((uint32_t)(32 * q + 16 * h) << 16), sv);
                    rt_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e) sv[e] = 0u;
                }
                const float2 g2 = make_float2(Gf, Gf);
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    __stcs(reinterpret_cast<float2 *>(o0 + 8 * m),
                           __fmul2_rn(make_float2(__uint_as_float(sv[4 * m]), __uint_as_float(sv[4 * m + 1])), g2));
                    __stcs(reinterpret_cast<float2 *>(o1 + 8 * m),
                           __fmul2_rn(make_float2(__uint_as_float(sv[4 * m + 2]), __uint_as_float(sv[4 * m + 3])), g2));
                }
            }
            rt_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(wg, kRtBarDone + buf));  // the unit's buffers are free
        }
    }
    rt_fence_before();
    __syncthreads();
    rt_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem0), "r"(kRtTmemCols));
}

}  // namespace gdn
