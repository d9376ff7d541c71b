// replay_stream.cu -- host side of the persistent TMA-fed replay
// (replay_stream.cuh): eligibility, tensor maps and launch.
#include <algorithm>
#include <atomic>
#include <climits>

#include "replay_stream.cuh"
#include "tma_host.h"

namespace gdn {

namespace {

// Set by the kernel when one of its bounded waits runs out.
__device__ unsigned g_replay_stream_wait_flag;

// Block counters of the persistent kernel, one pair per launch slot: the next
// block to hand out and the CTAs that have finished claiming.  Launches take
// the slots round robin; the last CTA of a launch resets its pair to zero, so
// a slot is ready again once its launch has completed.  Two launches share a
// slot only if kRsSchedSlots launches of this kernel are in flight at once,
// or if two instantiations of one captured graph run at the same time.
__device__ unsigned g_rs_sched[kRsSchedSlots][2];
std::atomic<unsigned> g_rs_next_slot{0};

template <typename TIn>
CUtensorMapDataType tape_map_type();
template <>
CUtensorMapDataType tape_map_type<float>() { return CU_TENSOR_MAP_DATA_TYPE_FLOAT32; }
template <>
CUtensorMapDataType tape_map_type<__nv_bfloat16>() { return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; }
template <>
CUtensorMapDataType tape_map_type<__half>() { return CU_TENSOR_MAP_DATA_TYPE_FLOAT16; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename TIn>
cudaError_t launch_t(const ReplayArgs &args, int sm_count, cudaStream_t st, bool *launched) {
    using S = RsStage<TIn>;
    ReplayArgs a = args;
    a.rows_cta = kRsRows;
    a.row_blocks = (a.Dv + kRsRows - 1) / kRsRows;
    const cuuint64_t es = sizeof(TIn);
    CUtensorMap tm_s, tm_k, tm_d;
    const int box_steps = (int)std::max<int64_t>(1, std::min<int64_t>(a.steps, kRsSteps));
    // state [B*Hv, Dv, 128] f32: one box of 64 whole rows of one tile
    const cuuint64_t sd[3] = {(cuuint64_t)kRsDk, (cuuint64_t)a.Dv, (cuuint64_t)(a.B * a.Hv)};
    const cuuint64_t ss[2] = {(cuuint64_t)kRsDk * 4, (cuuint64_t)a.Dv * kRsDk * 4};
    const cuuint32_t sb[3] = {(cuuint32_t)kRsDk, (cuuint32_t)kRsRows, 1};
    // k_log [B, T, Hv, 128]: the rows of steps 0 .. box_steps - 1 of one head
    const cuuint64_t kd[4] = {(cuuint64_t)kRsDk, (cuuint64_t)a.Hv, (cuuint64_t)a.T, (cuuint64_t)a.B};
    const cuuint64_t ks[3] = {kRsDk * es, (cuuint64_t)a.Hv * kRsDk * es, (cuuint64_t)(a.T * a.Hv) * kRsDk * es};
    const cuuint32_t kb[4] = {(cuuint32_t)kRsDk, 1, (cuuint32_t)box_steps, 1};
    // delta_log [B, T, Hv, Dv]: the block's 64 rows of steps 0 .. box_steps - 1
    const cuuint64_t dd[4] = {(cuuint64_t)a.Dv, (cuuint64_t)a.Hv, (cuuint64_t)a.T, (cuuint64_t)a.B};
    const cuuint64_t ds[3] = {(cuuint64_t)a.Dv * es, (cuuint64_t)(a.Hv * a.Dv) * es,
                              (cuuint64_t)(a.T * a.Hv * a.Dv) * es};
    const cuuint32_t db[4] = {(cuuint32_t)kRsRows, 1, (cuuint32_t)box_steps, 1};
    if (!tma_encode(&tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.state_in, sd, ss, sb, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tma_encode(&tm_k, tape_map_type<TIn>(), 4, a.k_log, kd, ks, kb, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !tma_encode(&tm_d, tape_map_type<TIn>(), 4, a.delta_log, dd, ds, db, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaSuccess;  // not launched: the caller runs the FP32 replay kernel
    void *flag = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&flag, g_replay_stream_wait_flag);
    if (e != cudaSuccess) return e;
    void *sched = nullptr;
    e = cudaGetSymbolAddress(&sched, g_rs_sched);
    if (e != cudaSuccess) return e;
    const unsigned slot = g_rs_next_slot.fetch_add(1u, std::memory_order_relaxed) % kRsSchedSlots;
    const ReplayStreamArgs ra{a, a.B * a.Hv * a.row_blocks, box_steps, static_cast<unsigned *>(flag),
                              wait_bound_cycles(), inject_wait_expiry(), static_cast<unsigned *>(sched) + 2 * slot};
    auto kern = replay_stream_kernel<TIn>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(sm_count > 0 ? sm_count : 1, ra.nblocks);
    *launched = true;
    return launch_dependent(kern, (unsigned)grid, kRsThreads, S::SMEM, st, tm_s, tm_k, tm_d, ra);
}

}  // namespace

cudaError_t launch_replay_stream(DType dt, int dk, const ReplayArgs &a, int sm_count, cudaStream_t st,
                                 bool *launched) {
    *launched = false;
    // Dk = 128, f32 state, 2 to 16 steps, whole 16-byte delta_log rows at
    // 16-byte aligned addresses, 16-byte aligned k_log and state, and
    // coordinates that fit the int32 fields of a TMA box.  Single-step calls
    // (decode) stay on the FP32 replay kernel: at B = 32, Hv = 32 it measured
    // 26.9 us there against 27.8-28.8 us here, while the 8- and 16-step
    // verify / rollback shapes measured 18.5-19.7 us against 19.8 us and
    // 93.7 us against 95.5 us.
    if (dk != kRsDk || a.tstate || a.steps < 2 || a.steps > kRsSteps || !a.vec_d || !aligned16(a.k_log) ||
        !aligned16(a.state_in) || !aligned16(a.state_out) || a.B > INT_MAX || a.T > INT_MAX || a.Hv > INT_MAX ||
        a.Dv > INT_MAX || a.B * a.Hv > INT_MAX / ((a.Dv + kRsRows - 1) / kRsRows) || !tma_encoder_available())
        return cudaSuccess;
    switch (dt) {
    case DType::F32: return launch_t<float>(a, sm_count, st, launched);
    case DType::BF16: return launch_t<__nv_bfloat16>(a, sm_count, st, launched);
    case DType::F16: return launch_t<__half>(a, sm_count, st, launched);
    }
    return cudaSuccess;
}

cudaError_t replay_stream_take_wait_flag(unsigned *was_set) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_replay_stream_wait_flag, sizeof v);
    if (e != cudaSuccess) return e;
    *was_set = v;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_replay_stream_wait_flag, &zero, sizeof zero);
    }
    return e;
}

}  // namespace gdn
