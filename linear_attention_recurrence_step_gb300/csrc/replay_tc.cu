// replay_tc.cu -- launches of the tensor-core replay (replay_tc.cuh) and its
// split plan / workspace layout.
#include "replay_tc.cuh"

namespace gdn {

namespace {
// Set by the kernel when one of its bounded waits runs out.
__device__ unsigned g_replay_tc_wait_flag;
}  // namespace

cudaError_t launch_replay_tc(DType dt, int dk, const ReplayTcArgs &args, cudaStream_t s, int sms) {
    ReplayTcArgs a = args;
    void *flag = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&flag, g_replay_tc_wait_flag);
    if (e != cudaSuccess) return e;
    a.wait_flag = static_cast<unsigned *>(flag);
    a.wait_cycles = wait_bound_cycles();
    a.inject_expiry = inject_wait_expiry();
    switch (dt) {
    case DType::F32: return launch_replay_tc_type<float>(dk, a, s, sms);
    case DType::BF16: return launch_replay_tc_type<__nv_bfloat16>(dk, a, s, sms);
    case DType::F16: return launch_replay_tc_type<__half>(dk, a, s, sms);
    }
    return cudaErrorInvalidValue;
}

cudaError_t replay_tc_take_wait_flag(unsigned *was_set) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_replay_tc_wait_flag, sizeof v);
    if (e != cudaSuccess) return e;
    *was_set = v;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_replay_tc_wait_flag, &zero, sizeof zero);
    }
    return e;
}

// Steps are split over CTAs only when the tiles alone give fewer than
// kTcPlanSms x (CTAs per SM) CTAs; the plan depends on the shapes only (not
// on the device), so the workspace size is a pure function of them.  The
// SM count it plans for is the GB300's: the splits fill all 152 SMs (with
// 128, the long prefill's 32 tiles took eight splits and left 24 SMs idle).
constexpr int64_t kTcPlanSms = 152;
ReplayTcPlan replay_tc_plan(int64_t B, int64_t T, int64_t Hv, int64_t Dk, int64_t Dv) {
    ReplayTcPlan p{};
    p.bytes = -1;
    p.row_blocks = (Dv + kTcRows - 1) / kTcRows;
    int64_t items = 0, nkb = (T + kTcSteps - 1) / kTcSteps;
    if (__builtin_mul_overflow(B, Hv, &items) || __builtin_mul_overflow(items, p.row_blocks, &items))
        return p;
    const int64_t want = kTcPlanSms * (int64_t)tc_ctas_per_sm((int)Dk);
    int64_t splits = items >= want ? 1 : std::min<int64_t>(nkb, want / items);
    if (splits < 1) splits = 1;
    p.split_steps = ((nkb + splits - 1) / splits) * kTcSteps;
    p.splits = (int)((T + p.split_steps - 1) / p.split_steps);
    int64_t w = 0, g = 0, part = 0;
    if (__builtin_mul_overflow(B * Hv, T * 4, &w)) return p;
    g = B * Hv * 4;
    if (p.splits > 1) {
        int64_t per = 0;
        if (__builtin_mul_overflow(B * Hv, Dv * Dk * 4, &per) || __builtin_mul_overflow(per, (int64_t)p.splits, &part))
            return p;
    }
    p.w_off = 0;
    p.gam_off = (w + 15) & ~(int64_t)15;
    p.partial_off = p.gam_off + ((g + 15) & ~(int64_t)15);
    p.bytes = p.partial_off + part;
    return p;
}

}  // namespace gdn
