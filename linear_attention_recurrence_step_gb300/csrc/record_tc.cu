// record_tc.cu -- host side of the tcgen05 record kernel (record_tc.cuh):
// tensor maps, eligibility and launch.
#include "record_tc.cuh"
#include "tma_host.h"

namespace gdn {

namespace {

// Set by the kernel when one of its bounded waits runs out.
__device__ unsigned g_record_tc_wait_flag;

cudaError_t launch_tc(const RecordArgs &args, int sm_count, cudaStream_t st) {
    RecordArgs a = args;
    a.row_blocks = a.Dv / kRtRows;  // units of 128 rows (the caller's geometry counts 64-row blocks)
    CUtensorMap tm_s, tm_k, tm_q, tm_v;
    {
        // state [B*Hv, Dv, Dk] f32: boxes of 32 columns x 128 rows of one tile
        const cuuint64_t dims[3] = {(cuuint64_t)kRtDk, (cuuint64_t)a.Dv, (cuuint64_t)(a.B * a.Hv)};
        const cuuint64_t strides[2] = {(cuuint64_t)kRtDk * 4, (cuuint64_t)a.Dv * kRtDk * 4};
        const cuuint32_t box[3] = {32, (cuuint32_t)kRtRows, 1};
        if (!tma_encode(&tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.state_in, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    {
        // q, k [B, T, Hk, Dk] bf16: boxes of 64 columns x 16 steps of one head
        const cuuint64_t dims[4] = {(cuuint64_t)kRtDk, (cuuint64_t)a.Hk, (cuuint64_t)a.T, (cuuint64_t)a.B};
        const cuuint64_t strides[3] = {(cuuint64_t)kRtDk * 2, (cuuint64_t)(a.Hk * kRtDk * 2),
                                       (cuuint64_t)(a.T * a.Hk * kRtDk * 2)};
        const cuuint32_t box[4] = {64, 1, (cuuint32_t)kMmaChunk, 1};
        if (!tma_encode(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.k, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
            !tma_encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.q, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    {
        // v [B, T, Hv, Dv] bf16: boxes of 128 rows x 16 steps of one head
        const cuuint64_t dims[4] = {(cuuint64_t)a.Dv, (cuuint64_t)a.Hv, (cuuint64_t)a.T, (cuuint64_t)a.B};
        const cuuint64_t strides[3] = {(cuuint64_t)a.Dv * 2, (cuuint64_t)(a.Hv * a.Dv * 2),
                                       (cuuint64_t)(a.T * a.Hv * a.Dv * 2)};
        const cuuint32_t box[4] = {(cuuint32_t)kRtRows, 1, (cuuint32_t)kMmaChunk, 1};
        if (!tma_encode(&tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.v, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    void *flag = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&flag, g_record_tc_wait_flag);
    if (e != cudaSuccess) return e;
    RecordTcArgs ta{a, a.B * a.Hv * (a.Dv / kRtRows), static_cast<unsigned *>(flag), wait_bound_cycles(),
                    inject_wait_expiry()};
    e = cudaFuncSetAttribute(record_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRtSmem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(sm_count > 0 ? sm_count : 1, ta.nunits);
    return launch_dependent(record_tc_kernel, (unsigned)grid, kRtThreads, kRtSmem, st, tm_s, tm_k, tm_q, tm_v, ta);
}

}  // namespace

bool record_tc_eligible(const RecordArgs &a, int dk, bool bf16) {
    // one chunk per call, f32 state, 128-row units, 16-byte aligned v rows,
    // and coordinates that fit the int32 fields of a TMA box
    return bf16 && !a.tstate && dk == kRtDk && a.Dv % kRtRows == 0 && a.T >= 1 && a.T <= kMmaChunk &&
           a.vec_v && a.B * a.Hv * (a.Dv / kRtRows) <= (int64_t)INT32_MAX && a.Dv <= (int64_t)INT32_MAX &&
           tma_encoder_available();
}

cudaError_t launch_record_tc(const RecordArgs &a, int sm_count, cudaStream_t st) {
    return launch_tc(a, sm_count, st);
}

cudaError_t record_tc_take_wait_flag(unsigned *was_set) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_record_tc_wait_flag, sizeof v);
    if (e != cudaSuccess) return e;
    *was_set = v;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_record_tc_wait_flag, &zero, sizeof zero);
    }
    return e;
}

}  // namespace gdn
