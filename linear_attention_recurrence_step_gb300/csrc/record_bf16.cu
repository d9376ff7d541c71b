// record_bf16.cu -- record kernels with bf16 inputs / outputs (state f32).
#include "record.cuh"
#include "record_mma.cuh"

namespace gdn {

template <int DK>
static cudaError_t run(const RecordArgs &a, const Geometry &geo, cudaStream_t s) {
    if constexpr (record_mma_supported(DK)) {
        if (geo.mma) return launch_record_mma<DK>(a, geo, s);
    }
    return launch_record_layout<__nv_bfloat16, typename DefaultLayout<DK>::type>(a, geo, s);
}

cudaError_t launch_record_bf16(int dk, const RecordArgs &a, const Geometry &geo, cudaStream_t s) {
    switch (dk) {
    case 32: return run<32>(a, geo, s);
    case 64: return run<64>(a, geo, s);
    case 128: return run<128>(a, geo, s);
    case 192: return run<192>(a, geo, s);
    case 256: return run<256>(a, geo, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
