// record_f16.cu -- record kernels with f16 inputs / outputs (state f32).
#include "record.cuh"

namespace gdn {

cudaError_t launch_record_f16(int dk, const RecordArgs &a, const Geometry &geo, cudaStream_t s) {
    switch (dk) {
    case 32: return launch_record_t<__half, 32>(a, geo, s);
    case 64: return launch_record_t<__half, 64>(a, geo, s);
    case 128: return launch_record_t<__half, 128>(a, geo, s);
    case 192: return launch_record_t<__half, 192>(a, geo, s);
    case 256: return launch_record_t<__half, 256>(a, geo, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
