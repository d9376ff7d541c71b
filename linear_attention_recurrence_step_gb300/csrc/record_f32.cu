// record_f32.cu -- record kernels with f32 inputs / outputs (state f32).
#include "record.cuh"

namespace gdn {

cudaError_t launch_record_f32(int dk, const RecordArgs &a, const Geometry &geo, cudaStream_t s) {
    switch (dk) {
    case 32: return launch_record_t<float, 32>(a, geo, s);
    case 64: return launch_record_t<float, 64>(a, geo, s);
    case 128: return launch_record_t<float, 128>(a, geo, s);
    case 192: return launch_record_t<float, 192>(a, geo, s);
    case 256: return launch_record_t<float, 256>(a, geo, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
