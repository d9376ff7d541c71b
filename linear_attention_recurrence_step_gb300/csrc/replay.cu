// replay.cu -- replay kernels for every element type (state f32).
#include "replay.cuh"

namespace gdn {

template <typename TIn, int DK>
static cudaError_t run(const ReplayArgs &a, const Geometry &geo, cudaStream_t s) {
    return launch_replay_layout<TIn, typename DefaultLayout<DK>::type>(a, geo, s);
}

template <typename TIn>
static cudaError_t replay_dk(int dk, const ReplayArgs &a, const Geometry &geo, cudaStream_t s) {
    switch (dk) {
    case 32: return run<TIn, 32>(a, geo, s);
    case 64: return run<TIn, 64>(a, geo, s);
    case 128: return run<TIn, 128>(a, geo, s);
    case 192: return run<TIn, 192>(a, geo, s);
    case 256: return run<TIn, 256>(a, geo, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_replay(DType dt, int dk, const ReplayArgs &a, const Geometry &geo,
                          cudaStream_t s) {
    switch (dt) {
    case DType::F32: return replay_dk<float>(dk, a, geo, s);
    case DType::BF16: return replay_dk<__nv_bfloat16>(dk, a, geo, s);
    case DType::F16: return replay_dk<__half>(dk, a, geo, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn
