// chunk.cu -- launches of the chunked-prefill kernels (chunk.cuh) for every
// element type and compiled Dk.
#include "chunk.cuh"

namespace gdn {

cudaError_t launch_chunk(DType dt, int dk, const ChunkArgs &a, cudaStream_t s) {
    switch (dt) {
    case DType::F32: return launch_chunk_type<float>(dk, a, s);
    case DType::BF16: return launch_chunk_type<__nv_bfloat16>(dk, a, s);
    case DType::F16: return launch_chunk_type<__half>(dk, a, s);
    }
    return cudaErrorInvalidValue;
}

int64_t chunk_workspace_bytes(int64_t B, int64_t T, int64_t Hv) {
    const int64_t nch = (T + kCkC - 1) / kCkC;
    int64_t r = (int64_t)kCkWsFloats * 4;
    if (__builtin_mul_overflow(r, B, &r) || __builtin_mul_overflow(r, Hv, &r) ||
        __builtin_mul_overflow(r, nch, &r))
        return -1;
    return r;
}

}  // namespace gdn
