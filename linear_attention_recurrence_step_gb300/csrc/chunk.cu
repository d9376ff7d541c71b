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

// Library-owned scratch for gdn_chunk_prefill_noalloc: one block of device
// memory per device, reserved when the module loads (never allocated at
// call time).  Calls that use it must not overlap in time on one device.
static __device__ __align__(256) float g_chunk_scratch[kChunkStaticScratchBytes / sizeof(float)];

// The address of a __device__ symbol belongs to the CUDA context that loaded
// the module, not to the device index: after cudaDeviceReset, or when a
// driver-API caller makes another context current on the same device, an
// address remembered from an earlier call would be stale.  So the address is
// looked up on every call (cheap next to the two launches that use it).
cudaError_t chunk_static_scratch(float **ptr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_chunk_scratch);
    if (e != cudaSuccess) return e;
    *ptr = static_cast<float *>(p);
    return cudaSuccess;
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
