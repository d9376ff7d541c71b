// common.cuh -- device helpers shared by the record / replay / repeat kernels.
//
// Element types: the page kernels are generic over T in {f32, f16, bf16}
// ("metaltile-std gated_delta_replay.rs", gdr_spec! dtypes) with all
// arithmetic in f32 (every load is `.cast::<f32>()`); the state here is
// always f32.  Loads widen exactly, stores round to nearest-even.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// Round a byte count up to a multiple of 16 (shared-memory carving).
__host__ __device__ constexpr size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

// ------------------------------------------------------------ dependent launch
// A kernel launched with launch_dependent may be scheduled while the kernel
// before it in the stream is still running (programmatic dependent launch):
// its CTAs take SMs as the earlier kernel's CTAs leave them, do their set-up
// (barriers, tensor memory, nothing that reads global memory) and then wait
// in pdl_wait() until the earlier kernel has completed and its writes are
// visible.  pdl_trigger() lets the next such kernel be scheduled; it is
// called once every CTA of the grid is resident, so a waiting dependent CTA
// never holds an SM that a CTA of the kernel it waits for still needs.  Each
// thread that touches global memory executes pdl_wait() first.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                                    cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// ------------------------------------------------------------ element types
template <typename T> struct Elem;

template <> struct Elem<float> {
    static __device__ __forceinline__ float to_f32(float x) { return x; }
    static __device__ __forceinline__ float from_f32(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};
template <> struct Elem<__half> {
    static __device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
    static __device__ __forceinline__ __half from_f32(float x) { return __float2half_rn(x); }
};

template <typename T>
__device__ __forceinline__ float ld_f32(const T *p) { return Elem<T>::to_f32(*p); }

template <typename T>
__device__ __forceinline__ void st_from_f32(T *p, float x) { *p = Elem<T>::from_f32(x); }

// Widen one 16-byte vector of T (4 f32 / 8 bf16 / 8 f16) into f32 in shared
// memory.  `dst` must be 16-byte aligned.
template <typename T>
__device__ __forceinline__ void widen16(float *dst, const uint4 raw);

template <>
__device__ __forceinline__ void widen16<float>(float *dst, const uint4 raw) {
    *reinterpret_cast<uint4 *>(dst) = raw;
}
template <>
__device__ __forceinline__ void widen16<__nv_bfloat16>(float *dst, const uint4 raw) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float4 lo, hi;
    // bf16 -> f32 is exact: the bf16 bits are the top half of the f32 bits.
    lo.x = __uint_as_float(w[0] << 16); lo.y = __uint_as_float(w[0] & 0xffff0000u);
    lo.z = __uint_as_float(w[1] << 16); lo.w = __uint_as_float(w[1] & 0xffff0000u);
    hi.x = __uint_as_float(w[2] << 16); hi.y = __uint_as_float(w[2] & 0xffff0000u);
    hi.z = __uint_as_float(w[3] << 16); hi.w = __uint_as_float(w[3] & 0xffff0000u);
    reinterpret_cast<float4 *>(dst)[0] = lo;
    reinterpret_cast<float4 *>(dst)[1] = hi;
}
template <>
__device__ __forceinline__ void widen16<__half>(float *dst, const uint4 raw) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
        const float2 f = __half22float2(h);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
    reinterpret_cast<float4 *>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// ----------------------------------------------------------- deferred decay
// The kernels keep each state row as s = G * s_hat with one f32 scale G per
// (b, hv) tile.  A decay step multiplies the scalar G instead of all Dk
// entries; the rank-1 update adds k * (delta / G) to s_hat.  When G leaves
// [kScaleMin, kScaleMax] (or is zero, negative or NaN) the scale is folded
// into s_hat (s_hat *= G', G = 1) and the step falls back to the page's
// direct form.  Record and replay apply this rule with identical f32
// operations, so a float32 tape replays bit-exactly.
constexpr float kScaleMin = 0x1p-32f;
constexpr float kScaleMax = 0x1p+32f;

__device__ __forceinline__ bool scale_in_range(float G) {
    return G >= kScaleMin && G <= kScaleMax;  // false for NaN
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 lo2(const float4 &x) { return make_float2(x.x, x.y); }
__device__ __forceinline__ float2 hi2(const float4 &x) { return make_float2(x.z, x.w); }
__device__ __forceinline__ float4 cat4(float2 a, float2 b) { return make_float4(a.x, a.y, b.x, b.y); }

}  // namespace gdn
