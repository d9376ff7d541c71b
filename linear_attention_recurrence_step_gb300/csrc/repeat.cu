// repeat.cu -- tiled GQA broadcast ("mlx-native repeat_tiled.rs", module doc
// "Mapping"): dst[t, hh, x] = src[t, hh % hg, x].
//
// The page dispatches one thread per OUTPUT element (grid (K, H, T)), so each
// source row is read h/hg times.  Here one thread owns one 16-byte vector (or
// one element) of a SOURCE row, reads it once and writes it to the h/hg
// destination heads hh = hs, hs + hg, hs + 2 hg, ... that map to it: the copy
// reads src once and writes dst once.
#include "common.cuh"
#include "launch.h"

namespace gdn {

template <typename V>
__global__ void __launch_bounds__(256) repeat_kernel(const V *__restrict__ src, V *__restrict__ dst,
                                                     int64_t seq, int64_t hg, int64_t h,
                                                     int64_t per_row) {
    pdl_trigger();
    pdl_wait();
    const int64_t total = seq * hg * per_row;
    const int64_t copies = h / hg;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t x = i % per_row;
        const int64_t r = i / per_row;  // source row (t, hs)
        const int64_t hs = r % hg;
        const int64_t t = r / hg;
        const V val = src[i];
        V *out = dst + (t * h + hs) * per_row + x;
        for (int64_t c = 0; c < copies; ++c) out[c * hg * per_row] = val;
    }
}

template <typename V>
static cudaError_t launch_v(const RepeatArgs &a, int64_t per_row, cudaStream_t s, int sm_count) {
    const int64_t total = a.seq * a.hg * per_row;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)(sm_count > 0 ? sm_count : 152) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_dependent(repeat_kernel<V>, (unsigned)blocks, threads, 0, s, static_cast<const V *>(a.src),
                            static_cast<V *>(a.dst), a.seq, a.hg, a.h, per_row);
}

cudaError_t launch_repeat(const RepeatArgs &a, cudaStream_t s, int sm_count) {
    if (a.vec16) return launch_v<uint4>(a, a.row_bytes / 16, s, sm_count);
    switch (a.elem_bytes) {
    case 4: return launch_v<uint32_t>(a, a.row_bytes / 4, s, sm_count);
    case 2: return launch_v<uint16_t>(a, a.row_bytes / 2, s, sm_count);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
