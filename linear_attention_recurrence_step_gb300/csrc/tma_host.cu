// tma_host.cu -- cuTensorMapEncodeTiled through the runtime's driver entry
// point lookup (tma_host.h).
#include <cudaTypedefs.h>

#include <mutex>

#include "tma_host.h"

namespace gdn {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

bool tma_encoder_available() { return tensor_map_encoder() != nullptr; }

bool tma_encode(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *ptr, const cuuint64_t *dims,
                const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle sw) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, dt, (cuuint32_t)rank, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gdn
