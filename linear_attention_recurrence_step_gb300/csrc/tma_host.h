// tma_host.h -- host side of the TMA copies: building CUtensorMap
// descriptors through the driver's cuTensorMapEncodeTiled, reached with
// cudaGetDriverEntryPointByVersion so that the library needs no link against
// libcuda.
#pragma once

#include <cuda.h>

namespace gdn {

// Whether the driver exposes cuTensorMapEncodeTiled (looked up once).
bool tma_encoder_available();

// Encode a tiled map of `rank` dimensions (innermost first): dims in
// elements, strides in bytes for dimensions 1..rank-1, box in elements,
// element strides 1, no interleave, 256-byte L2 promotion, zero fill for
// out-of-bounds elements.  False when the encoder is missing or rejects the
// arguments (misaligned base or strides, box too large, ...).
bool tma_encode(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *ptr, const cuuint64_t *dims,
                const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle sw);

}  // namespace gdn
