// tmap.h -- host-side TMA tensor-map encoding (cuTensorMapEncodeTiled through
// the runtime's driver entry-point query; no libcuda link needed).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace dsv4 {

// Encode a tiled tensor map; dims[0] is innermost; strides_bytes[i] is the
// stride of dims[i + 1].  Returns false if the driver rejects it.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle);

// Number of SMs of the current device (152 when no device is visible).
int sm_count();

}  // namespace dsv4
