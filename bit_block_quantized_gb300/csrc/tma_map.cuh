// tma_map.cuh -- host access to the driver's tiled tensor-map encoder, shared
// by the kernels that stream weights with the tensor-memory accelerator.
#pragma once

#include <cuda.h>  // CUtensorMap and the encode signature; the function is fetched at run time

namespace q4 {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (null if
// the driver does not provide it).
EncodeTiledFn encode_fn();

}  // namespace q4
