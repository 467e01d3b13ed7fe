// Host side of the TMA tensor copies: cuTensorMapEncodeTiled, reached
// through the runtime's driver entry point so that the library does not
// link the driver library directly.
#pragma once

#include <cuda.h>  // CUtensorMap and the encoder's argument types
#include <cuda_runtime.h>

namespace tt {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The encoder, looked up once per process; nullptr if the driver lacks it.
EncodeTiledFn tensor_map_encoder();

}  // namespace tt
