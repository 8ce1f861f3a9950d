// cuTensorMapEncodeTiled through the runtime's driver entry point: the
// library does not link libcuda directly, so it loads on machines without a
// driver.
#pragma once
#include <cuda.h>

namespace mla {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The encoder, or nullptr when the driver does not provide it.
EncodeTiledFn tensor_map_encoder();

}  // namespace mla
