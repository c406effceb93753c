// Host-side tensor-map helpers shared by the tensor-core conv launchers.
#pragma once
#include <cuda.h>

namespace vd {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver (resolved once through the runtime), or null.
EncodeTiledFn get_encode_fn();

// Swizzle mode whose span equals a K chunk of `bk` bf16 values (64 -> 128B, 32 -> 64B, 16 -> 32B).
CUtensorMapSwizzle swizzle_for(int bk);

}  // namespace vd
