// Tensor-core (tcgen05) contraction path.
#pragma once

#include <cuda_runtime.h>

#include "hcmix.h"
#include "hcmix_common.cuh"

namespace hcmix {

inline hcmix_status tc_launch(const uint16_t*, int64_t, const float*, int64_t, int64_t, int64_t,
                              uint16_t*, float*, int, uint32_t*, cudaStream_t) {
  return HCMIX_ERR_UNSUPPORTED;
}

}  // namespace hcmix
