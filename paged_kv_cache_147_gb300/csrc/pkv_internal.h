// pkv_internal.h -- host helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/pkv.h"

namespace pkv {

// Status for a CUDA runtime error code.
inline int cuda_status(cudaError_t e) {
  return e == cudaSuccess ? PKV_OK : PKV_ECUDA_BASE - static_cast<int>(e);
}

// Device address of the current device's error word (nullptr if it cannot be resolved).
unsigned int* device_error_ptr();

// SM count of the current device (0 on failure).
int sm_count();

// cuTensorMapEncodeTiled from the driver, resolved once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool valid_block_size(int bs) {
  return bs == 16 || bs == 32 || bs == 64 || bs == 128 || bs == 256;
}

}  // namespace pkv
