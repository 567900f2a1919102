// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsa_cp.h"

namespace dsa {

// Device address of the library's error word on the current device (set up
// once per device); nullptr if the lookup failed (the CUDA error is recorded).
int *device_error_word();

// Record `e` as the last CUDA error of this thread and return DSA_ERR_CUDA.
dsa_status cuda_fail(cudaError_t e);
dsa_status cuda_fail_msg(const char *msg);

// Launch-error check after a kernel launch.
inline dsa_status check_launch() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
// rank <= 3; dims/strides in elements/bytes as the driver API expects
// (strides exclude the innermost dimension).
dsa_status encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t rank, const void *base,
                             const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                             CUtensorMapSwizzle swizzle);

int num_sms();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace dsa
