// fp8gb_host.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8gb.h"

namespace fp8gb {

// Number of SMs of the current device (cached per device).
int num_sms();

// Device address of the library's error word on the current device (looked
// up once per device; NULL if the lookup failed).
unsigned int *device_error_word();

// Record a CUDA error (thread-local message) and return FP8_ERR_CUDA.
fp8_status_t cuda_fail_with(cudaError_t e);
inline fp8_status_t cuda_fail() { return cuda_fail_with(cudaGetLastError()); }

// Status of the last kernel launch.
inline fp8_status_t check_launch()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FP8_OK : cuda_fail_with(e);
}

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace fp8gb
