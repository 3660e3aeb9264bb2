// pkv_internal.h -- host-side helpers shared by the libpagedkv translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

struct ErrorRecord;

// Device address of the current device's error record (nullptr on failure;
// the CUDA error is then stored for pkv_last_error_string).
ErrorRecord *device_error_record();

// Remember a CUDA error's text for pkv_last_error_string; returns PKV_ERR_CUDA.
int cuda_failure(cudaError_t e, const char *where);

// Remember a message for pkv_last_error_string.
void set_last_error(const char *msg);

// Number of SMs of the current device (cached per device).
int sm_count();

inline bool aligned(const void *p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

}  // namespace pkv
