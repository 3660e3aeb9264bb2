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

// Readies kernel `fn` for launches of `threads` threads with `smem` bytes of
// dynamic shared memory on the current device and returns (in *ctas_per_sm,
// if not null) how many such CTAs fit on an SM.  The attribute call and the
// occupancy query run once per (device, kernel, shape); later calls hit a
// small cache, so a launch costs the host little more than the launch itself.
int prepare_kernel(const void *fn, int threads, int smem, int *ctas_per_sm);

inline bool aligned(const void *p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

}  // namespace pkv
