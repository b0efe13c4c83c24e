// pkv_host.h -- host-side helpers shared by the libpagedkv translation units
// (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

// Device address of the current device's status word (nullptr on failure).
unsigned int *status_word_ptr();

// Streaming-multiprocessor count of the current device (0 on failure).
int current_sm_count();

// Count one kernel launch made through the library.
void count_launch();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline pkv_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
