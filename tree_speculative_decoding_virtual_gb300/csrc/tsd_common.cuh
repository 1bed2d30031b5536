// Internal helpers shared by the libtsd translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tsd.h"

#define TSD_API extern "C" __attribute__((visibility("default")))

namespace tsd {

constexpr int kPage = 16;        // token slots per KV-cache block
constexpr int kMaxNodes = 256;   // N_max limit
constexpr int kMaxDepth = 32;    // D_max limit

inline cudaStream_t as_cuda(tsd_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? TSD_OK : TSD_ERR_CUDA;
}

// Streaming multiprocessor count of the current device (cached per device).
int sm_count();

// Process-wide option (see tsd_set_option).
int64_t option(int key);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned(const void *p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

}  // namespace tsd
