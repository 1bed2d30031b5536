// Internal helpers shared by the libtsd translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

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

// Programmatic dependent launch: every kernel of the library is launched so
// that it may start while the previous kernel on the stream finishes; each
// kernel lets its own dependents launch at entry (pdl_trigger; the kernels
// that write the K/V cache or the slot record release them only when they
// end) and waits for the previous grid's completion and memory (pdl_wait)
// before it reads that grid's results and before its first global write
// (the attention under the uniform split reads its inputs before the wait).
// After a kernel that does not trigger, this is an ordinary stream-ordered
// launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Opt a kernel in to `bytes` of dynamic shared memory (needed once static
// plus dynamic exceeds 48 KB), once per (kernel, device).
bool set_smem(const void *kernel, size_t bytes);

inline bool aligned(const void *p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

}  // namespace tsd
