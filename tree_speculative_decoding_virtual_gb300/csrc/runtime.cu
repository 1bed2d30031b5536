// Host-side state shared by the entry points: device properties, process-wide
// options, version.

#include <atomic>
#include <mutex>

#include "tsd_common.cuh"

namespace tsd {

int sm_count() {
  // one value per device; a relaxed atomic is enough (every thread that fills
  // it stores the same number)
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

static int64_t g_options[TSD_OPT_COUNT] = {
    2000000000LL,  // TSD_OPT_WAIT_LIMIT_NS: 2 s
    0,             // TSD_OPT_TEST_STALL: off
};

int64_t option(int key) { return (key >= 0 && key < TSD_OPT_COUNT) ? g_options[key] : 0; }

bool set_smem(const void *kernel, size_t bytes) {
  // (kernel, device) pairs whose limit is already raised, under a mutex so
  // that concurrent first calls from several host threads are safe
  struct Entry {
    const void *fn;
    int dev;
  };
  static std::mutex mu;
  static Entry done[64];
  static int n_done = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i].fn == kernel && done[i].dev == dev) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess)
    return false;
  if (n_done < 64) done[n_done++] = Entry{kernel, dev};
  return true;
}

}  // namespace tsd

TSD_API const char *tsd_version(void) { return "tsd 0.2 (sm_103a)"; }

TSD_API int tsd_set_option(int key, int64_t value) {
  if (key < 0 || key >= TSD_OPT_COUNT) return TSD_ERR_ARG;
  if (key == TSD_OPT_WAIT_LIMIT_NS && value < 0) return TSD_ERR_ARG;
  if (key == TSD_OPT_TEST_STALL && (value < 0 || value > 1)) return TSD_ERR_ARG;
  tsd::g_options[key] = value;
  return TSD_OK;
}

TSD_API int64_t tsd_get_option(int key) { return tsd::option(key); }
