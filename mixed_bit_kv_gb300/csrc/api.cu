// Host-side support shared by the rdkv_* entry points: the thread-local error
// message, CUDA error mapping and the cached SM count used for grid sizing.
#include <atomic>
#include <cstdarg>

#include "common.cuh"

namespace rdkv {

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

rdkv_status cuda_status(cudaError_t e, const char* what) {
  set_error("%s: CUDA error %d (%s)", what, (int)e, cudaGetErrorString(e));
  return RDKV_ERR_CUDA;
}

static std::atomic<unsigned long long> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int num_sms() {
  static thread_local int cached_dev = -1, cached_n = 0;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev == cached_dev) return cached_n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  cached_dev = dev;
  cached_n = n;
  return n;
}

}  // namespace rdkv

extern "C" const char* rdkv_last_error_string(void) { return rdkv::g_err; }

extern "C" int32_t rdkv_version(void) { return 1; }

extern "C" uint64_t rdkv_launch_count(void) { return rdkv::g_launches.load(std::memory_order_relaxed); }
