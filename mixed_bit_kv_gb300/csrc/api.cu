// Host-side support shared by the rdkv_* entry points: the thread-local error
// message, CUDA error mapping and the cached SM count used for grid sizing.
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

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

}  // namespace rdkv

extern "C" const char* rdkv_last_error_string(void) { return rdkv::g_err; }

extern "C" int32_t rdkv_version(void) { return 1; }
