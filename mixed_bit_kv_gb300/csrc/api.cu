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

// One workspace query for the calls that take a shape.  The decode's value is a bound over every
// single cache of the shape: its grid holds at most one dealt block per SM plus one spare block per
// head, each with a partial of G (D + 2) floats (rounded up to four), then the per-head tickets, the
// status word and the fused step's head counter (the layout of the decode's own workspace query).
extern "C" size_t rdkv_workspace_bytes(const rdkv_shape* shape, int32_t which_call) {
  using namespace rdkv;
  if (check_shape(shape) != RDKV_OK) return 0;
  switch (which_call) {
    case RDKV_CALL_SCORE:
      return rdkv_score_workspace_bytes(shape);
    case RDKV_CALL_ALLOCATE:
      return rdkv_allocate_workspace_bytes(shape);
    case RDKV_CALL_DECODE: {
      const int64_t n_heads = (int64_t)shape->batch * shape->h_kv;
      const int64_t partial = decode_partial_stride(shape->h_q / shape->h_kv, shape->head_dim);
      // up to two blocks per SM plus one spare block per head (launches over many heads)
      return (size_t)(align_up((2 * num_sms() + n_heads) * partial * 4, 256) + decode_ticket_bytes(n_heads));
    }
    default:
      return 0;
  }
}
