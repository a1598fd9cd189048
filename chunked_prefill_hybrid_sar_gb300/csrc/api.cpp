// Error reporting and small process-wide bookkeeping of the C ABI.
#include <atomic>
#include <cstdlib>
#include <string>

#include "internal.h"

namespace sar {

namespace {
thread_local std::string g_last_error = "no error";
std::atomic<int64_t> g_launches{0};
}  // namespace

int set_error(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_error(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return SAR_OK;
  const int code = (e == cudaErrorMemoryAllocation) ? SAR_ERR_OOM : SAR_ERR_CUDA;
  return set_error(code, std::string(what) + ": " + cudaGetErrorString(e));
}

void count_launches(int64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("SAR_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  return n;
}

}  // namespace sar

extern "C" {

const char* sar_last_error(void) { return sar::g_last_error.c_str(); }

int64_t sar_launch_count(void) { return sar::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
