// Error reporting and small process-wide bookkeeping of the C ABI.
#include <atomic>
#include <cstdlib>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "internal.h"

namespace sar {

namespace {
thread_local std::string g_last_error = "no error";
std::atomic<int64_t> g_launches{0};
std::mutex g_attr_mu;
std::map<std::pair<const void*, int>, int> g_smem_set;         // (kernel, device) -> bytes set
std::map<std::tuple<const void*, int, int>, int> g_clusters;  // (kernel, cluster, device) -> clusters
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

int ensure_smem_attr(const void* fn, int bytes, const char* what) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, what);
  std::lock_guard<std::mutex> lk(g_attr_mu);
  auto it = g_smem_set.find({fn, dev});
  if (it != g_smem_set.end() && it->second >= bytes) return SAR_OK;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return cuda_error(e, what);
  g_smem_set[{fn, dev}] = bytes;
  return SAR_OK;
}

int max_active_clusters(const void* fn, const cudaLaunchConfig_t& qc, int cl, int* out, const char* what) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, what);
  std::lock_guard<std::mutex> lk(g_attr_mu);
  auto key = std::make_tuple(fn, cl, dev);
  auto it = g_clusters.find(key);
  if (it != g_clusters.end()) {
    *out = it->second;
    return SAR_OK;
  }
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, fn, &qc);
  if (e != cudaSuccess) return cuda_error(e, what);
  if (n < 1) return set_error(SAR_ERR_UNSUPPORTED, std::string(what) + ": no cluster fits an SM group");
  g_clusters[key] = n;
  *out = n;
  return SAR_OK;
}

}  // namespace sar

extern "C" {

const char* sar_last_error(void) { return sar::g_last_error.c_str(); }

int64_t sar_launch_count(void) { return sar::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
