// Per-device launch facts of the CSA2 library (host code only).
//
// A few launch parameters depend on the device a call runs on: its SM count, how many
// CTAs of a kernel fit on one SM, and the opt-in to more than 48 KB of dynamic shared
// memory, which CUDA records per function and per device.  They are computed on a
// device's first call and kept in one table keyed by (device, site, key), guarded by a
// mutex, so calls from several host threads and on several devices each see their own
// device's values.  This table is the only state the library keeps between calls, apart
// from the workspace-free Reindex entry's static scratch array.
#include <map>
#include <mutex>
#include <tuple>


#include "launch.h"

namespace csa2 {

namespace {
std::mutex g_memo_mu;
std::map<std::tuple<int, int, int64_t>, int> g_memo;
}  // namespace

int memo_lookup(int device, int site, int64_t key, const std::function<int()> &make) {
  const auto k = std::make_tuple(device, site, key);
  std::lock_guard<std::mutex> lock(g_memo_mu);
  auto it = g_memo.find(k);
  if (it != g_memo.end()) return it->second;
  const int v = make();
  if (v >= 0) g_memo.emplace(k, v);       // a failure (negative) is retried on the next call
  return v;
}

int device_memo(int site, int64_t key, const std::function<int()> &make) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return make();
  return memo_lookup(dev, site, key, make);
}

int opt_in_smem(const void *kernel, size_t bytes, int site, int64_t key) {
  return device_memo(site, key, [&] {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess ? 1
                                                                                                              : -1;
  });
}

int num_sms() {
  return device_memo(kSiteNumSms, 0, [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || n <= 0)
      return -1;
    return n;
  });
}

}  // namespace csa2

// Test-only view of the table with an explicit device id (no CUDA call): the value stored
// for (device, site, key), or `value` stored now if there is none.
extern "C" int csa2_test_device_memo(int device, int site, int64_t key, int value) {
  return csa2::memo_lookup(device, site, key, [value] { return value; });
}
