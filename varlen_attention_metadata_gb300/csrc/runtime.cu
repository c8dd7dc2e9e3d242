// Host-side state of libpseq: error text, launch counter, device properties,
// bounded-wait settings.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <set>
#include <tuple>

#include "common.cuh"

namespace pseq {

namespace {
thread_local char g_last_error[512] = "";
std::atomic<int64_t> g_launches{0};
constexpr int64_t kDefaultWaitNs = 1000000000;  // 1 s
std::atomic<int64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int64_t> g_withhold{-1};
std::mutex g_dev_mu;
int g_sm_count[64] = {0};
}  // namespace

pseq_status fail(pseq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_last_error[0] = '\0'; }

pseq_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return PSEQ_OK;
}

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int occupancy(const void* kernel, int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, size_t>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_tuple(dev, kernel, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) n = 1;
  cache[key] = n;
  return n;
}

cudaError_t allow_dynamic_smem(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::set<std::tuple<int, const void*, size_t>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_tuple(dev, kernel, bytes);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count(key)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done.insert(key);
  return e;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (dev >= 64) {
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
  }
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

int64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int64_t withhold_tile() { return g_withhold.load(std::memory_order_relaxed); }

}  // namespace pseq

extern "C" {

int pseq_version(void) { return 100; }

const char* pseq_last_error(void) { return pseq::g_last_error; }

int64_t pseq_launch_count(void) { return pseq::g_launches.load(std::memory_order_relaxed); }

void pseq_debug_set_wait(int64_t spin_limit_ns, int64_t withhold_tile) {
  // a negative limit restores the default; no limit may exceed it, so no
  // caller can make a device-side wait (withheld tile or not) unbounded
  int64_t ns = spin_limit_ns >= 0 ? spin_limit_ns : pseq::kDefaultWaitNs;
  if (ns > pseq::kDefaultWaitNs) ns = pseq::kDefaultWaitNs;
  pseq::g_wait_ns.store(ns);
  pseq::g_withhold.store(withhold_tile >= 0 ? withhold_tile : -1);
}

int64_t pseq_debug_wait_limit_ns(void) { return pseq::wait_limit_ns(); }

}  // extern "C"
