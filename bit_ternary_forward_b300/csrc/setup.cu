// Per-device, thread-safe kernel set-up.
//
// A kernel that needs more than 48 KB of dynamic shared memory must have its
// limit raised with cudaFuncSetAttribute, which acts on the device current in
// the calling thread; the resident CTAs per SM that the launch plans use
// follow from that limit. Both are done once per (device, kernel) and kept in
// one table under a mutex, so several host threads and several devices in one
// process may make their first calls at the same time.

#include <map>
#include <mutex>
#include <tuple>

#include "kernels.cuh"

namespace bl {

namespace {

std::mutex g_setup_mu;
// (device, kernel) -> the largest dynamic shared-memory limit set so far
std::map<std::pair<int, const void*>, size_t> g_smem_limit;
// (device, kernel, threads, bytes) -> resident CTAs per SM
std::map<std::tuple<int, const void*, int, size_t>, int> g_resident;

cudaError_t ensure_smem_locked(int dev, const void* func, size_t bytes) {
  size_t& done = g_smem_limit[{dev, func}];
  if (bytes <= done) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) done = bytes;
  return e;
}

}  // namespace

cudaError_t ensure_smem(const void* func, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;   // the default limit
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  return ensure_smem_locked(dev, func, bytes);
}

int resident_ctas(const void* func, int threads, size_t bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  const auto key = std::make_tuple(dev, func, threads, bytes);
  const auto it = g_resident.find(key);
  if (it != g_resident.end()) return it->second;
  int n = 0;
  if ((bytes > 48 * 1024 && ensure_smem_locked(dev, func, bytes) != cudaSuccess) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, bytes) != cudaSuccess)
    return 0;   // not cached: a later call may succeed
  g_resident[key] = n;
  return n;
}

}  // namespace bl
