// Small thread-safe host cache for launch plans, keyed by the raw bytes of
// a zero-initialised key struct (so padding never makes two keys differ).
#pragma once

#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>

namespace gconv {

template <typename V>
class PlanCache {
 public:
  template <typename K>
  bool get(const K& key, V* out) {
    std::lock_guard<std::mutex> g(mu_);
    auto it = map_.find(bytes(key));
    if (it == map_.end()) return false;
    *out = it->second;
    return true;
  }
  template <typename K>
  void put(const K& key, const V& v) {
    std::lock_guard<std::mutex> g(mu_);
    if (map_.size() > 4096) map_.clear();
    map_[bytes(key)] = v;
  }

 private:
  template <typename K>
  static std::string bytes(const K& k) {
    return std::string(reinterpret_cast<const char*>(&k), sizeof(K));
  }
  std::mutex mu_;
  std::unordered_map<std::string, V> map_;
};

// Raises a kernel's dynamic shared-memory limit once per device (and again
// only if a larger size is needed).
struct SmemAttr {
  std::atomic<int> done[64] = {};
  template <typename F>
  cudaError_t ensure(F* kern, int device, int bytes) {
    if (device < 0 || device >= 64) return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (done[device].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) {
      int cur = done[device].load();
      while (cur < bytes && !done[device].compare_exchange_weak(cur, bytes)) {
      }
    }
    return e;
  }
};

}  // namespace gconv
