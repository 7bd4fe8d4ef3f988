// launch_cache.h -- per-device launch facts of the library's kernels (host code).
//
// Grid sizes depend on the device they run on (SM count, occupancy at a given
// shared-memory size), and kernel attributes such as the dynamic shared-memory
// limit are set per device. A process may drive several GPUs from several host
// threads, so every such fact is cached per (device, kernel, shared memory, tag):
// the first lookup of a key runs its query (which may call the CUDA runtime and
// set attributes on the current device), later lookups return the stored value.
// Thread-safe; queries run outside the lock, and when two threads race on a new
// key the first stored value wins (both computed the same fact).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include <mutex>
#include <vector>

namespace sv {

class LaunchCache {
 public:
  template <typename Query>
  cudaError_t get(int dev, const void* fn, size_t smem, int tag, int* out, Query&& query) {
    if (find(dev, fn, smem, tag, out)) return cudaSuccess;
    int v = 0;
    const cudaError_t e = query(&v);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> g(mu_);
    for (const Entry& x : entries_)
      if (x.dev == dev && x.fn == fn && x.smem == smem && x.tag == tag) {
        *out = x.value;
        return cudaSuccess;
      }
    entries_.push_back(Entry{dev, fn, smem, tag, v});
    *out = v;
    return cudaSuccess;
  }
  size_t size() {
    std::lock_guard<std::mutex> g(mu_);
    return entries_.size();
  }

 private:
  struct Entry {
    int dev;
    const void* fn;
    size_t smem;
    int tag;
    int value;
  };
  bool find(int dev, const void* fn, size_t smem, int tag, int* out) {
    std::lock_guard<std::mutex> g(mu_);
    for (const Entry& x : entries_)
      if (x.dev == dev && x.fn == fn && x.smem == smem && x.tag == tag) {
        *out = x.value;
        return true;
      }
    return false;
  }
  std::mutex mu_;
  std::vector<Entry> entries_;
};

}  // namespace sv
