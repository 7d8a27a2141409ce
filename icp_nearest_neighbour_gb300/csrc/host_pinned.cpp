// Process-wide cache of page-locked host blocks for the tree's host arrays.
//
// A tree is built on the host and uploaded once; from pageable memory the
// driver stages the copy through pinned buffers of its own, from page-locked
// memory it is one DMA.  Page-locking is slow (it maps and pins every page),
// so freed blocks are kept and handed out again to requests they can hold
// without wasting more than half of themselves; at most kKeepBytes stay
// cached, the rest is returned to the system.  Without a CUDA device (or if
// page-locking fails) the blocks are ordinary aligned memory.
#include <atomic>
#include <cstdlib>
#include <map>
#include <mutex>
#include <new>
#include <unordered_map>

#include "icpnn_internal.h"

namespace icpnn {
namespace {

constexpr size_t kGranule = size_t{64} << 10;
constexpr size_t kKeepBytes = size_t{512} << 20;

struct Block {
  size_t capacity;
  bool pinned;
};

struct PinnedCache {
  std::mutex mu;
  std::unordered_map<void*, Block> live;      // every block handed out
  std::multimap<size_t, void*> idle;          // freed blocks by capacity
  std::unordered_map<void*, Block> idle_info;
  size_t idle_bytes = 0;
};

PinnedCache& cache() {
  static PinnedCache* c = new PinnedCache();  // never destroyed: CUDA may be gone at exit
  return *c;
}

void release(void* p, const Block& b) {
  if (b.pinned) {
    cudaFreeHost(p);
    cudaGetLastError();
  } else {
    std::free(p);
  }
}

}  // namespace

void* pinned_alloc(size_t bytes) {
  const size_t want = ((bytes == 0 ? 1 : bytes) + kGranule - 1) / kGranule * kGranule;
  PinnedCache& c = cache();
  {
    std::lock_guard<std::mutex> lock(c.mu);
    auto it = c.idle.lower_bound(want);
    if (it != c.idle.end() && it->first <= 2 * want) {
      void* p = it->second;
      const Block b = c.idle_info[p];
      c.idle_info.erase(p);
      c.idle.erase(it);
      c.idle_bytes -= b.capacity;
      c.live[p] = b;
      return p;
    }
  }
  void* p = nullptr;
  bool pinned = false;
  // no device or driver: ordinary memory from now on, without asking again
  static std::atomic<bool> no_device{false};
  if (!no_device.load(std::memory_order_relaxed)) {
    const cudaError_t e = cudaHostAlloc(&p, want, cudaHostAllocPortable);
    if (e == cudaSuccess) {
      pinned = true;
    } else {
      cudaGetLastError();
      p = nullptr;
      if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver || e == cudaErrorInitializationError)
        no_device.store(true, std::memory_order_relaxed);
    }
  }
  if (p == nullptr) {
    p = std::aligned_alloc(256, want);
    if (p == nullptr) throw std::bad_alloc();
  }
  std::lock_guard<std::mutex> lock(c.mu);
  c.live[p] = Block{want, pinned};
  return p;
}

void pinned_free(void* p) noexcept {
  if (p == nullptr) return;
  PinnedCache& c = cache();
  std::lock_guard<std::mutex> lock(c.mu);
  auto it = c.live.find(p);
  if (it == c.live.end()) return;
  const Block b = it->second;
  c.live.erase(it);
  if (c.idle_bytes + b.capacity > kKeepBytes) {
    release(p, b);
    return;
  }
  c.idle.emplace(b.capacity, p);
  c.idle_info[p] = b;
  c.idle_bytes += b.capacity;
}

}  // namespace icpnn
