// Internal declarations shared by the host and device parts of libicpnn.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <functional>
#include <memory>
#include <string>
#include <utility>
#include <vector>

#include "icpnn.h"

namespace icpnn {

// ---------------------------------------------------------------------------
// Device tree layout.
//
// The page's node (section 3.1) is a 24-byte record with explicit child links
// and a [start, end) range into a separate leaf index table.  Here the tree is
// stored as an implicit binary heap, 1-based: the root is node 1 and the
// children of node i are 2i and 2i+1, so siblings share one 16-byte-aligned
// pair and a single vector load fetches both children of a node.  With median
// splits every node at depth k holds floor or ceil of n / 2^k points, so leaves
// sit on at most two adjacent levels and the heap wastes at most half its
// slots.
//
// Each node is 8 bytes {uint32 a, uint32 meta}:
//   inner: a = float bits of the split value, meta = split axis (0, 1, 2)
//   leaf : a = first point record,            meta = 3 | (count << 2)
// Slot 0 is unused (zeroed).
//
// Beside the nodes, every node has the tight bounding box of its points (two
// float4, lo and hi).  The search keeps the page's splitting-plane test and
// adds the box test where it prunes most: before it takes up a pending sibling
// subtree and before it scans a leaf it descended to.
//
// Points are stored in leaf order as float4 records {x, y, z, index bits}:
// one 16-byte load returns both the coordinates and the original target index
// (the page's leaf_index indirection, section 3.2, disappears).
// ---------------------------------------------------------------------------
struct Node {
  uint32_t a;
  uint32_t meta;
};
static_assert(sizeof(Node) == 8, "node must be 8 bytes");

constexpr uint32_t kLeafTag = 3u;

inline bool node_is_leaf(const Node& n) { return (n.meta & 3u) == kLeafTag; }

struct DeviceTree {
  int device = -1;
  Node* nodes = nullptr;      // heap_slots entries; the boxes follow in the same allocation
  float* boxes = nullptr;     // heap_slots x 8 floats
  float* points = nullptr;    // n float4 records (x, y, z, index bits)
  // Recorded after the upload's copies, which the upload does not wait for:
  // every call that uses the tree makes its stream wait on it first.
  cudaEvent_t ready = nullptr;
};

}  // namespace icpnn

namespace icpnn {

// Allocator whose value-less construct leaves the element uninitialised, so
// that resizing a vector the caller is about to overwrite costs no fill.
template <class T>
struct UninitAllocator : std::allocator<T> {
  template <class U>
  struct rebind {
    using other = UninitAllocator<U>;
  };
  UninitAllocator() = default;
  template <class U>
  UninitAllocator(const UninitAllocator<U>&) noexcept {}
  template <class U>
  void construct(U* p) noexcept {
    ::new (static_cast<void*>(p)) U;
  }
  template <class U, class... A>
  void construct(U* p, A&&... a) {
    ::new (static_cast<void*>(p)) U(std::forward<A>(a)...);
  }
};
// Page-locked host memory when a CUDA device is present (ordinary memory
// otherwise), from a process-wide cache of freed blocks (host_pinned.cpp):
// the tree's host arrays, so that the upload is a plain DMA rather than a
// copy staged through the driver's pinned buffers.
void* pinned_alloc(size_t bytes);
void pinned_free(void* p) noexcept;

template <class T>
struct PinnedAllocator : UninitAllocator<T> {
  using value_type = T;
  template <class U>
  struct rebind {
    using other = PinnedAllocator<U>;
  };
  PinnedAllocator() = default;
  template <class U>
  PinnedAllocator(const PinnedAllocator<U>&) noexcept {}
  T* allocate(size_t n) { return static_cast<T*>(pinned_alloc(n * sizeof(T))); }
  void deallocate(T* p, size_t) noexcept { pinned_free(p); }
  template <class U>
  bool operator==(const PinnedAllocator<U>&) const noexcept { return true; }
  template <class U>
  bool operator!=(const PinnedAllocator<U>&) const noexcept { return false; }
};
template <class T>
using PinnedVector = std::vector<T, PinnedAllocator<T>>;

}  // namespace icpnn

struct icpnn_tree {
  int64_t n = 0;
  int32_t leaf_size = 0;
  int32_t max_depth = 0;
  int32_t depth = 0;          // deepest level holding a node (root = 0)
  bool round_robin = false;   // split axis = depth mod 3 (else largest variance)
  int64_t n_nodes = 0;        // nodes in use
  int64_t heap_slots = 0;     // 2^(depth+1)
  float bbox_lo[3] = {0, 0, 0};
  float bbox_hi[3] = {0, 0, 0};
  icpnn::PinnedVector<icpnn::Node> nodes;   // heap layout, heap_slots entries
  icpnn::PinnedVector<float> records;       // 4 floats per point, leaf order
  // Tight bounding box of each node's points, 8 floats per heap slot:
  // lo.x, lo.y, lo.z, 0, hi.x, hi.y, hi.z, 0 (unused slots zero).
  icpnn::PinnedVector<float> boxes;
  icpnn::DeviceTree dev;
  // Built on the device: nodes, boxes and records exist there only until a
  // caller needs them on the host (export, upload to another device).
  bool host_stale = false;
};

namespace icpnn {

// Thread-local error message; returns `code` so callers can `return fail(...)`.
int fail(int code, const std::string& msg);
void clear_error();

// Stream-ordered allocation from the library's own memory pool on the
// current device (api.cu); free with cudaFreeAsync.  Up to 1 GiB of freed
// memory stays reserved between calls, and a block freed on one stream is
// reused on another only through an event dependency: with the default
// pool's opportunistic cross-stream reuse, registrations that had run on
// eight streams left every later tree build on a ninth 40% slower.
cudaError_t pool_alloc(void** p, size_t bytes, cudaStream_t s);

// Host tree build (kdtree_build.cpp).
int build_tree(const float* xyz, int64_t n, int32_t leaf_size, int32_t max_depth, bool round_robin,
               icpnn_tree* t);
int32_t tree_depth(int64_t n, int32_t leaf_size, int32_t max_depth);

// Device tree build (kdtree_build_gpu.cu): the same tree from device points,
// left in t->dev; the host arrays are filled on demand (host_stale).
int build_tree_device(const float* xyz_dev, int64_t n, int32_t leaf_size, int32_t max_depth, bool round_robin,
                      icpnn_tree* t, cudaStream_t s);

// Process-wide host worker pool (host_pool.cpp).  pool_submit queues a job
// (ensuring at least min_threads workers); parallel_for runs fn(0..tasks-1)
// on the pool with the caller taking part, so nested use cannot deadlock;
// the first exception a task throws is rethrown to the caller.
void pool_submit(std::function<void()> job, int min_threads);
void parallel_for(int tasks, const std::function<void(int)>& fn);
// Wakes parked workers ahead of a burst of parallel_for calls.
void pool_wake();

// Host Kabsch solve (kabsch.cpp).  Returns ICPNN_OK or ICPNN_ERR_DEGENERATE.
int kabsch_solve(const icpnn_moments& m, double T[16]);

}  // namespace icpnn
