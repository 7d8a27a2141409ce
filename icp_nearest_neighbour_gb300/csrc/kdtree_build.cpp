// Host KD-tree build ("Implementing ICP with CUDA-KDTree", sections 2.2, 2.3,
// 4.2, 5.1, 5.2): split on the axis of largest variance (or, as the section
// 4.2 alternative, round robin x, y, z by depth) at the median, stop at
// leaf_size points or at the depth cap, partition in place with nth_element.
// The array partitioned is the 16-byte point records themselves (x, y, z,
// original index), reserved once up front: every pass over a node reads
// memory sequentially, and when the build ends the array is already the
// leaf-ordered record array the device search reads.  Subtrees near the root
// are built on separate threads; the result does not depend on the threading.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <exception>
#include <future>
#include <new>
#include <thread>

#include "icpnn_internal.h"

namespace icpnn {
namespace {

struct Rec {
  float c[3];
  int32_t idx;
};
static_assert(sizeof(Rec) == 16, "record must match the device float4 layout");

struct Builder {
  int32_t leaf_size = 0;
  int32_t max_depth = 0;
  Rec* recs = nullptr;  // point records, partitioned in place
  Node* heap = nullptr;
  int parallel_depth = 0;
  bool round_robin = false;  // axis = depth mod 3 instead of largest variance
  std::atomic<int64_t> n_nodes{0};

  // Axis of largest population variance; axes within a relative 1e-9 of the
  // largest are tied and the lowest of them wins.
  int split_axis(int64_t lo, int64_t hi) const {
    // two passes (mean, then squared deviations) with the three axes fused;
    // each axis still sums its terms in index-array order
    const double cnt = static_cast<double>(hi - lo);
    double sum[3] = {0.0, 0.0, 0.0};
    for (int64_t i = lo; i < hi; ++i) {
      const float* p = recs[i].c;
      sum[0] += p[0];
      sum[1] += p[1];
      sum[2] += p[2];
    }
    const double mean[3] = {sum[0] / cnt, sum[1] / cnt, sum[2] / cnt};
    double ss[3] = {0.0, 0.0, 0.0};
    for (int64_t i = lo; i < hi; ++i) {
      const float* p = recs[i].c;
      for (int d = 0; d < 3; ++d) {
        const double e = p[d] - mean[d];
        ss[d] += e * e;
      }
    }
    double var[3];
    for (int d = 0; d < 3; ++d) var[d] = ss[d] / cnt;
    const double vmax = std::max(var[0], std::max(var[1], var[2]));
    for (int d = 0; d < 3; ++d)
      if (var[d] >= vmax * (1.0 - 1e-9)) return d;
    return 0;
  }

  void build(uint64_t node, int64_t lo, int64_t hi, int depth) {
    n_nodes.fetch_add(1, std::memory_order_relaxed);
    const int64_t count = hi - lo;
    if (count <= leaf_size || depth >= max_depth) {
      heap[node].a = static_cast<uint32_t>(lo);
      heap[node].meta = kLeafTag | (static_cast<uint32_t>(count) << 2);
      return;
    }
    const int axis = round_robin ? depth % 3 : split_axis(lo, hi);
    const int64_t m = count / 2;
    std::nth_element(recs + lo, recs + lo + m, recs + hi, [axis](const Rec& a, const Rec& b) {
      return a.c[axis] < b.c[axis] || (a.c[axis] == b.c[axis] && a.idx < b.idx);
    });
    const float split = recs[lo + m].c[axis];
    uint32_t bits;
    std::memcpy(&bits, &split, sizeof(bits));
    heap[node].a = bits;
    heap[node].meta = static_cast<uint32_t>(axis);
    if (depth < parallel_depth && count >= (1 << 13)) {
      std::future<void> left;
      try {
        left = std::async(std::launch::async, [=] { build(2 * node, lo, lo + m, depth + 1); });
      } catch (const std::exception&) {
        build(2 * node, lo, lo + m, depth + 1);
        build(2 * node + 1, lo + m, hi, depth + 1);
        return;
      }
      build(2 * node + 1, lo + m, hi, depth + 1);
      left.get();
    } else {
      build(2 * node, lo, lo + m, depth + 1);
      build(2 * node + 1, lo + m, hi, depth + 1);
    }
  }
};

// Deepest level that holds a node.  With median splits the nodes at depth k
// hold floor or ceil of n / 2^k points, so the tree stops at the first k whose
// largest node fits in a leaf, or at the cap.
int32_t tree_depth(int64_t n, int32_t leaf_size, int32_t max_depth) {
  int32_t d = 0;
  while (d < max_depth) {
    const int64_t largest = (n + (int64_t{1} << d) - 1) >> d;
    if (largest <= leaf_size) break;
    ++d;
  }
  return d;
}

}  // namespace

int build_tree(const float* xyz, int64_t n, int32_t leaf_size, int32_t max_depth, bool round_robin,
               icpnn_tree* t) {
  for (int64_t i = 0; i < 3 * n; ++i)
    if (!std::isfinite(xyz[i]))
      return fail(ICPNN_ERR_NONFINITE, "kdtree_build: non-finite coordinate at point " +
                                           std::to_string(i / 3));
  const int32_t depth = tree_depth(n, leaf_size, max_depth);
  const int64_t largest_leaf = (n + (int64_t{1} << depth) - 1) >> depth;
  if (largest_leaf >= (int64_t{1} << 30))
    return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build: a leaf would hold 2^30 points or more");
  try {
    t->n = n;
    t->leaf_size = leaf_size;
    t->max_depth = max_depth;
    t->round_robin = round_robin;
    t->depth = depth;
    t->heap_slots = int64_t{1} << (depth + 1);
    t->nodes.assign(static_cast<size_t>(t->heap_slots), Node{0u, 0u});
    t->records.resize(static_cast<size_t>(4 * n));
    Rec* recs = reinterpret_cast<Rec*>(t->records.data());
    float lo[3] = {INFINITY, INFINITY, INFINITY};
    float hi[3] = {-INFINITY, -INFINITY, -INFINITY};
    for (int64_t i = 0; i < n; ++i) {
      for (int d = 0; d < 3; ++d) {
        const float v = xyz[3 * i + d];
        recs[i].c[d] = v;
        lo[d] = std::min(lo[d], v);
        hi[d] = std::max(hi[d], v);
      }
      recs[i].idx = static_cast<int32_t>(i);
    }
    for (int d = 0; d < 3; ++d) {
      t->bbox_lo[d] = lo[d];
      t->bbox_hi[d] = hi[d];
    }

    Builder b;
    b.leaf_size = leaf_size;
    b.max_depth = max_depth;
    b.recs = recs;
    b.heap = t->nodes.data();
    b.round_robin = round_robin;
    const unsigned hw = std::max(1u, std::thread::hardware_concurrency());
    int pd = 0;
    while ((1u << pd) < 4 * hw && pd < 8) ++pd;
    b.parallel_depth = pd;
    b.build(1, 0, n, 0);
    t->n_nodes = b.n_nodes.load();
  } catch (const std::bad_alloc&) {
    return fail(ICPNN_ERR_NO_MEMORY, "kdtree_build: host allocation failed");
  }
  return ICPNN_OK;
}

}  // namespace icpnn
