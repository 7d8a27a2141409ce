// Host KD-tree build ("Implementing ICP with CUDA-KDTree", sections 2.2, 2.3,
// 4.2, 5.1, 5.2): split on the axis of largest variance at the median, stop at
// leaf_size points or at the depth cap, partition in place with nth_element
// into one index array reserved up front.  Subtrees near the root are built
// on separate threads; the result does not depend on the threading.
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

struct Builder {
  const float* xyz = nullptr;
  int32_t leaf_size = 0;
  int32_t max_depth = 0;
  int32_t* order = nullptr;  // point indices, partitioned in place
  Node* heap = nullptr;
  int parallel_depth = 0;
  std::atomic<int64_t> n_nodes{0};

  float coord(int32_t p, int d) const { return xyz[3 * static_cast<int64_t>(p) + d]; }

  // Axis of largest population variance; axes within a relative 1e-9 of the
  // largest are tied and the lowest of them wins.
  int split_axis(int64_t lo, int64_t hi) const {
    const double cnt = static_cast<double>(hi - lo);
    double var[3];
    for (int d = 0; d < 3; ++d) {
      double sum = 0.0;
      for (int64_t i = lo; i < hi; ++i) sum += coord(order[i], d);
      const double mean = sum / cnt;
      double ss = 0.0;
      for (int64_t i = lo; i < hi; ++i) {
        const double e = coord(order[i], d) - mean;
        ss += e * e;
      }
      var[d] = ss / cnt;
    }
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
    const int axis = split_axis(lo, hi);
    const int64_t m = count / 2;
    std::nth_element(order + lo, order + lo + m, order + hi, [this, axis](int32_t a, int32_t b) {
      const float fa = coord(a, axis), fb = coord(b, axis);
      return fa < fb || (fa == fb && a < b);
    });
    const float split = coord(order[lo + m], axis);
    uint32_t bits;
    std::memcpy(&bits, &split, sizeof(bits));
    heap[node].a = bits;
    heap[node].meta = static_cast<uint32_t>(axis);
    if (depth < parallel_depth && count >= (1 << 16)) {
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

int build_tree(const float* xyz, int64_t n, int32_t leaf_size, int32_t max_depth, icpnn_tree* t) {
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
    t->depth = depth;
    t->heap_slots = int64_t{1} << (depth + 1);
    t->nodes.assign(static_cast<size_t>(t->heap_slots), Node{0u, 0u});
    std::vector<int32_t> order(static_cast<size_t>(n));
    for (int64_t i = 0; i < n; ++i) order[static_cast<size_t>(i)] = static_cast<int32_t>(i);

    Builder b;
    b.xyz = xyz;
    b.leaf_size = leaf_size;
    b.max_depth = max_depth;
    b.order = order.data();
    b.heap = t->nodes.data();
    const unsigned hw = std::max(1u, std::thread::hardware_concurrency());
    int pd = 0;
    while ((1u << pd) < hw && pd < 6) ++pd;
    b.parallel_depth = pd;
    b.build(1, 0, n, 0);
    t->n_nodes = b.n_nodes.load();

    t->records.resize(static_cast<size_t>(4 * n));
    float lo[3] = {INFINITY, INFINITY, INFINITY};
    float hi[3] = {-INFINITY, -INFINITY, -INFINITY};
    for (int64_t k = 0; k < n; ++k) {
      const int32_t p = order[static_cast<size_t>(k)];
      float* r = &t->records[static_cast<size_t>(4 * k)];
      for (int d = 0; d < 3; ++d) {
        r[d] = xyz[3 * static_cast<int64_t>(p) + d];
        lo[d] = std::min(lo[d], r[d]);
        hi[d] = std::max(hi[d], r[d]);
      }
      std::memcpy(&r[3], &p, sizeof(float));
    }
    for (int d = 0; d < 3; ++d) {
      t->bbox_lo[d] = lo[d];
      t->bbox_hi[d] = hi[d];
    }
  } catch (const std::bad_alloc&) {
    return fail(ICPNN_ERR_NO_MEMORY, "kdtree_build: host allocation failed");
  }
  return ICPNN_OK;
}

}  // namespace icpnn
