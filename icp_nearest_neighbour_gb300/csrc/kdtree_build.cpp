// Host KD-tree build ("Implementing ICP with CUDA-KDTree", sections 2.2, 2.3,
// 4.2, 5.1, 5.2): split on the axis of largest variance (or, as the section
// 4.2 alternative, round robin x, y, z by depth) at the median, stop at
// leaf_size points or at the depth cap.
// The array partitioned is the 16-byte point records themselves (x, y, z,
// original index): every pass over a node reads memory sequentially, and when
// the build ends the array is already the leaf-ordered record array the device
// search reads.
//
// How a node is split.  The median under the (coordinate, index) order is
// unique, so which records end up left of it does not depend on how it is
// found.  A node of kBucketMin records or more finds it with one histogram
// pass (records binned by where their coordinate falls in mean +- one standard
// deviation of the node, which always holds the median; outside values clamp
// to the end bins) and one scatter pass that writes the records below, inside
// and above the median's bin to the node's range of a second buffer; an
// nth_element over that bin alone then places the median.  Smaller nodes use
// nth_element.  One more pass sums the two children's coordinates and squares,
// so a child knows its mean and variance without reading its records again.
//
// Variance: sums of x - c and (x - c)^2 in double about the parent's mean c,
// var = q/n - (s/n)^2.  The page fixes no formula; the rounding differs from
// a two-pass sum by parts in 1e15, far inside the relative 1e-9 within which
// axes count as tied (the lowest tied axis wins).  The root's sums are taken
// about its first point, in the same pass that writes the records.
//
// Each node also gets the tight bounding box of its points (leaves from their
// records, inner nodes as the union of their children's) for the search's
// box test.
//
// Parallelism.  The subtrees of nodes near the root are tasks of the library's
// host pool, and a node of two or more kChunk-record chunks runs its passes
// chunk-parallel, summing per chunk and adding the chunk sums in chunk order.
// The chunking depends on the node's size only, so the tree is the same on
// every machine and thread count.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <new>
#include <thread>
#include <vector>

#include "icpnn_internal.h"

namespace icpnn {
namespace {

struct Rec {
  float c[3];
  int32_t idx;
};
static_assert(sizeof(Rec) == 16, "record must match the device float4 layout");

constexpr int64_t kChunk = 8192;    // records per chunk of a parallel node pass
constexpr int64_t kMaxChunks = 64;
constexpr int64_t kBucketMin = 16;  // smaller nodes use nth_element

int64_t chunks_for(int64_t count) { return std::min<int64_t>(kMaxChunks, count / kChunk); }

// Sums over a set of records of x - c and (x - c)^2 per axis, c a fixed
// centre, and (kRange) the coordinate range per axis.
template <bool kRange>
struct SumsT {
  double n = 0.0;
  double s[3] = {0.0, 0.0, 0.0};
  double q[3] = {0.0, 0.0, 0.0};
  float mn[3] = {INFINITY, INFINITY, INFINITY};
  float mx[3] = {-INFINITY, -INFINITY, -INFINITY};
  void add(const Rec& r, const double c[3]) {
    n += 1.0;
    for (int d = 0; d < 3; ++d) {
      const double x = static_cast<double>(r.c[d]) - c[d];
      s[d] += x;
      q[d] += x * x;
      if (kRange) {
        mn[d] = std::min(mn[d], r.c[d]);
        mx[d] = std::max(mx[d], r.c[d]);
      }
    }
  }
  void add(const SumsT& o) {
    n += o.n;
    for (int d = 0; d < 3; ++d) {
      s[d] += o.s[d];
      q[d] += o.q[d];
      if (kRange) {
        mn[d] = std::min(mn[d], o.mn[d]);
        mx[d] = std::max(mx[d], o.mx[d]);
      }
    }
  }
};
using Sums = SumsT<true>;
using FastSums = SumsT<false>;  // the children's sums, the build's hottest pass

// A node's mean and population variance per axis.  An axis on which all
// coordinates are equal has variance exactly 0 (as a direct two-pass sum of
// float coordinates gives), not the rounding left over by q/n - (s/n)^2.
// `accurate` is false when the subtraction lost too much: the mean of
// (x - c)^2 is more than 16 times the variance, i.e. c lies far from the
// records; the caller then sums again about the mean just found.  Sums
// without the range cannot tell an axis of equal coordinates (unless all
// equal c) from a narrow one: its variance comes out as rounding, is flagged
// as not accurate, and the second sum, which has the range, settles it.
struct Moments {
  double mean[3];
  double var[3];
  bool accurate;
  template <bool kRange>
  static Moments from(const SumsT<kRange>& u, const double c[3]) {
    Moments m;
    m.accurate = true;
    for (int d = 0; d < 3; ++d) {
      const double a = u.s[d] / u.n;
      const double q = u.q[d] / u.n;
      const bool flat = kRange && u.mn[d] == u.mx[d];
      m.mean[d] = c[d] + a;
      m.var[d] = flat ? 0.0 : std::max(0.0, q - a * a);
      if (!flat && !(q <= 16.0 * m.var[d])) m.accurate = false;
    }
    return m;
  }
};

bool rec_less(const Rec& a, const Rec& b, int axis) {
  return a.c[axis] < b.c[axis] || (a.c[axis] == b.c[axis] && a.idx < b.idx);
}

struct Builder {
  int32_t leaf_size = 0;
  int32_t max_depth = 0;
  Rec* buf[2] = {nullptr, nullptr};  // records ([0], the output) and scratch
  Node* heap = nullptr;
  float* box = nullptr;  // 8 floats per heap slot
  int parallel_depth = 0;
  bool round_robin = false;  // axis = depth mod 3 instead of largest variance

  bool is_leaf(int64_t count, int depth) const { return count <= leaf_size || depth >= max_depth; }

  // Axis of largest variance; axes within a relative 1e-9 of the largest are
  // tied and the lowest of them wins.
  static int widest_axis(const Moments& mo) {
    const double vmax = std::max(mo.var[0], std::max(mo.var[1], mo.var[2]));
    for (int d = 0; d < 3; ++d)
      if (mo.var[d] >= vmax * (1.0 - 1e-9)) return d;
    return 0;
  }

  // Splits node [lo, hi) of buf[b] at rank m on `axis`; returns the buffer
  // that now holds the node (records of rank < m first, rank m at lo + m).
  int split(int b, int64_t lo, int64_t hi, int64_t m, int axis, const Moments& mo) {
    const int64_t count = hi - lo;
    Rec* src = buf[b];
    if (count < kBucketMin) {
      std::nth_element(src + lo, src + lo + m, src + hi,
                       [axis](const Rec& x, const Rec& y) { return rec_less(x, y, axis); });
      return b;
    }
    Rec* dst = buf[b ^ 1];
    int nb = 16;
    while (nb < count / 4 && nb < 1024) nb *= 2;
    const double sd = std::sqrt(mo.var[axis]);
    const float base = static_cast<float>(mo.mean[axis] - sd);
    // a spread too small to scale (or none) puts every record in one bin
    const double scale_d = nb / (2.0 * sd);
    const float scale = sd > 0.0 && scale_d < 1e30 ? static_cast<float>(scale_d) : 0.f;
    const float top = static_cast<float>(nb - 1);
    // Monotone in v, since float rounding is monotone and the scale is not
    // negative: a lower bin never holds a larger coordinate.  A difference
    // that overflows clamps to an end bin.
    auto bin = [=](float v) {
      const float x = scale == 0.f ? 0.f : (v - base) * scale;
      return static_cast<int>(std::min(std::max(x, 0.f), top));
    };
    const int64_t C = std::max<int64_t>(1, chunks_for(count));
    auto chunk_lo = [=](int64_t k) { return lo + count * k / C; };
    // per-thread scratch: split never runs twice at once on one thread
    thread_local std::vector<int32_t> hist;
    thread_local std::vector<int64_t> at;
    hist.assign(static_cast<size_t>(C * nb), 0);
    at.resize(static_cast<size_t>(3 * C));
    int32_t* const hp = hist.data();
    int64_t* const ap = at.data();
    // Both passes first compute the bins of a block of records, then update
    // the counters: when many records share a bin (the clamped ends), a
    // counter update per record would wait for the previous one.
    constexpr int kBlock = 64;
    auto histogram = [=](int k) {
      int32_t* h = hp + static_cast<int64_t>(k) * nb;
      const int64_t b1 = chunk_lo(k + 1);
      int32_t bins[kBlock];
      for (int64_t i = chunk_lo(k); i < b1; i += kBlock) {
        const int len = static_cast<int>(std::min<int64_t>(kBlock, b1 - i));
        for (int t = 0; t < len; ++t) bins[t] = bin(src[i + t].c[axis]);
        for (int t = 0; t < len; ++t) ++h[bins[t]];
      }
    };
    if (C > 1) parallel_for(static_cast<int>(C), histogram); else histogram(0);
    // the bin j holding rank m and the records below it
    int64_t n_lt = 0, n_eq = 0;
    int j = 0;
    for (;; ++j) {
      n_eq = 0;
      for (int64_t k = 0; k < C; ++k) n_eq += hp[k * nb + j];
      if (n_lt + n_eq > m || j == nb - 1) break;
      n_lt += n_eq;
    }
    // write offsets per chunk of the three groups, chunks in order
    int64_t o[3] = {lo, lo + n_lt, lo + n_lt + n_eq};
    for (int64_t k = 0; k < C; ++k) {
      const int32_t* h = hp + k * nb;
      int64_t lt = 0;
      for (int i = 0; i < j; ++i) lt += h[i];
      const int64_t eq = h[j];
      ap[3 * k] = o[0];
      ap[3 * k + 1] = o[1];
      ap[3 * k + 2] = o[2];
      o[0] += lt;
      o[1] += eq;
      o[2] += chunk_lo(k + 1) - chunk_lo(k) - lt - eq;
    }
    auto scatter = [=](int k) {
      int64_t w[3] = {ap[3 * k], ap[3 * k + 1], ap[3 * k + 2]};
      const int64_t b1 = chunk_lo(k + 1);
      int32_t grp[kBlock];
      for (int64_t i = chunk_lo(k); i < b1; i += kBlock) {
        const int len = static_cast<int>(std::min<int64_t>(kBlock, b1 - i));
        for (int t = 0; t < len; ++t) {
          const int g = bin(src[i + t].c[axis]);
          grp[t] = (g >= j) + (g > j);
        }
        for (int t = 0; t < len; ++t) dst[w[grp[t]]++] = src[i + t];
      }
    };
    if (C > 1) parallel_for(static_cast<int>(C), scatter); else scatter(0);
    Rec* band = dst + lo + n_lt;
    std::nth_element(band, band + (m - n_lt), band + n_eq,
                     [axis](const Rec& x, const Rec& y) { return rec_less(x, y, axis); });
    return b ^ 1;
  }

  // Sums about c of the records [lo, lo + m) and [lo + m, hi) of buf[b].
  void child_sums(int b, int64_t lo, int64_t hi, int64_t m, const double c[3], FastSums* left, FastSums* right) const {
    const int64_t count = hi - lo;
    const Rec* r = buf[b];
    const int64_t C = std::max<int64_t>(1, chunks_for(count));
    FastSums part_small[2];
    std::vector<FastSums> part_big(C > 1 ? static_cast<size_t>(2 * C) : 0);
    FastSums* part = C > 1 ? part_big.data() : part_small;
    auto body = [=](int k) {
      const int64_t b0 = lo + count * k / C, b1 = lo + count * (k + 1) / C, mid = lo + m;
      FastSums sl, sr;
      for (int64_t i = b0; i < std::min(b1, mid); ++i) sl.add(r[i], c);
      for (int64_t i = std::max(b0, mid); i < b1; ++i) sr.add(r[i], c);
      part[2 * k] = sl;
      part[2 * k + 1] = sr;
    };
    if (C > 1) parallel_for(static_cast<int>(C), body); else body(0);
    for (int64_t k = 0; k < C; ++k) {
      left->add(part[2 * k]);
      right->add(part[2 * k + 1]);
    }
  }

  // Builds the subtree of `node` over [lo, hi) of buf[b]; mo are the node's
  // moments.  Leaves copy their records into buf[0] if they sit in buf[1].
  // Returns the number of nodes in the subtree.  (Not a shared atomic
  // counter: on the 16 Arm cores of a GB300 host, every thread incrementing
  // one cache line per node made the build three times slower.)
  int64_t build(uint64_t node, int b, int64_t lo, int64_t hi, int depth, const Moments& mo) {
    const int64_t count = hi - lo;
    if (is_leaf(count, depth)) {
      if (b == 1) std::memcpy(buf[0] + lo, buf[1] + lo, static_cast<size_t>(count) * sizeof(Rec));
      heap[node].a = static_cast<uint32_t>(lo);
      heap[node].meta = kLeafTag | (static_cast<uint32_t>(count) << 2);
      float* bx = box + 8 * node;
      for (int d = 0; d < 3; ++d) {
        bx[d] = INFINITY;
        bx[4 + d] = -INFINITY;
      }
      for (int64_t i = lo; i < hi; ++i)
        for (int d = 0; d < 3; ++d) {
          bx[d] = std::min(bx[d], buf[0][i].c[d]);
          bx[4 + d] = std::max(bx[4 + d], buf[0][i].c[d]);
        }
      return 1;
    }
    const int axis = round_robin ? depth % 3 : widest_axis(mo);
    const int64_t m = count / 2;
    const int nb = split(b, lo, hi, m, axis, mo);
    const float split_value = buf[nb][lo + m].c[axis];
    uint32_t bits;
    std::memcpy(&bits, &split_value, sizeof(bits));
    heap[node].a = bits;
    heap[node].meta = static_cast<uint32_t>(axis);
    // the children's moments, unless both are leaves (which need none)
    Moments ml{}, mr{};
    if (!is_leaf(count - m, depth + 1)) {
      FastSums sl, sr;
      child_sums(nb, lo, hi, m, mo.mean, &sl, &sr);
      ml = Moments::from(sl, mo.mean);
      mr = Moments::from(sr, mo.mean);
      if (!ml.accurate) ml = moments_about(nb, lo, lo + m, ml.mean);
      if (!mr.accurate) mr = moments_about(nb, lo + m, hi, mr.mean);
    }
    int64_t below[2];
    if (depth < parallel_depth && count >= (1 << 13)) {
      parallel_for(2, [&](int side) {
        if (side == 0) below[0] = build(2 * node, nb, lo, lo + m, depth + 1, ml);
        else below[1] = build(2 * node + 1, nb, lo + m, hi, depth + 1, mr);
      });
    } else {
      below[0] = build(2 * node, nb, lo, lo + m, depth + 1, ml);
      below[1] = build(2 * node + 1, nb, lo + m, hi, depth + 1, mr);
    }
    float* bx = box + 8 * node;
    const float* l = box + 16 * node;
    const float* r = l + 8;
    for (int d = 0; d < 3; ++d) {
      bx[d] = std::min(l[d], r[d]);
      bx[4 + d] = std::max(l[4 + d], r[4 + d]);
    }
    return 1 + below[0] + below[1];
  }

  // Moments of the records [lo, hi) of buf[b] from sums about c.
  Moments moments_about(int b, int64_t lo, int64_t hi, const double c[3]) const {
    const int64_t count = hi - lo;
    const int64_t C = std::max<int64_t>(1, chunks_for(count));
    Sums part_small[1];
    std::vector<Sums> part_big(C > 1 ? static_cast<size_t>(C) : 0);
    Sums* part = C > 1 ? part_big.data() : part_small;
    const Rec* r = buf[b];
    auto body = [=](int k) {
      Sums u;
      const int64_t e = lo + count * (k + 1) / C;
      for (int64_t i = lo + count * k / C; i < e; ++i) u.add(r[i], c);
      part[k] = u;
    };
    if (C > 1) parallel_for(static_cast<int>(C), body); else body(0);
    Sums tot;
    for (int64_t k = 0; k < C; ++k) tot.add(part[k]);
    return Moments::from(tot, c);
  }

};

}  // namespace

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

int build_tree(const float* xyz, int64_t n, int32_t leaf_size, int32_t max_depth, bool round_robin,
               icpnn_tree* t) {
  // One pass, chunked over the pool: finiteness check, records, the root's
  // sums (about the first point) and range, and the zeroing of the node and
  // box arrays.  Chunk sums are added in chunk order.
  const int64_t C = std::max<int64_t>(1, std::min<int64_t>(kMaxChunks, n / kChunk));
  if (C > 1) pool_wake();  // the workers come up while the arrays are allocated
  try {
    std::vector<int64_t> first_bad(static_cast<size_t>(C), -1);
    std::vector<Sums> part(static_cast<size_t>(C));
    const int32_t depth = tree_depth(n, leaf_size, max_depth);
    const int64_t largest_leaf = (n + (int64_t{1} << depth) - 1) >> depth;
    if (largest_leaf >= (int64_t{1} << 30))
      return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build: a leaf would hold 2^30 points or more");
    const int64_t slots = int64_t{1} << (depth + 1);
    t->records.resize(static_cast<size_t>(4 * n));
    t->nodes.resize(static_cast<size_t>(slots));
    t->boxes.resize(static_cast<size_t>(8 * slots));
    Rec* recs = reinterpret_cast<Rec*>(t->records.data());
    const double c0[3] = {xyz[0], xyz[1], xyz[2]};
    parallel_for(static_cast<int>(C), [&](int c) {
      const int64_t s0 = slots * c / C, s1 = slots * (c + 1) / C;
      std::memset(t->nodes.data() + s0, 0, static_cast<size_t>(s1 - s0) * sizeof(Node));
      std::memset(t->boxes.data() + 8 * s0, 0, static_cast<size_t>(s1 - s0) * 8 * sizeof(float));
      Sums u;
      for (int64_t i = n * c / C; i < n * (c + 1) / C; ++i) {
        Rec r;
        for (int d = 0; d < 3; ++d) {
          r.c[d] = xyz[3 * i + d];
          if (!std::isfinite(r.c[d])) {
            first_bad[static_cast<size_t>(c)] = i;
            return;
          }
        }
        r.idx = static_cast<int32_t>(i);
        recs[i] = r;
        u.add(r, c0);
      }
      part[static_cast<size_t>(c)] = u;
    });
    for (int64_t c = 0; c < C; ++c)
      if (first_bad[static_cast<size_t>(c)] >= 0)
        return fail(ICPNN_ERR_NONFINITE, "kdtree_build: non-finite coordinate at point " +
                                             std::to_string(first_bad[static_cast<size_t>(c)]));
    Sums root;
    for (int64_t c = 0; c < C; ++c) root.add(part[static_cast<size_t>(c)]);
    for (int d = 0; d < 3; ++d) {
      t->bbox_lo[d] = root.mn[d];
      t->bbox_hi[d] = root.mx[d];
    }
    t->n = n;
    t->leaf_size = leaf_size;
    t->max_depth = max_depth;
    t->round_robin = round_robin;
    t->depth = depth;
    t->heap_slots = slots;

    std::unique_ptr<Rec[]> temp(new Rec[static_cast<size_t>(n)]);
    Builder b;
    b.leaf_size = leaf_size;
    b.max_depth = max_depth;
    b.buf[0] = recs;
    b.buf[1] = temp.get();
    b.heap = t->nodes.data();
    b.box = t->boxes.data();
    b.round_robin = round_robin;
    const unsigned hw = std::max(1u, std::thread::hardware_concurrency());
    int pd = 0;
    while ((1u << pd) < 4 * hw && pd < 8) ++pd;
    b.parallel_depth = pd;
    Moments mo = Moments::from(root, c0);
    if (!mo.accurate) mo = b.moments_about(0, 0, n, mo.mean);
    t->n_nodes = b.build(1, 0, 0, n, 0, mo);
  } catch (const std::bad_alloc&) {
    return fail(ICPNN_ERR_NO_MEMORY, "kdtree_build: host allocation failed");
  }
  return ICPNN_OK;
}

}  // namespace icpnn
