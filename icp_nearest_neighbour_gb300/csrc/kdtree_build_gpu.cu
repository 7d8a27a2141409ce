// Device KD-tree build: the same tree as the host build ("Implementing ICP
// with CUDA-KDTree", sections 2.2, 2.3, 4.2, 5.1, 5.2 -- axis of largest
// variance or round robin, median split by (coordinate, index), leaves of at
// most leaf_size points or at the depth cap), made on the GPU from points
// already in device memory, for pipelines where the host build would be the
// longest step.
//
// Method.  The points are sorted once per axis by (coordinate, index): three
// lists of point ids.  Throughout, the points of every node sit in one range
// [lo, lo + count) of each list, sorted there by that list's axis, and the
// ranges follow from n alone (a node of c points has a left child of c/2).
// Then level by level, for all nodes of the level at once:
//   1. sums of x, y, z and the bounding box, per node (blocks over chunks of
//      the node, partial sums added in chunk order);
//   2. the mean, then the sums of squared deviations about it (the population
//      variance in two passes, as the definition reads);
//   3. the split axis (largest variance, ties within a relative 1e-9 to the
//      lowest axis) and the median: the point at position lo + count/2 of the
//      axis's list -- the list is sorted by (coordinate, index), so no
//      selection is needed;
//   4. each point learns its side from its position in the chosen axis's list;
//      the other two lists are partitioned stably within the node, which keeps
//      them sorted (the chosen list already is: left half, then right half).
// Leaves take their points from the lists when they are reached.  Every sum
// runs in a fixed order, and ties in the variance are resolved by the same
// band as on the host, so the tree is the host tree node for node; only the
// order of points inside a leaf may differ.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "icpnn_internal.h"
#include "kernels.cuh"

namespace icpnn {

extern std::atomic<int64_t> g_launch_count;

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kBT = 256;          // threads per block of the level kernels
constexpr int kChunk = 2048;      // list positions per block of a node
constexpr int kBWarps = kBT / 32;
constexpr int kWarpNode = 256;    // levels whose nodes hold at most this many points: one warp per node
constexpr int kBlockNode = 4096;  // ... at most this many (and more than kWarpNode): one block per node

// Range of heap node k at depth d under the median rule; false when the node
// does not exist (an ancestor is a leaf).
__host__ __device__ inline bool node_range(uint32_t k, int d, int64_t n, int32_t leaf, int32_t max_depth,
                                           int64_t* lo, int64_t* cnt) {
  int64_t l = 0, c = n;
  for (int lvl = 0; lvl < d; ++lvl) {
    if (c <= leaf || lvl >= max_depth) return false;
    const int64_t m = c / 2;
    if ((k >> (d - 1 - lvl)) & 1u) {
      l += m;
      c -= m;
    } else {
      c = m;
    }
  }
  *lo = l;
  *cnt = c;
  return true;
}

struct LevelArgs {
  int d;                 // depth of the level
  int blocks_per_node;   // B: blocks (chunks) per node
  int64_t n;
  int32_t leaf;
  int32_t max_depth;
  bool round_robin;
};

__host__ __device__ inline bool is_leaf_node(int64_t cnt, int d, const LevelArgs& a) {
  return cnt <= a.leaf || d >= a.max_depth;
}

// Orderable bits of a float: the unsigned order of the result is the numeric
// order, with -0 mapped onto +0 (they compare equal).
__device__ __forceinline__ uint32_t orderable(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float coord(const float4& r, int axis) { return axis == 0 ? r.x : (axis == 1 ? r.y : r.z); }
__device__ __forceinline__ uint32_t rec_id(const float4& r) { return static_cast<uint32_t>(__float_as_int(r.w)); }

__global__ void __launch_bounds__(256) build_records_kernel(const float* __restrict__ xyz, int64_t n,
                                                            float4* __restrict__ P, uint32_t* __restrict__ keys,
                                                            uint32_t* __restrict__ ids,
                                                            unsigned long long* __restrict__ first_bad) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float x = xyz[3 * i], y = xyz[3 * i + 1], z = xyz[3 * i + 2];
    if (!(isfinite(x) && isfinite(y) && isfinite(z))) atomicMin(first_bad, static_cast<unsigned long long>(i));
    P[i] = make_float4(x, y, z, __int_as_float(static_cast<int32_t>(i)));
    keys[i] = orderable(x);
    keys[n + i] = orderable(y);
    keys[2 * n + i] = orderable(z);
    ids[i] = ids[n + i] = ids[2 * n + i] = static_cast<uint32_t>(i);
  }
}

// List l = the records in the order of the sorted ids of axis l.
__global__ void __launch_bounds__(256) gather_lists_kernel(const float4* __restrict__ P, int64_t n,
                                                           const uint32_t* __restrict__ ids,
                                                           float4* __restrict__ L) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < 3 * n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    L[i] = __ldg(&P[ids[i]]);
}

// Fixed-order reductions: butterfly in the warp (every lane gets the result);
// blocks then add the warps' results in warp order.
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
  return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, off));
  return v;
}
// The block's node and chunk; false (block-uniform) when there is none.
__device__ __forceinline__ bool block_chunk(const LevelArgs& a, uint32_t* k, int64_t* lo, int64_t* cnt,
                                            int64_t* b0, int64_t* b1, int* j) {
  *k = (1u << a.d) + static_cast<uint32_t>(blockIdx.x / a.blocks_per_node);
  *j = static_cast<int>(blockIdx.x % a.blocks_per_node);
  if (!node_range(*k, a.d, a.n, a.leaf, a.max_depth, lo, cnt)) return false;
  *b0 = *lo + static_cast<int64_t>(*j) * kChunk;
  *b1 = min(*lo + *cnt, *b0 + static_cast<int64_t>(kChunk));
  return true;
}

// ------------------------------------------------ levels of large nodes --
//
// Each pass over a level runs one block per (node, chunk); the last block of
// a node to finish (a per-node counter, reset by that block) combines the
// node's chunk partials in chunk order.

// True in every thread of the block that finishes the node's pass last.
__device__ __forceinline__ bool last_of_node(unsigned int* counter, int chunks, bool* s_last) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    *s_last = atomicAdd(counter, 1u) == static_cast<unsigned int>(chunks - 1);
    if (*s_last) *counter = 0u;
  }
  __syncthreads();
  if (*s_last) __threadfence();
  return *s_last;
}

// Per node, one warp: the chunk partials added in a fixed order (lanes over
// chunks, then a butterfly); the mean and the box, and for a leaf its node
// record.
__device__ __forceinline__ void node_mean(const LevelArgs& a, uint32_t k, int64_t slot, int64_t lo, int64_t cnt,
                                          int chunks, const double* __restrict__ part, double* __restrict__ mean,
                                          Node* __restrict__ nodes, float4* __restrict__ boxes) {
  const int lane = threadIdx.x & 31;
  double s[3] = {0.0, 0.0, 0.0}, nmn[3] = {-INFINITY, -INFINITY, -INFINITY}, mx[3] = {-INFINITY, -INFINITY, -INFINITY};
  for (int j = lane; j < chunks; j += 32) {
    const double* p = part + (slot * a.blocks_per_node + j) * 9;
#pragma unroll
    for (int e = 0; e < 3; ++e) {
      s[e] += __ldcg(&p[e]);
      nmn[e] = fmax(nmn[e], __ldcg(&p[3 + e]));
      mx[e] = fmax(mx[e], __ldcg(&p[6 + e]));
    }
  }
#pragma unroll
  for (int e = 0; e < 3; ++e) {
    s[e] = warp_sum(s[e]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      nmn[e] = fmax(nmn[e], __shfl_xor_sync(kFull, nmn[e], off));
      mx[e] = fmax(mx[e], __shfl_xor_sync(kFull, mx[e], off));
    }
  }
  if (lane == 0) {
    boxes[2 * k] = make_float4(static_cast<float>(-nmn[0]), static_cast<float>(-nmn[1]),
                               static_cast<float>(-nmn[2]), 0.f);
    boxes[2 * k + 1] = make_float4(static_cast<float>(mx[0]), static_cast<float>(mx[1]), static_cast<float>(mx[2]), 0.f);
    const double c = static_cast<double>(cnt);
    for (int e = 0; e < 3; ++e) mean[slot * 3 + e] = s[e] / c;
    if (is_leaf_node(cnt, a.d, a)) {
      nodes[k].a = static_cast<uint32_t>(lo);
      nodes[k].meta = kLeafTag | (static_cast<uint32_t>(cnt) << 2);
    }
  }
}


// Pass 1 over each chunk of list 0: coordinate sums and box.  part[block] =
// {sx, sy, sz, -minx, -miny, -minz, maxx, maxy, maxz}.
__global__ void __launch_bounds__(kBT) level_sums_kernel(LevelArgs a, const float4* __restrict__ L0,
                                                         double* __restrict__ part, unsigned int* __restrict__ counter,
                                                         double* __restrict__ mean, Node* __restrict__ nodes,
                                                         float4* __restrict__ boxes) {
  __shared__ bool s_last;
  uint32_t k;
  int64_t lo, cnt, b0, b1;
  int j;
  if (!block_chunk(a, &k, &lo, &cnt, &b0, &b1, &j) || b0 >= b1) return;
  double s[3] = {0.0, 0.0, 0.0};
  float mn[3] = {INFINITY, INFINITY, INFINITY}, mx[3] = {-INFINITY, -INFINITY, -INFINITY};
#pragma unroll 4
  for (int64_t i = b0 + threadIdx.x; i < b1; i += kBT) {
    const float4 p = L0[i];
    const float c[3] = {p.x, p.y, p.z};
#pragma unroll
    for (int e = 0; e < 3; ++e) {
      s[e] += static_cast<double>(c[e]);
      mn[e] = fminf(mn[e], c[e]);
      mx[e] = fmaxf(mx[e], c[e]);
    }
  }
  // all nine values in one round: butterfly in each warp, then the warps in
  // order (a fixed association)
  double r[9];
#pragma unroll
  for (int e = 0; e < 3; ++e) {
    r[e] = warp_sum(s[e]);
    r[3 + e] = static_cast<double>(-warp_min(mn[e]));
    r[6 + e] = static_cast<double>(-warp_min(-mx[e]));
  }
  __shared__ double sh9[kBWarps][9];
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int e = 0; e < 9; ++e) sh9[threadIdx.x >> 5][e] = r[e];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int e = 0; e < 9; ++e) {
      double v = sh9[0][e];
      for (int w = 1; w < kBWarps; ++w) v = e < 3 ? v + sh9[w][e] : fmax(v, sh9[w][e]);
      part[static_cast<int64_t>(blockIdx.x) * 9 + e] = v;
    }
  }
  const int64_t slot = k - (1u << a.d);
  const int chunks = static_cast<int>((cnt + kChunk - 1) / kChunk);
  if (!last_of_node(&counter[slot], chunks, &s_last) || threadIdx.x >= 32) return;
  node_mean(a, k, slot, lo, cnt, chunks, part, mean, nodes, boxes);
}

// Axis by the largest variance, ties within a relative 1e-9 to the lowest.
__device__ __forceinline__ int widest(double v0, double v1, double v2) {
  const double vmax = fmax(v0, fmax(v1, v2));
  const double lim = vmax * (1.0 - 1e-9);
  return v0 >= lim ? 0 : (v1 >= lim ? 1 : 2);
}

// Per inner node, one warp: the variance, the split axis, the median (the
// record at position lo + count/2 of the axis's list) and the node record.
__device__ __forceinline__ void node_split(const LevelArgs& a, uint32_t k, int64_t slot, int64_t lo, int64_t cnt,
                                           int chunks, const double* __restrict__ part,
                                           const float4* __restrict__ L0, const float4* __restrict__ L1,
                                           const float4* __restrict__ L2, Node* __restrict__ nodes) {
  const int lane = threadIdx.x & 31;
  double q[3] = {0.0, 0.0, 0.0};
  for (int j = lane; j < chunks; j += 32) {
    const double* p = part + (slot * a.blocks_per_node + j) * 9;
#pragma unroll
    for (int e = 0; e < 3; ++e) q[e] += __ldcg(&p[e]);
  }
#pragma unroll
  for (int e = 0; e < 3; ++e) q[e] = warp_sum(q[e]);
  if (lane != 0) return;
  const double c = static_cast<double>(cnt);
  const int axis = a.round_robin ? a.d % 3 : widest(q[0] / c, q[1] / c, q[2] / c);
  const float4* L = axis == 0 ? L0 : (axis == 1 ? L1 : L2);
  nodes[k].a = __float_as_uint(coord(L[lo + cnt / 2], axis));
  nodes[k].meta = static_cast<uint32_t>(axis);
}

// Pass 2: sums of squared deviations about the node's mean (inner nodes).
__global__ void __launch_bounds__(kBT) level_sq_kernel(LevelArgs a, const float4* __restrict__ L0,
                                                       const float4* __restrict__ L1,
                                                       const float4* __restrict__ L2,
                                                       const double* __restrict__ mean,
                                                       double* __restrict__ part, unsigned int* __restrict__ counter,
                                                       Node* __restrict__ nodes) {
  __shared__ bool s_last;
  uint32_t k;
  int64_t lo, cnt, b0, b1;
  int j;
  if (!block_chunk(a, &k, &lo, &cnt, &b0, &b1, &j) || b0 >= b1 || is_leaf_node(cnt, a.d, a)) return;
  const int64_t slot = k - (1u << a.d);
  const double m0 = mean[slot * 3], m1 = mean[slot * 3 + 1], m2 = mean[slot * 3 + 2];
  double q0 = 0.0, q1 = 0.0, q2 = 0.0;
#pragma unroll 4
  for (int64_t i = b0 + threadIdx.x; i < b1; i += kBT) {
    const float4 p = L0[i];
    const double e0 = static_cast<double>(p.x) - m0;
    const double e1 = static_cast<double>(p.y) - m1;
    const double e2 = static_cast<double>(p.z) - m2;
    q0 += e0 * e0;
    q1 += e1 * e1;
    q2 += e2 * e2;
  }
  q0 = warp_sum(q0);
  q1 = warp_sum(q1);
  q2 = warp_sum(q2);
  __shared__ double sh3[kBWarps][3];
  if ((threadIdx.x & 31) == 0) {
    sh3[threadIdx.x >> 5][0] = q0;
    sh3[threadIdx.x >> 5][1] = q1;
    sh3[threadIdx.x >> 5][2] = q2;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int e = 0; e < 3; ++e) {
      double v = 0.0;
      for (int w = 0; w < kBWarps; ++w) v += sh3[w][e];
      part[static_cast<int64_t>(blockIdx.x) * 9 + e] = v;
    }
  }
  const int chunks = static_cast<int>((cnt + kChunk - 1) / kChunk);
  if (!last_of_node(&counter[slot], chunks, &s_last) || threadIdx.x >= 32) return;
  node_split(a, k, slot, lo, cnt, chunks, part, L0, L1, L2, nodes);
}


// Inner nodes: each point's side from its position in the chosen axis's list
// (1 = left).  Leaves: their records, in the order of list 0.
__global__ void __launch_bounds__(kBT) level_flag_kernel(LevelArgs a, const float4* __restrict__ L0,
                                                         const float4* __restrict__ L1,
                                                         const float4* __restrict__ L2,
                                                         const Node* __restrict__ nodes,
                                                         uint8_t* __restrict__ left,
                                                         float4* __restrict__ records) {
  uint32_t k;
  int64_t lo, cnt, b0, b1;
  int j;
  if (!block_chunk(a, &k, &lo, &cnt, &b0, &b1, &j)) return;
  if (is_leaf_node(cnt, a.d, a)) {
    for (int64_t i = b0 + threadIdx.x; i < b1; i += kBT) records[i] = L0[i];
    return;
  }
  const uint32_t axis = nodes[k].meta;
  const float4* L = axis == 0 ? L0 : (axis == 1 ? L1 : L2);
  const int64_t mid = lo + cnt / 2;
#pragma unroll 4
  for (int64_t i = b0 + threadIdx.x; i < b1; i += kBT) left[rec_id(L[i])] = i < mid ? 1 : 0;
}

// Left points per chunk of each list (inner nodes): cntl[block * 3 + list].
__global__ void __launch_bounds__(kBT) level_count_kernel(LevelArgs a, const float4* __restrict__ L0,
                                                          const float4* __restrict__ L1,
                                                          const float4* __restrict__ L2,
                                                          const uint8_t* __restrict__ left,
                                                          uint32_t* __restrict__ cntl,
                                                          unsigned int* __restrict__ counter) {
  __shared__ uint32_t sh[3][kBWarps];
  __shared__ bool s_last;
  uint32_t k;
  int64_t lo, cnt, b0, b1;
  int j;
  if (!block_chunk(a, &k, &lo, &cnt, &b0, &b1, &j) || b0 >= b1 || is_leaf_node(cnt, a.d, a)) return;
  uint32_t c0 = 0, c1 = 0, c2 = 0;
#pragma unroll 4
  for (int64_t i = b0 + threadIdx.x; i < b1; i += kBT) {
    c0 += left[rec_id(L0[i])];
    c1 += left[rec_id(L1[i])];
    c2 += left[rec_id(L2[i])];
  }
  c0 = __reduce_add_sync(kFull, c0);
  c1 = __reduce_add_sync(kFull, c1);
  c2 = __reduce_add_sync(kFull, c2);
  if ((threadIdx.x & 31) == 0) {
    sh[0][threadIdx.x >> 5] = c0;
    sh[1][threadIdx.x >> 5] = c1;
    sh[2][threadIdx.x >> 5] = c2;
  }
  __syncthreads();
  if (threadIdx.x < 3) {
    uint32_t t = 0;
    for (int w = 0; w < kBWarps; ++w) t += sh[threadIdx.x][w];
    cntl[static_cast<int64_t>(blockIdx.x) * 3 + threadIdx.x] = t;
  }
  // the node's last block: exclusive prefix of the chunks' counts, in chunk
  // order, per list (in place)
  const int64_t slot = k - (1u << a.d);
  const int chunks = static_cast<int>((cnt + kChunk - 1) / kChunk);
  if (!last_of_node(&counter[slot], chunks, &s_last) || threadIdx.x >= 3) return;
  uint32_t run = 0;
  for (int c = 0; c < chunks; ++c) {
    uint32_t* p = cntl + (slot * a.blocks_per_node + c) * 3 + threadIdx.x;
    const uint32_t v = __ldcg(p);
    *p = run;
    run += v;
  }
}

// Stable partition of each list within every inner node: left points first,
// then right ones, both in list order.  Out of place into T0..T2.
__global__ void __launch_bounds__(kBT) level_scatter_kernel(LevelArgs a, const float4* __restrict__ L0,
                                                            const float4* __restrict__ L1,
                                                            const float4* __restrict__ L2,
                                                            float4* __restrict__ T0, float4* __restrict__ T1,
                                                            float4* __restrict__ T2,
                                                            const uint8_t* __restrict__ left,
                                                            const uint32_t* __restrict__ cntl) {
  __shared__ uint32_t sh[3][kBWarps];
  uint32_t k;
  int64_t lo, cnt, b0, b1;
  int j;
  if (!block_chunk(a, &k, &lo, &cnt, &b0, &b1, &j) || is_leaf_node(cnt, a.d, a)) return;
  const float4* Ls[3] = {L0, L1, L2};
  float4* Ts[3] = {T0, T1, T2};
  const int64_t mid = lo + cnt / 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t nl[3], nr[3];
#pragma unroll
  for (int l = 0; l < 3; ++l) {
    const uint32_t before = cntl[static_cast<int64_t>(blockIdx.x) * 3 + l];
    nl[l] = before;
    nr[l] = (b0 - lo) - static_cast<int64_t>(before);
  }
  for (int64_t base = b0; base < b1; base += kBT) {
    const int64_t i = base + threadIdx.x;
    const bool valid = i < b1;
    float4 r[3];
    uint32_t f[3], bal[3];
#pragma unroll
    for (int l = 0; l < 3; ++l) r[l] = valid ? Ls[l][i] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int l = 0; l < 3; ++l) {
      f[l] = valid ? left[rec_id(r[l])] : 0u;
      bal[l] = __ballot_sync(kFull, f[l] != 0u);
    }
    __syncthreads();
    if (lane == 0) {
#pragma unroll
      for (int l = 0; l < 3; ++l) sh[l][warp] = __popc(bal[l]);
    }
    __syncthreads();
    const int64_t round_n = min(static_cast<int64_t>(kBT), b1 - base);
#pragma unroll
    for (int l = 0; l < 3; ++l) {
      uint32_t before = 0, round_left = 0;
#pragma unroll
      for (int w = 0; w < kBWarps; ++w) {
        if (w < warp) before += sh[l][w];
        round_left += sh[l][w];
      }
      if (valid) {
        const int64_t rl = before + __popc(bal[l] & ((1u << lane) - 1u));
        const int64_t rr = (i - base) - rl;
        Ts[l][f[l] ? lo + nl[l] + rl : mid + nr[l] + rr] = r[l];
      }
      nl[l] += round_left;
      nr[l] += round_n - round_left;
    }
  }
}

// ------------------------------------------------ levels of small nodes --

// One warp per node of a level whose nodes hold at most kWarpNode points:
// sums, box, variance, split, sides and the stable partition of the three
// lists, all within the warp.
__global__ void __launch_bounds__(256) level_warp_kernel(LevelArgs a, const float4* __restrict__ L0,
                                                         const float4* __restrict__ L1,
                                                         const float4* __restrict__ L2,
                                                         float4* __restrict__ T0, float4* __restrict__ T1,
                                                         float4* __restrict__ T2, uint8_t* __restrict__ left,
                                                         Node* __restrict__ nodes, float4* __restrict__ boxes,
                                                         float4* __restrict__ records) {
  const int64_t slot = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (slot >= (int64_t{1} << a.d)) return;
  const uint32_t k = (1u << a.d) + static_cast<uint32_t>(slot);
  int64_t lo, cnt;
  if (!node_range(k, a.d, a.n, a.leaf, a.max_depth, &lo, &cnt)) return;
  const int64_t hi = lo + cnt;
  double s0 = 0.0, s1 = 0.0, s2 = 0.0;
  float mn0 = INFINITY, mn1 = INFINITY, mn2 = INFINITY, mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY;
  for (int64_t i = lo + lane; i < hi; i += 32) {
    const float4 p = L0[i];
    s0 += static_cast<double>(p.x);
    s1 += static_cast<double>(p.y);
    s2 += static_cast<double>(p.z);
    mn0 = fminf(mn0, p.x);
    mn1 = fminf(mn1, p.y);
    mn2 = fminf(mn2, p.z);
    mx0 = fmaxf(mx0, p.x);
    mx1 = fmaxf(mx1, p.y);
    mx2 = fmaxf(mx2, p.z);
  }
  s0 = warp_sum(s0);
  s1 = warp_sum(s1);
  s2 = warp_sum(s2);
  mn0 = warp_min(mn0);
  mn1 = warp_min(mn1);
  mn2 = warp_min(mn2);
  mx0 = -warp_min(-mx0);
  mx1 = -warp_min(-mx1);
  mx2 = -warp_min(-mx2);
  if (lane == 0) {
    boxes[2 * k] = make_float4(mn0, mn1, mn2, 0.f);
    boxes[2 * k + 1] = make_float4(mx0, mx1, mx2, 0.f);
  }
  if (is_leaf_node(cnt, a.d, a)) {
    for (int64_t i = lo + lane; i < hi; i += 32) records[i] = L0[i];
    if (lane == 0) {
      nodes[k].a = static_cast<uint32_t>(lo);
      nodes[k].meta = kLeafTag | (static_cast<uint32_t>(cnt) << 2);
    }
    return;
  }
  const double c = static_cast<double>(cnt);
  int axis;
  if (a.round_robin) {
    axis = a.d % 3;
  } else {
    const double m0 = s0 / c, m1 = s1 / c, m2 = s2 / c;
    double q0 = 0.0, q1 = 0.0, q2 = 0.0;
    for (int64_t i = lo + lane; i < hi; i += 32) {
      const float4 p = L0[i];
      const double e0 = static_cast<double>(p.x) - m0;
      const double e1 = static_cast<double>(p.y) - m1;
      const double e2 = static_cast<double>(p.z) - m2;
      q0 += e0 * e0;
      q1 += e1 * e1;
      q2 += e2 * e2;
    }
    axis = widest(warp_sum(q0) / c, warp_sum(q1) / c, warp_sum(q2) / c);
  }
  const float4* L = axis == 0 ? L0 : (axis == 1 ? L1 : L2);
  const int64_t mid = lo + cnt / 2;
  if (lane == 0) {
    nodes[k].a = __float_as_uint(coord(L[mid], axis));
    nodes[k].meta = static_cast<uint32_t>(axis);
  }
  for (int64_t i = lo + lane; i < hi; i += 32) left[rec_id(L[i])] = i < mid ? 1 : 0;
  __syncwarp();
  // the three lists in the same rounds: their loads are in flight together
  const float4* Ls[3] = {L0, L1, L2};
  float4* Ts[3] = {T0, T1, T2};
  int64_t nl[3] = {0, 0, 0}, nr[3] = {0, 0, 0};
  for (int64_t base = lo; base < hi; base += 32) {
    const int64_t i = base + lane;
    const bool valid = i < hi;
    const int64_t round_n = min(static_cast<int64_t>(32), hi - base);
    float4 r[3];
#pragma unroll
    for (int l = 0; l < 3; ++l) r[l] = valid ? Ls[l][i] : make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t f[3];
#pragma unroll
    for (int l = 0; l < 3; ++l) f[l] = valid ? left[rec_id(r[l])] : 0u;
#pragma unroll
    for (int l = 0; l < 3; ++l) {
      const uint32_t bal = __ballot_sync(kFull, f[l] != 0u);
      if (valid) {
        const int64_t rl = __popc(bal & ((1u << lane) - 1u));
        Ts[l][f[l] ? lo + nl[l] + rl : mid + nr[l] + (i - base - rl)] = r[l];
      }
      nl[l] += __popc(bal);
      nr[l] += round_n - __popc(bal);
    }
  }
}

// ----------------------------------------------- levels of medium nodes --

// One block per node of a level whose nodes hold at most kBlockNode points:
// the steps of the multi-block passes, with block barriers in place of
// kernel boundaries and block reductions (warp butterflies, then the warps
// in order) in place of the chunk partials.
__global__ void __launch_bounds__(kBT) level_block_kernel(LevelArgs a, const float4* __restrict__ L0,
                                                          const float4* __restrict__ L1,
                                                          const float4* __restrict__ L2,
                                                          float4* __restrict__ T0, float4* __restrict__ T1,
                                                          float4* __restrict__ T2, uint8_t* __restrict__ left,
                                                          Node* __restrict__ nodes, float4* __restrict__ boxes,
                                                          float4* __restrict__ records) {
  __shared__ double sh[kBWarps][9];
  __shared__ double s_tot[9];
  __shared__ uint32_t s_cnt[3][kBWarps];
  const uint32_t k = (1u << a.d) + blockIdx.x;
  int64_t lo, cnt;
  if (!node_range(k, a.d, a.n, a.leaf, a.max_depth, &lo, &cnt)) return;
  const int64_t hi = lo + cnt;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // sums and box; the minima are kept negated so that one max combines both
  {
    double v[9] = {0.0, 0.0, 0.0, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY, -INFINITY};
    for (int64_t i = lo + threadIdx.x; i < hi; i += kBT) {
      const float4 p = L0[i];
      const float c3[3] = {p.x, p.y, p.z};
#pragma unroll
      for (int e = 0; e < 3; ++e) {
        v[e] += static_cast<double>(c3[e]);
        v[3 + e] = fmax(v[3 + e], -static_cast<double>(c3[e]));
        v[6 + e] = fmax(v[6 + e], static_cast<double>(c3[e]));
      }
    }
#pragma unroll
    for (int e = 0; e < 9; ++e) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const double o = __shfl_xor_sync(kFull, v[e], off);
        v[e] = e < 3 ? v[e] + o : fmax(v[e], o);
      }
      if (lane == 0) sh[warp][e] = v[e];
    }
  }
  __syncthreads();
  if (threadIdx.x < 9) {
    const int e = threadIdx.x;
    double t = sh[0][e];
    for (int w = 1; w < kBWarps; ++w) t = e < 3 ? t + sh[w][e] : fmax(t, sh[w][e]);
    s_tot[e] = t;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    boxes[2 * k] = make_float4(static_cast<float>(-s_tot[3]), static_cast<float>(-s_tot[4]),
                               static_cast<float>(-s_tot[5]), 0.f);
    boxes[2 * k + 1] = make_float4(static_cast<float>(s_tot[6]), static_cast<float>(s_tot[7]),
                                   static_cast<float>(s_tot[8]), 0.f);
  }
  if (is_leaf_node(cnt, a.d, a)) {
    for (int64_t i = lo + threadIdx.x; i < hi; i += kBT) records[i] = L0[i];
    if (threadIdx.x == 0) {
      nodes[k].a = static_cast<uint32_t>(lo);
      nodes[k].meta = kLeafTag | (static_cast<uint32_t>(cnt) << 2);
    }
    return;
  }
  const double c = static_cast<double>(cnt);
  int axis;
  if (a.round_robin) {
    axis = a.d % 3;
  } else {
    const double m0 = s_tot[0] / c, m1 = s_tot[1] / c, m2 = s_tot[2] / c;
    double q[3] = {0.0, 0.0, 0.0};
    for (int64_t i = lo + threadIdx.x; i < hi; i += kBT) {
      const float4 p = L0[i];
      const double e0 = static_cast<double>(p.x) - m0;
      const double e1 = static_cast<double>(p.y) - m1;
      const double e2 = static_cast<double>(p.z) - m2;
      q[0] += e0 * e0;
      q[1] += e1 * e1;
      q[2] += e2 * e2;
    }
    __syncthreads();  // s_tot and sh are reused below
#pragma unroll
    for (int e = 0; e < 3; ++e) {
      q[e] = warp_sum(q[e]);
      if (lane == 0) sh[warp][e] = q[e];
    }
    __syncthreads();
    if (threadIdx.x < 3) {
      double t = sh[0][threadIdx.x];
      for (int w = 1; w < kBWarps; ++w) t += sh[w][threadIdx.x];
      s_tot[threadIdx.x] = t / c;
    }
    __syncthreads();
    axis = widest(s_tot[0], s_tot[1], s_tot[2]);
  }
  const float4* L = axis == 0 ? L0 : (axis == 1 ? L1 : L2);
  const int64_t mid = lo + cnt / 2;
  if (threadIdx.x == 0) {
    nodes[k].a = __float_as_uint(coord(L[mid], axis));
    nodes[k].meta = static_cast<uint32_t>(axis);
  }
  for (int64_t i = lo + threadIdx.x; i < hi; i += kBT) left[rec_id(L[i])] = i < mid ? 1 : 0;
  __syncthreads();
  // stable partition of the three lists, kBT positions per round
  const float4* Ls[3] = {L0, L1, L2};
  float4* Ts[3] = {T0, T1, T2};
  int64_t nl[3] = {0, 0, 0}, nr[3] = {0, 0, 0};
  for (int64_t base = lo; base < hi; base += kBT) {
    const int64_t i = base + threadIdx.x;
    const bool valid = i < hi;
    const int64_t round_n = min(static_cast<int64_t>(kBT), hi - base);
    float4 r[3];
    uint32_t f[3], bal[3];
#pragma unroll
    for (int l = 0; l < 3; ++l) r[l] = valid ? Ls[l][i] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int l = 0; l < 3; ++l) {
      f[l] = valid ? left[rec_id(r[l])] : 0u;
      bal[l] = __ballot_sync(kFull, f[l] != 0u);
      if (lane == 0) s_cnt[l][warp] = __popc(bal[l]);
    }
    __syncthreads();
#pragma unroll
    for (int l = 0; l < 3; ++l) {
      uint32_t before = 0, round_left = 0;
#pragma unroll
      for (int w = 0; w < kBWarps; ++w) {
        if (w < warp) before += s_cnt[l][w];
        round_left += s_cnt[l][w];
      }
      if (valid) {
        const int64_t rl = before + __popc(bal[l] & ((1u << lane) - 1u));
        const int64_t rr = (i - base) - rl;
        Ts[l][f[l] ? lo + nl[l] + rl : mid + nr[l] + rr] = r[l];
      }
      nl[l] += round_left;
      nr[l] += round_n - round_left;
    }
    __syncthreads();  // s_cnt is rewritten by the next round
  }
}

inline int grid_for(int64_t items) { return static_cast<int>(std::max<int64_t>(1, (items + 255) / 256)); }

struct DeviceMem {
  std::vector<void*> ptrs;
  cudaStream_t s;
  explicit DeviceMem(cudaStream_t st) : s(st) {}
  ~DeviceMem() {
    for (void* p : ptrs) cudaFreeAsync(p, s);
  }
  template <typename T>
  cudaError_t alloc(T** out, int64_t count) {
    void* p = nullptr;
    const cudaError_t e = pool_alloc(&p, static_cast<size_t>(std::max<int64_t>(count, 1)) * sizeof(T), s);
    if (e != cudaSuccess) return e;
    ptrs.push_back(p);
    *out = static_cast<T*>(p);
    return cudaSuccess;
  }
};

}  // namespace

int build_tree_device(const float* xyz_dev, int64_t n, int32_t leaf_size, int32_t max_depth, bool round_robin,
                      icpnn_tree* t, cudaStream_t s) {
  const int32_t depth = tree_depth(n, leaf_size, max_depth);
  const int64_t largest_leaf = (n + (int64_t{1} << depth) - 1) >> depth;
  if (largest_leaf >= (int64_t{1} << 30))
    return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build_device: a leaf would hold 2^30 points or more");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ICPNN_ERR_CUDA, std::string("kdtree_build_device: ") + cudaGetErrorString(e));
  const int64_t slots = int64_t{1} << (depth + 1);

  // the tree's own device arrays (kept), as kdtree_upload lays them out
  Node* nodes = nullptr;
  float* pts = nullptr;
  const size_t nb = static_cast<size_t>(slots) * sizeof(Node);
  const size_t bb = static_cast<size_t>(slots) * 8 * sizeof(float);
  e = pool_alloc(reinterpret_cast<void**>(&nodes), nb + bb, s);
  if (e == cudaSuccess) e = pool_alloc(reinterpret_cast<void**>(&pts), static_cast<size_t>(n) * 4 * sizeof(float), s);
  auto release = [&]() {
    if (nodes) cudaFreeAsync(nodes, s);
    if (pts) cudaFreeAsync(pts, s);
    cudaStreamSynchronize(s);
    cudaGetLastError();
  };
  if (e != cudaSuccess) {
    cudaGetLastError();
    release();
    return fail(e == cudaErrorMemoryAllocation ? ICPNN_ERR_NO_MEMORY : ICPNN_ERR_CUDA,
                std::string("kdtree_build_device: ") + cudaGetErrorString(e));
  }
  float4* boxes = reinterpret_cast<float4*>(reinterpret_cast<char*>(nodes) + nb);
  unsigned long long first_bad_host = ~0ull;
  float root_box[8];
  {
    DeviceMem m(s);
    float4* P = nullptr;
    uint32_t *keys = nullptr, *ids = nullptr, *alt_k = nullptr, *alt_v = nullptr, *temp = nullptr;
    float4* lists[2][3] = {};
    uint8_t* left = nullptr;
    double *part = nullptr, *mean = nullptr;
    uint32_t* cntl = nullptr;
    unsigned long long* first_bad = nullptr;
    int64_t max_blocks = 1;
    for (int d = 0; d <= depth; ++d) {
      const int64_t per = std::max<int64_t>(1, (((n + (int64_t{1} << d) - 1) >> d) + kChunk - 1) / kChunk);
      max_blocks = std::max(max_blocks, (int64_t{1} << d) * per);
    }
    if (e == cudaSuccess) e = m.alloc(&P, n);
    if (e == cudaSuccess) e = m.alloc(&keys, 3 * n);
    if (e == cudaSuccess) e = m.alloc(&ids, 3 * n);
    if (e == cudaSuccess) e = m.alloc(&alt_k, 3 * n);
    if (e == cudaSuccess) e = m.alloc(&alt_v, 3 * n);
    if (e == cudaSuccess) e = m.alloc(&temp, 3 * radix_temp_words(n));
    if (e == cudaSuccess) e = m.alloc(&lists[0][0], 3 * n);
    if (e == cudaSuccess) e = m.alloc(&lists[1][0], 3 * n);
    if (e == cudaSuccess) e = m.alloc(&left, n);
    if (e == cudaSuccess) e = m.alloc(&part, max_blocks * 9);
    if (e == cudaSuccess) e = m.alloc(&mean, (int64_t{1} << depth) * 3);
    if (e == cudaSuccess) e = m.alloc(&cntl, max_blocks * 3);
    if (e == cudaSuccess) e = m.alloc(&first_bad, 1);
    unsigned int* node_count = nullptr;  // per node of a level, zero between passes
    if (e == cudaSuccess) e = m.alloc(&node_count, int64_t{1} << depth);
    if (e == cudaSuccess) e = cudaMemsetAsync(node_count, 0, sizeof(unsigned int) << depth, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(nodes, 0, nb + bb, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(first_bad, 0xff, sizeof(unsigned long long), s);
    const int big_grid = static_cast<int>(std::min<int64_t>(grid_for(3 * n), 8 * 1024));
    if (e == cudaSuccess) {
      build_records_kernel<<<big_grid, 256, 0, s>>>(xyz_dev, n, P, keys, ids, first_bad);
      e = cudaGetLastError();
    }
    // one stable sort per axis by (coordinate, index): equal keys keep the
    // index order they start in
    uint32_t* sorted = ids;
    if (e == cudaSuccess) e = radix_sort(keys, ids, alt_k, alt_v, temp, n, 0, 32, s, &sorted, 3);
    if (e == cudaSuccess) {
      gather_lists_kernel<<<big_grid, 256, 0, s>>>(P, n, sorted, lists[0][0]);
      e = cudaGetLastError();
    }
    for (int b = 0; b < 2; ++b) {
      lists[b][1] = lists[b][0] + n;
      lists[b][2] = lists[b][0] + 2 * n;
    }
    int cur = 0;
    for (int d = 0; d <= depth && e == cudaSuccess; ++d) {
      LevelArgs a;
      a.d = d;
      a.n = n;
      a.leaf = leaf_size;
      a.max_depth = max_depth;
      a.round_robin = round_robin;
      const int64_t largest = (n + (int64_t{1} << d) - 1) >> d;
      a.blocks_per_node = static_cast<int>(std::max<int64_t>(1, (largest + kChunk - 1) / kChunk));
      const int blocks = static_cast<int>((int64_t{1} << d) * a.blocks_per_node);
      const int warp_grid = grid_for((int64_t{1} << d) * 32);  // one warp per node
      float4** L = lists[cur];
      float4** T = lists[cur ^ 1];
      float4* records = reinterpret_cast<float4*>(pts);
      const bool inner_level = d < depth;
      if (largest <= kWarpNode) {
        level_warp_kernel<<<warp_grid, 256, 0, s>>>(a, L[0], L[1], L[2], T[0], T[1], T[2], left, nodes, boxes,
                                                    records);
        g_launch_count.fetch_add(1, std::memory_order_relaxed);
      } else if (largest <= kBlockNode) {
        level_block_kernel<<<static_cast<int>(int64_t{1} << d), kBT, 0, s>>>(a, L[0], L[1], L[2], T[0], T[1], T[2],
                                                                            left, nodes, boxes, records);
        g_launch_count.fetch_add(1, std::memory_order_relaxed);
      } else {
        level_sums_kernel<<<blocks, kBT, 0, s>>>(a, L[0], part, node_count, mean, nodes, boxes);
        if (inner_level) level_sq_kernel<<<blocks, kBT, 0, s>>>(a, L[0], L[1], L[2], mean, part, node_count, nodes);
        level_flag_kernel<<<blocks, kBT, 0, s>>>(a, L[0], L[1], L[2], nodes, left, records);
        if (inner_level) {
          level_count_kernel<<<blocks, kBT, 0, s>>>(a, L[0], L[1], L[2], left, cntl, node_count);
          level_scatter_kernel<<<blocks, kBT, 0, s>>>(a, L[0], L[1], L[2], T[0], T[1], T[2], left, cntl);
        }
        g_launch_count.fetch_add(inner_level ? 5 : 2, std::memory_order_relaxed);
      }
      if (inner_level) cur ^= 1;
      e = cudaGetLastError();
    }
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(&first_bad_host, first_bad, sizeof(first_bad_host), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(root_box, boxes + 2, sizeof(root_box), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    release();
    return fail(e == cudaErrorMemoryAllocation ? ICPNN_ERR_NO_MEMORY : ICPNN_ERR_CUDA,
                std::string("kdtree_build_device: ") + cudaGetErrorString(e));
  }
  if (first_bad_host != ~0ull) {
    release();
    return fail(ICPNN_ERR_NONFINITE,
                "kdtree_build_device: non-finite coordinate at point " + std::to_string(first_bad_host));
  }
  // the number of nodes follows from the shape alone
  int64_t count = 0;
  std::vector<uint32_t> level{1u};
  for (int d = 0; !level.empty(); ++d) {
    std::vector<uint32_t> next;
    for (uint32_t k : level) {
      ++count;
      int64_t lo, cnt;
      node_range(k, d, n, leaf_size, max_depth, &lo, &cnt);
      if (!(cnt <= leaf_size || d >= max_depth)) {
        next.push_back(2 * k);
        next.push_back(2 * k + 1);
      }
    }
    level.swap(next);
  }
  t->n = n;
  t->leaf_size = leaf_size;
  t->max_depth = max_depth;
  t->round_robin = round_robin;
  t->depth = depth;
  t->heap_slots = slots;
  t->n_nodes = count;
  for (int d = 0; d < 3; ++d) {
    t->bbox_lo[d] = root_box[d];
    t->bbox_hi[d] = root_box[4 + d];
  }
  t->host_stale = true;
  t->dev.device = dev;
  t->dev.nodes = nodes;
  t->dev.boxes = reinterpret_cast<float*>(boxes);
  t->dev.points = pts;
  return ICPNN_OK;
}

}  // namespace icpnn
