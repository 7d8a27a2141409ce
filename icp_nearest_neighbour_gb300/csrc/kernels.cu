// Device code of libicpnn for sm_103a.
//
//  * Morton ordering of queries ("Implementing ICP with CUDA-KDTree",
//    section 5.3): bounding box, 30-bit Morton code per point, stable LSD
//    radix sort of (code, index), gather into float4 records.
//  * Exact KD-tree 1-NN search (section 3.2): depth-first, near child first,
//    far child kept on a per-thread stack with the squared distance to its
//    splitting plane and skipped when that bound exceeds the best distance.
//    The top levels of the tree are staged in shared memory.
//  * The fused ICP pass (sections 2.1, 3.3, 4.4): transform the original
//    source point, search, reject beyond the maximum distance, accumulate the
//    centroid and cross-covariance moments; warp-shuffle, then block, then a
//    last-block grid reduction, all in a fixed order so the result is
//    bit-reproducible run to run.
//
// Exactness.  Distances are d2 = (dx*dx + dy*dy) + dz*dz with dx = r.x - q.x,
// every operation an explicit round-to-nearest intrinsic, so no FMA
// contraction can change a bit.  The far child of a node is skipped only when
// fl(delta*delta) > best, where delta = fl(q_dim - split): rounding is
// monotone, so every point beyond the plane has |fl(r_dim - q_dim)| >=
// |delta| and hence d2 >= fl(delta*delta); a point at the best distance (a
// tie that may carry a lower index) is therefore never pruned, and the search
// returns the lexicographic minimum of (d2, index) whatever the tree shape or
// visiting order.
#include <cuda_runtime.h>

#include <cfloat>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "kernels.cuh"

namespace icpnn {

std::atomic<int64_t> g_launch_count{0};

namespace {

constexpr int kThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

// ------------------------------------------------------------ helpers ---

__host__ __device__ inline int32_t ordered_from_bits(int32_t i) { return i >= 0 ? i : (i ^ 0x7fffffff); }

__device__ __forceinline__ bool finite3(float x, float y, float z) {
  return isfinite(x) && isfinite(y) && isfinite(z);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

inline int num_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

inline int blocks_for(int64_t n, int per_block, int cap) {
  int64_t b = (n + per_block - 1) / per_block;
  if (b < 1) b = 1;
  if (b > cap) b = cap;
  return static_cast<int>(b);
}

// ------------------------------------------------------------ bbox ------

__global__ void bbox_init_kernel(int32_t* bbox6) {
  const int i = threadIdx.x;
  if (i < 3) bbox6[i] = INT_MAX;
  else if (i < 6) bbox6[i] = INT_MIN;
}

__global__ void __launch_bounds__(kThreads) bbox_kernel(const float* __restrict__ xyz, int64_t n,
                                                        int32_t* __restrict__ bbox6) {
  int32_t lo[3] = {INT_MAX, INT_MAX, INT_MAX};
  int32_t hi[3] = {INT_MIN, INT_MIN, INT_MIN};
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float x = xyz[3 * i], y = xyz[3 * i + 1], z = xyz[3 * i + 2];
    if (!finite3(x, y, z)) continue;
    const int32_t o[3] = {ordered_from_bits(__float_as_int(x)), ordered_from_bits(__float_as_int(y)),
                          ordered_from_bits(__float_as_int(z))};
#pragma unroll
    for (int d = 0; d < 3; ++d) {
      lo[d] = min(lo[d], o[d]);
      hi[d] = max(hi[d], o[d]);
    }
  }
  // warp, then block, then one atomic per block and bound (per-warp atomics
  // on the six words serialised: 14 us for 100k points)
  __shared__ int32_t s_box[kThreads / 32][6];
#pragma unroll
  for (int d = 0; d < 3; ++d) {
    lo[d] = __reduce_min_sync(kFull, lo[d]);
    hi[d] = __reduce_max_sync(kFull, hi[d]);
  }
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int d = 0; d < 3; ++d) {
      s_box[threadIdx.x >> 5][d] = lo[d];
      s_box[threadIdx.x >> 5][3 + d] = hi[d];
    }
  }
  __syncthreads();
  if (threadIdx.x < 6) {
    const int d = threadIdx.x;
    int32_t v = s_box[0][d];
    for (int w = 1; w < kThreads / 32; ++w) v = d < 3 ? min(v, s_box[w][d]) : max(v, s_box[w][d]);
    if (d < 3 && v != INT_MAX) atomicMin(&bbox6[d], v);
    if (d >= 3 && v != INT_MIN) atomicMax(&bbox6[d], v);
  }
}

// ------------------------------------------------------------ Morton ----

__device__ __forceinline__ uint32_t spread10(uint32_t v) {
  v &= 0x3ffu;
  v = (v | (v << 16)) & 0x030000ffu;
  v = (v | (v << 8)) & 0x0300f00fu;
  v = (v | (v << 4)) & 0x030c30c3u;
  v = (v | (v << 2)) & 0x09249249u;
  return v;
}

__device__ __forceinline__ float decode_ordered(int32_t o) {
  return __int_as_float(ordered_from_bits(o));
}

// shift_s from the device-computed source box (see IcpPassParams).
__device__ __forceinline__ void resolve_shift(IcpPassParams& p) {
  if (p.src_bbox6 == nullptr) return;
#pragma unroll
  for (int d = 0; d < 3; ++d)
    p.shift_s[d] = __fmul_rn(0.5f, __fadd_rn(decode_ordered(__ldg(&p.src_bbox6[d])),
                                             decode_ordered(__ldg(&p.src_bbox6[3 + d]))));
}

__global__ void __launch_bounds__(kThreads) morton_kernel(const float* __restrict__ xyz, int64_t n,
                                                          const int32_t* __restrict__ bbox6,
                                                          uint32_t* __restrict__ keys,
                                                          uint32_t* __restrict__ vals) {
  float lo[3], scale[3];
#pragma unroll
  for (int d = 0; d < 3; ++d) {
    const int32_t a = bbox6[d], b = bbox6[3 + d];
    if (a == INT_MAX || b == INT_MIN) {
      lo[d] = 0.f;
      scale[d] = 0.f;
    } else {
      lo[d] = decode_ordered(a);
      const float ext = decode_ordered(b) - lo[d];
      scale[d] = ext > 0.f ? 1024.f / ext : 0.f;
    }
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    uint32_t c[3];
#pragma unroll
    for (int d = 0; d < 3; ++d) {
      float q = (xyz[3 * i + d] - lo[d]) * scale[d];
      q = fminf(fmaxf(q, 0.f), 1023.f);  // NaN -> 0
      c[d] = static_cast<uint32_t>(q);
    }
    keys[i] = (spread10(c[0]) << 2) | (spread10(c[1]) << 1) | spread10(c[2]);
    vals[i] = static_cast<uint32_t>(i);
  }
}

// ------------------------------------------------------- radix sort -----
// One 8-bit digit per pass.  A pass is: per-tile digit histogram
// (hist[digit][tile]); an exclusive scan of every digit's row of tile counts,
// one block per digit, which also leaves each digit's total; a stable scatter
// whose blocks first turn the 256 digit totals into digit offsets.  The
// scatter is stable because ranks follow (round, warp, lane) = position
// order: a key's destination is its digit's offset, plus its tile's prefix
// for the digit, plus the counts of earlier rounds, earlier warps of this
// round, and earlier lanes of its warp (from __match_any_sync).

constexpr int kRadixBits = 8;
constexpr int kRadix = 1 << kRadixBits;
constexpr int kSortItems = 8;
constexpr int kSortTile = kThreads * kSortItems;

// Segments: blockIdx.y sorts its own array of n keys (offset blockIdx.y * n)
// with its own histogram region (offset blockIdx.y * (tiles + 1) * kRadix).
__device__ __forceinline__ int64_t seg_temp(int tiles) {
  return static_cast<int64_t>(blockIdx.y) * (static_cast<int64_t>(tiles) + 1) * kRadix;
}

__global__ void __launch_bounds__(kThreads) radix_hist_kernel(const uint32_t* __restrict__ keys, int64_t n,
                                                              int shift, uint32_t* __restrict__ hist,
                                                              int tiles) {
  __shared__ uint32_t cnt[kRadix];
  keys += static_cast<int64_t>(blockIdx.y) * n;
  hist += seg_temp(tiles);
  for (int i = threadIdx.x; i < kRadix; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kSortTile;
#pragma unroll
  for (int r = 0; r < kSortItems; ++r) {
    const int64_t p = base + r * kThreads + threadIdx.x;
    if (p < n) atomicAdd(&cnt[(keys[p] >> shift) & (kRadix - 1)], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kRadix; i += blockDim.x)
    hist[static_cast<int64_t>(i) * tiles + blockIdx.x] = cnt[i];
}

// Exclusive scan of the block's values (one per thread, blockDim.x == kThreads).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t u = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x += u;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kThreads / 32 ? warp_sums[lane] : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t u = __shfl_up_sync(kFull, w, off);
      if (lane >= off) w += u;
    }
    if (lane < kThreads / 32) warp_sums[lane] = w;
  }
  __syncthreads();
  const uint32_t excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0u);
  if (total != nullptr) *total = warp_sums[kThreads / 32 - 1];
  __syncthreads();
  return excl;
}

// Block d: exclusive scan of hist[d][0..tiles) in place; digit_total[d] = row sum.
__global__ void __launch_bounds__(kThreads) digit_row_scan_kernel(uint32_t* __restrict__ hist, int tiles,
                                                                  uint32_t* __restrict__ digit_total) {
  __shared__ uint32_t warp_sums[kThreads / 32];
  hist += seg_temp(tiles);
  digit_total += seg_temp(tiles);
  uint32_t* row = hist + static_cast<int64_t>(blockIdx.x) * tiles;
  uint32_t carry = 0;
  for (int base = 0; base < tiles; base += kThreads) {
    const int i = base + threadIdx.x;
    const uint32_t v = i < tiles ? row[i] : 0u;
    uint32_t chunk_total;
    const uint32_t excl = block_exclusive_scan(v, warp_sums, &chunk_total);
    if (i < tiles) row[i] = carry + excl;
    carry += chunk_total;
  }
  if (threadIdx.x == 0) digit_total[blockIdx.x] = carry;
}

__global__ void __launch_bounds__(kThreads) radix_scatter_kernel(
    const uint32_t* __restrict__ keys_in, const uint32_t* __restrict__ vals_in,
    uint32_t* __restrict__ keys_out, uint32_t* __restrict__ vals_out, int64_t n, int shift,
    const uint32_t* __restrict__ row_prefix, const uint32_t* __restrict__ digit_total, int tiles) {
  static_assert(kThreads == kRadix, "one thread per digit when forming offsets");
  constexpr int kWarps = kThreads / 32;
  __shared__ uint32_t base[kRadix];
  __shared__ uint32_t wcount[kWarps][kRadix];
  __shared__ uint32_t warp_sums[kWarps];
  const int t = threadIdx.x, warp = t >> 5;
  {
    const int64_t e = static_cast<int64_t>(blockIdx.y) * n;
    keys_in += e;
    vals_in += e;
    keys_out += e;
    vals_out += e;
    row_prefix += seg_temp(tiles);
    digit_total += seg_temp(tiles);
  }
  const uint32_t digit_offset = block_exclusive_scan(digit_total[t], warp_sums, nullptr);
  base[t] = digit_offset + row_prefix[static_cast<int64_t>(t) * tiles + blockIdx.x];
  const int64_t tile0 = static_cast<int64_t>(blockIdx.x) * kSortTile;
  for (int r = 0; r < kSortItems; ++r) {
    for (int i = t; i < kWarps * kRadix; i += kThreads) (&wcount[0][0])[i] = 0;
    __syncthreads();
    const int64_t p = tile0 + r * kThreads + t;
    const bool valid = p < n;
    const uint32_t key = valid ? keys_in[p] : 0u;
    const uint32_t val = valid ? vals_in[p] : 0u;
    const uint32_t digit = valid ? ((key >> shift) & (kRadix - 1)) : 0xffffffffu;
    const uint32_t peers = __match_any_sync(kFull, digit);
    const uint32_t rank = __popc(peers & lanemask_lt());
    if (valid && rank == 0) wcount[warp][digit] = __popc(peers);
    __syncthreads();
    if (valid) {
      uint32_t off = base[digit] + rank;
      for (int w = 0; w < warp; ++w) off += wcount[w][digit];
      keys_out[off] = key;
      vals_out[off] = val;
    }
    __syncthreads();
    uint32_t sum = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) sum += wcount[w][t];
    base[t] += sum;
    __syncthreads();
  }
}

// ------------------------------------------------------------ voxels ----
// Voxel-grid downsampling ("Implementing ICP with CUDA-KDTree", section 4.3):
// voxel index floor(x / v) per axis (float32 division, grid anchored at the
// origin), one output point per occupied voxel, the centroid of its points
// summed in input order in double and rounded to float32, voxels ordered by
// (ix, iy, iz).  Non-finite points are dropped.

constexpr double kVoxelIndexLimit = 1099511627776.0;  // 2^40

__device__ __forceinline__ bool voxel_index(const float* __restrict__ xyz, int64_t i, float v,
                                            long long (&k)[3]) {
  const float x = xyz[3 * i], y = xyz[3 * i + 1], z = xyz[3 * i + 2];
  if (!finite3(x, y, z)) return false;
  k[0] = static_cast<long long>(floorf(__fdiv_rn(x, v)));
  k[1] = static_cast<long long>(floorf(__fdiv_rn(y, v)));
  k[2] = static_cast<long long>(floorf(__fdiv_rn(z, v)));
  return true;
}

// bounds: lo[3], hi[3] (int64 voxel indices), [6] finite points, [7] out-of-range flag
__global__ void voxel_bounds_init_kernel(long long* bounds) {
  const int i = threadIdx.x;
  if (i < 3) bounds[i] = LLONG_MAX;
  else if (i < 6) bounds[i] = LLONG_MIN;
  else if (i < 8) bounds[i] = 0;
}

__global__ void __launch_bounds__(kThreads) voxel_bounds_kernel(const float* __restrict__ xyz, int64_t n,
                                                                float v, long long* __restrict__ bounds) {
  long long lo[3] = {LLONG_MAX, LLONG_MAX, LLONG_MAX}, hi[3] = {LLONG_MIN, LLONG_MIN, LLONG_MIN};
  unsigned long long cnt = 0, bad = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float x = xyz[3 * i], y = xyz[3 * i + 1], z = xyz[3 * i + 2];
    if (!finite3(x, y, z)) continue;
    const float q[3] = {floorf(__fdiv_rn(x, v)), floorf(__fdiv_rn(y, v)), floorf(__fdiv_rn(z, v))};
    bool ok = true;
#pragma unroll
    for (int d = 0; d < 3; ++d) ok = ok && fabsf(q[d]) < static_cast<float>(kVoxelIndexLimit);
    if (!ok) {
      ++bad;
      continue;
    }
    ++cnt;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
      const long long k = static_cast<long long>(q[d]);
      lo[d] = min(lo[d], k);
      hi[d] = max(hi[d], k);
    }
  }
#pragma unroll
  for (int d = 0; d < 3; ++d) {
    for (int off = 16; off > 0; off >>= 1) {
      lo[d] = min(lo[d], __shfl_xor_sync(kFull, lo[d], off));
      hi[d] = max(hi[d], __shfl_xor_sync(kFull, hi[d], off));
    }
  }
  for (int off = 16; off > 0; off >>= 1) {
    cnt += __shfl_xor_sync(kFull, cnt, off);
    bad += __shfl_xor_sync(kFull, bad, off);
  }
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int d = 0; d < 3; ++d) {
      if (lo[d] != LLONG_MAX) atomicMin(&bounds[d], lo[d]);
      if (hi[d] != LLONG_MIN) atomicMax(&bounds[3 + d], hi[d]);
    }
    if (cnt) atomicAdd(reinterpret_cast<unsigned long long*>(&bounds[6]), cnt);
    if (bad) atomicAdd(reinterpret_cast<unsigned long long*>(&bounds[7]), bad);
  }
}

struct VoxelGrid {
  float v;
  long long lo[3];
  unsigned long long ry, rz;      // index ranges of y and z
  unsigned long long sentinel;    // key of a dropped point: sorts after every voxel
};

__device__ __forceinline__ unsigned long long voxel_key(const float* __restrict__ xyz, int64_t i,
                                                        const VoxelGrid& g) {
  long long k[3];
  if (!voxel_index(xyz, i, g.v, k)) return g.sentinel;
  return (static_cast<unsigned long long>(k[0] - g.lo[0]) * g.ry + static_cast<unsigned long long>(k[1] - g.lo[1])) *
             g.rz +
         static_cast<unsigned long long>(k[2] - g.lo[2]);
}

__global__ void __launch_bounds__(kThreads) voxel_keys_kernel(const float* __restrict__ xyz, int64_t n,
                                                              VoxelGrid g, uint32_t* __restrict__ key_lo,
                                                              uint32_t* __restrict__ key_hi,
                                                              uint32_t* __restrict__ vals) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const unsigned long long k = voxel_key(xyz, i, g);
    key_lo[i] = static_cast<uint32_t>(k);
    if (key_hi) key_hi[i] = static_cast<uint32_t>(k >> 32);
    vals[i] = static_cast<uint32_t>(i);
  }
}

__global__ void __launch_bounds__(kThreads) gather_u32_kernel(const uint32_t* __restrict__ src,
                                                              const uint32_t* __restrict__ perm, int64_t n,
                                                              uint32_t* __restrict__ dst) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = src[perm[i]];
}

// Voxel key of every kept point in sorted order (computed once; the run
// boundaries and centroids below compare these instead of recomputing).
__global__ void __launch_bounds__(kThreads) voxel_sorted_keys_kernel(const float* __restrict__ xyz,
                                                                     const uint32_t* __restrict__ order, int64_t m,
                                                                     VoxelGrid g,
                                                                     unsigned long long* __restrict__ skey) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < m; i += stride)
    skey[i] = voxel_key(xyz, order[i], g);
}

__device__ __forceinline__ bool voxel_head(const unsigned long long* __restrict__ skey, int64_t i, int64_t m) {
  if (i >= m) return false;
  return i == 0 || skey[i] != skey[i - 1];
}

// per block of kThreads sorted positions: number of voxel heads
__global__ void __launch_bounds__(kThreads) voxel_head_count_kernel(const unsigned long long* __restrict__ skey,
                                                                    int64_t m, uint32_t* __restrict__ block_heads) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const uint32_t h = voxel_head(skey, i, m) ? 1u : 0u;
  const uint32_t c = __reduce_add_sync(kFull, h);
  __shared__ uint32_t warp_c[kThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_c[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int w = 0; w < kThreads / 32; ++w) t += warp_c[w];
    block_heads[blockIdx.x] = t;
  }
}

// exclusive scan of `count` words in place by one block; total to *total
__global__ void __launch_bounds__(kThreads) scan_one_block_kernel(uint32_t* __restrict__ data, int64_t count,
                                                                  unsigned long long* __restrict__ total) {
  __shared__ uint32_t warp_sums[kThreads / 32];
  uint32_t carry = 0;
  for (int64_t base = 0; base < count; base += kThreads) {
    const int64_t i = base + threadIdx.x;
    const uint32_t v = i < count ? data[i] : 0u;
    uint32_t chunk_total;
    const uint32_t excl = block_exclusive_scan(v, warp_sums, &chunk_total);
    if (i < count) data[i] = carry + excl;
    carry += chunk_total;
  }
  if (threadIdx.x == 0) *total = carry;
}

// every voxel head: its ordinal (block offset + rank in block), then the
// centroid of its run of equal keys, summed in sorted (= input) order; the
// run's keys and indices are read four at a time.
__global__ void __launch_bounds__(kThreads) voxel_emit_kernel(const float* __restrict__ xyz,
                                                              const uint32_t* __restrict__ order, int64_t m,
                                                              const unsigned long long* __restrict__ skey,
                                                              const uint32_t* __restrict__ block_offset,
                                                              float* __restrict__ out) {
  __shared__ uint32_t warp_sums[kThreads / 32];
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const bool head = voxel_head(skey, i, m);
  const uint32_t rank = block_exclusive_scan(head ? 1u : 0u, warp_sums, nullptr);
  if (!head) return;
  const int64_t ord = static_cast<int64_t>(block_offset[blockIdx.x]) + rank;
  const unsigned long long key = skey[i];
  double sx = 0.0, sy = 0.0, sz = 0.0;
  int64_t j = i;
  for (bool more = true; more;) {
    uint32_t p[4];
    bool in[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t jj = j + u;
      in[u] = jj < m && skey[jj] == key;
      p[u] = in[u] ? order[jj] : 0u;
    }
    float c[4][3];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t q = static_cast<int64_t>(p[u]);
      c[u][0] = in[u] ? xyz[3 * q] : 0.f;
      c[u][1] = in[u] ? xyz[3 * q + 1] : 0.f;
      c[u][2] = in[u] ? xyz[3 * q + 2] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (!in[u]) {
        more = false;
        break;
      }
      sx += static_cast<double>(c[u][0]);
      sy += static_cast<double>(c[u][1]);
      sz += static_cast<double>(c[u][2]);
      ++j;
    }
  }
  const double cnt = static_cast<double>(j - i);
  out[3 * ord] = static_cast<float>(sx / cnt);
  out[3 * ord + 1] = static_cast<float>(sy / cnt);
  out[3 * ord + 2] = static_cast<float>(sz / cnt);
}

// ------------------------------------------------------------ gather ----

__global__ void __launch_bounds__(kThreads) gather_kernel(const float* __restrict__ xyz, int64_t n,
                                                          const uint32_t* __restrict__ perm,
                                                          float4* __restrict__ rec) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t p = perm ? static_cast<int64_t>(perm[i]) : i;
    rec[i] = make_float4(xyz[3 * p], xyz[3 * p + 1], xyz[3 * p + 2], __int_as_float(static_cast<int32_t>(p)));
  }
}

// ------------------------------------------------------------ search ----

struct TreeView {
  const uint2* __restrict__ nodes;   // heap, 1-based
  const float4* __restrict__ boxes;  // per heap slot: lo, hi (tight box of the node's points)
  const float4* __restrict__ pts;    // leaf-ordered records
  const uint2* smem;                 // copy of heap slots [0, smem_slots)
  uint32_t smem_slots;
};

// The running best as one 64-bit key (d2 bits << 32) | original index.  d2
// is a sum of squares, never negative zero or NaN for a finite query, so its
// IEEE bits order exactly like its values, and one unsigned 64-bit compare is
// the lexicographic (d2, index) test of the exact-neighbour definition.  The
// index field starts at INT_MAX, above every real index.
struct Best {
  unsigned long long key;
  uint32_t slot;  // position of the best point's record
  __device__ __forceinline__ float d2() const { return __uint_as_float(static_cast<uint32_t>(key >> 32)); }
  __device__ __forceinline__ int32_t idx() const { return static_cast<int32_t>(key & 0xffffffffu); }
};
__device__ __forceinline__ Best make_best(float d2) {
  return Best{(static_cast<unsigned long long>(__float_as_uint(d2)) << 32) | 0x7fffffffull, 0u};
}

// One generic load: the top levels come from the shared-memory copy, the rest
// from global memory, selected by pointer rather than by branch.
__device__ __forceinline__ uint2 load_node(const TreeView& tv, uint32_t i) {
  const uint2* p = i < tv.smem_slots ? tv.smem : tv.nodes;
  return p[i];
}

__device__ __forceinline__ float dist2(const float4& r, float qx, float qy, float qz) {
  const float dx = __fsub_rn(r.x, qx);
  const float dy = __fsub_rn(r.y, qy);
  const float dz = __fsub_rn(r.z, qz);
  return __fadd_rn(__fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy)), __fmul_rn(dz, dz));
}

__device__ __forceinline__ void consider(const float4& r, uint32_t slot, float qx, float qy, float qz,
                                         Best& b) {
  const float d = dist2(r, qx, qy, qz);
  const unsigned long long key = (static_cast<unsigned long long>(__float_as_uint(d)) << 32) | __float_as_uint(r.w);
  if (key < b.key) {
    b.key = key;
    b.slot = slot;
  }
}

// Exact nearest neighbour of a finite query point, depth first, near child
// first.  Instead of a stack of pending far children the search keeps a
// 32-bit trail: bit d is set while the far child at depth d of the current
// path still has to be visited (at most one per level, depth <= 20).  In the
// implicit heap the pending node is the sibling of the current path's node at
// that depth, (node >> (depth - d)) ^ 1, and its bound is recomputed from its
// parent's splitting plane when it is taken up -- against the best distance
// of that moment, which has usually shrunk.  All state lives in registers:
// no local-memory stack.  (A restart trail in the sense of Laine, "Restart
// trail for stackless BVH traversal", 2010; the heap numbering makes the
// restart from the root unnecessary.)
__device__ __forceinline__ void scan_leaf(const TreeView& tv, uint2 nd, float qx, float qy, float qz, Best& b) {
  const uint32_t start = nd.x;
  const uint32_t count = nd.y >> 2;
  uint32_t k = 0;
  for (; k + 4 <= count; k += 4) {
    const float4 r0 = __ldg(&tv.pts[start + k]);
    const float4 r1 = __ldg(&tv.pts[start + k + 1]);
    const float4 r2 = __ldg(&tv.pts[start + k + 2]);
    const float4 r3 = __ldg(&tv.pts[start + k + 3]);
    consider(r0, start + k, qx, qy, qz, b);
    consider(r1, start + k + 1, qx, qy, qz, b);
    consider(r2, start + k + 2, qx, qy, qz, b);
    consider(r3, start + k + 3, qx, qy, qz, b);
  }
  for (; k < count; ++k) consider(__ldg(&tv.pts[start + k]), start + k, qx, qy, qz, b);
}

// Lower bound for the subtree of `node` given its parent's record: 0 when the
// query lies on node's side of the parent's splitting plane, else the squared
// distance to that plane.
__device__ __forceinline__ float sibling_bound(uint2 parent, uint32_t node, float qx, float qy, float qz) {
  const float qd = parent.y == 0 ? qx : (parent.y == 1 ? qy : qz);
  const float split = __uint_as_float(parent.x);
  const bool same_side = ((node & 1u) == 0u) == (qd < split);
  const float delta = __fsub_rn(qd, split);
  return same_side ? 0.f : __fmul_rn(delta, delta);
}

// Lower bound for every point of a node: the squared distance from the query
// to the node's box, with the rounding of dist2 (per-axis offset rounded,
// squared, summed as (x + y) + z).  Rounding is monotone, so no point in the
// box has a smaller dist2, and a node whose bound exceeds the best distance
// cannot hold an equal or better point.
__device__ __forceinline__ float box_dist2(const float4& lo, const float4& hi, float qx, float qy, float qz) {
  const float ox = fmaxf(fmaxf(__fsub_rn(lo.x, qx), __fsub_rn(qx, hi.x)), 0.f);
  const float oy = fmaxf(fmaxf(__fsub_rn(lo.y, qy), __fsub_rn(qy, hi.y)), 0.f);
  const float oz = fmaxf(fmaxf(__fsub_rn(lo.z, qz), __fsub_rn(qz, hi.z)), 0.f);
  return __fadd_rn(__fadd_rn(__fmul_rn(ox, ox), __fmul_rn(oy, oy)), __fmul_rn(oz, oz));
}
__device__ __forceinline__ float box_bound(const TreeView& tv, uint32_t node, float qx, float qy, float qz) {
  return box_dist2(__ldg(&tv.boxes[2 * node]), __ldg(&tv.boxes[2 * node + 1]), qx, qy, qz);
}

// Scan a leaf reached by descent if its box is within reach.  The box and the
// leaf's first records are fetched together, so the test adds no round trip
// when it passes.  kWide: records six at a time, the last batch padded with
// repeated loads of the last record -- for queries in no particular order,
// whose leaves mostly miss L1, one round trip more per leaf costs more than
// the registers (1M unordered queries: 0.47 -> 0.36 ms); the ICP passes,
// warm in L1, keep four at a time (six measured slower on LiDAR's 16-record
// leaves).
template <bool kWide>
__device__ __forceinline__ void scan_leaf_boxed(const TreeView& tv, uint32_t node, uint2 nd, float qx, float qy,
                                                float qz, Best& b) {
  const uint32_t start = nd.x;
  const uint32_t count = nd.y >> 2;  // >= 1
  const float4 lo = __ldg(&tv.boxes[2 * node]);
  const float4 hi = __ldg(&tv.boxes[2 * node + 1]);
  if (kWide) {
    float4 r[6];
#pragma unroll
    for (int u = 0; u < 6; ++u) r[u] = __ldg(&tv.pts[start + min(static_cast<uint32_t>(u), count - 1)]);
    if (box_dist2(lo, hi, qx, qy, qz) > b.d2()) return;
#pragma unroll
    for (int u = 0; u < 6; ++u)
      if (static_cast<uint32_t>(u) < count) consider(r[u], start + u, qx, qy, qz, b);
    for (uint32_t k = 6; k < count; k += 6) {
#pragma unroll
      for (int u = 0; u < 6; ++u) r[u] = __ldg(&tv.pts[start + min(k + u, count - 1)]);
#pragma unroll
      for (int u = 0; u < 6; ++u)
        if (k + u < count) consider(r[u], start + k + u, qx, qy, qz, b);
    }
    return;
  }
  const float4 r0 = __ldg(&tv.pts[start]);
  const float4 r1 = count > 1 ? __ldg(&tv.pts[start + 1]) : r0;
  const float4 r2 = count > 2 ? __ldg(&tv.pts[start + 2]) : r0;
  const float4 r3 = count > 3 ? __ldg(&tv.pts[start + 3]) : r0;
  if (box_dist2(lo, hi, qx, qy, qz) > b.d2()) return;
  consider(r0, start, qx, qy, qz, b);
  if (count > 1) consider(r1, start + 1, qx, qy, qz, b);
  if (count > 2) consider(r2, start + 2, qx, qy, qz, b);
  if (count > 3) consider(r3, start + 3, qx, qy, qz, b);
  uint32_t k = 4;
  for (; k + 4 <= count; k += 4) {
    const float4 s0 = __ldg(&tv.pts[start + k]);
    const float4 s1 = __ldg(&tv.pts[start + k + 1]);
    const float4 s2 = __ldg(&tv.pts[start + k + 2]);
    const float4 s3 = __ldg(&tv.pts[start + k + 3]);
    consider(s0, start + k, qx, qy, qz, b);
    consider(s1, start + k + 1, qx, qy, qz, b);
    consider(s2, start + k + 2, qx, qy, qz, b);
    consider(s3, start + k + 3, qx, qy, qz, b);
  }
  for (; k < count; ++k) consider(__ldg(&tv.pts[start + k]), start + k, qx, qy, qz, b);
}

// Exact nearest neighbour, optionally warm-started at a leaf (start > 1: the
// leaf where this query's best point was found in the previous pass).
// Returns the leaf holding the best point found by this search (0 if none).
// The descent takes the near side of each splitting plane (8-byte node loads);
// the far child is recorded as pending only if its plane and its box are both
// within reach, a pending sibling is taken up if its plane still is, and a
// leaf reached by descent is scanned only if its box is.  For points off a
// sampled surface -- every query of an early ICP pass, or a scan against
// another scan -- the boxes are far tighter than the planes (a cell of a flat
// region is unbounded across it): several-fold fewer leaves and pending
// siblings.
template <bool kWide = false>
__device__ __forceinline__ uint32_t search_from(const TreeView& tv, float qx, float qy, float qz, Best& b,
                                                uint32_t start) {
  uint32_t node = 1, depth = 0, trail = 0, best_leaf = 0;
  uint2 nd;
  bool scanned = false;
  if (start > 1) {
    // Warm start: scan the leaf, then bound every sibling along its root path
    // by its box at once (independent loads), keeping the ones still within
    // reach as pending; with the leaf they cover the whole tree, so the result
    // is the same exact neighbour from any starting leaf.
    node = start;
    depth = 31u - __clz(start);
    const unsigned long long before = b.key;
    scan_leaf(tv, load_node(tv, node), qx, qy, qz, b);
    if (b.key != before) best_leaf = node;
#pragma unroll
    for (uint32_t lvl = 1; lvl <= ICPNN_MAX_DEPTH; ++lvl) {
      if (lvl <= depth) {
        const uint32_t sib = (node >> (depth - lvl)) ^ 1u;
        if (box_bound(tv, sib, qx, qy, qz) <= b.d2()) trail |= 1u << lvl;
      }
    }
    scanned = true;
  } else {
    if (box_bound(tv, 1u, qx, qy, qz) > b.d2()) return 0u;  // nothing within the initial radius
    nd = load_node(tv, node);
  }
  for (;;) {
    if (!scanned) {
      while ((nd.y & 3u) != kLeafTag) {
        const float qd = nd.y == 0 ? qx : (nd.y == 1 ? qy : qz);
        const float split = __uint_as_float(nd.x);
        const float delta = __fsub_rn(qd, split);
        const uint32_t near = 2 * node + (qd < split ? 0u : 1u);
        const uint2 next = load_node(tv, near);
        ++depth;
        // the far child becomes pending only if both its plane and its box
        // are within reach (the box loads overlap the near child's load)
        if (__fmul_rn(delta, delta) <= b.d2() && box_bound(tv, near ^ 1u, qx, qy, qz) <= b.d2())
          trail |= 1u << depth;
        node = near;
        nd = next;
      }
      const unsigned long long before = b.key;
      scan_leaf_boxed<kWide>(tv, node, nd, qx, qy, qz, b);
      if (b.key != before) best_leaf = node;
    }
    scanned = false;
    // take up the deepest pending sibling still within reach of the best
    for (;;) {
      if (trail == 0) return best_leaf;
      const uint32_t d = 31u - __clz(trail);
      trail &= ~(1u << d);
      node = (node >> (depth - d)) ^ 1u;
      depth = d;
      const uint2 parent = load_node(tv, node >> 1);
      nd = load_node(tv, node);
      // the box passed when the sibling was recorded; the best may have
      // shrunk since, so the cheap plane test is repeated
      if (sibling_bound(parent, node, qx, qy, qz) <= b.d2()) break;
    }
  }
}

template <bool kWide = false>
__device__ __forceinline__ void search(const TreeView& tv, float qx, float qy, float qz, Best& b) {
  search_from<kWide>(tv, qx, qy, qz, b, 1u);
}

// Work distribution of the search kernels: queries are taken in chunks of 32
// consecutive (Morton-ordered, so spatially coherent) records, one chunk per
// warp, and the warps of a block take consecutive chunks, so a block -- and
// the L1 cache of the SM it runs on -- works on one region of the cloud.
// (Dealing chunks round-robin over the blocks balances the SMs better but
// loses that locality and was measured slower.)  The mapping depends only on
// n and the grid, so every reduction order stays fixed.
__device__ __forceinline__ int64_t first_chunk() {
  return static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
}
__device__ __forceinline__ int64_t chunk_stride() {
  return static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
}

__device__ __forceinline__ void stage_top(const uint2* __restrict__ nodes, uint2* s_nodes, int slots) {
  const uint4* src = reinterpret_cast<const uint4*>(nodes);
  uint4* dst = reinterpret_cast<uint4*>(s_nodes);
  for (int i = threadIdx.x; i < slots / 2; i += blockDim.x) dst[i] = __ldg(src + i);
  __syncthreads();
}

// ------------------------------------------------------------ NN query --

__global__ void __launch_bounds__(kThreads) nn_kernel(const uint2* __restrict__ nodes,
                                                      const float4* __restrict__ boxes,
                                                      const float4* __restrict__ pts, int smem_slots,
                                                      const float4* __restrict__ q, int64_t n,
                                                      int32_t* __restrict__ out_idx,
                                                      float* __restrict__ out_d2,
                                                      unsigned int* __restrict__ chunk_counter) {
  extern __shared__ __align__(16) uint2 s_nodes[];
  stage_top(nodes, s_nodes, smem_slots);
  const TreeView tv{nodes, boxes, pts, s_nodes, static_cast<uint32_t>(smem_slots)};
  const int lane = threadIdx.x & 31;
  // The grid is one wave; with more queries than resident warps each warp
  // starts at its own chunk (warps of a block on consecutive chunks) and then
  // takes the next unclaimed chunk from a counter, so that warps whose chunks
  // were cheap take over the rest instead of waiting for a fixed share.
  for (int64_t c = first_chunk(); c * 32 < n;) {
    const int64_t i = c * 32 + lane;
    if (i < n) {
      const float4 r = q[i];
      const int32_t slot = __float_as_int(r.w);
      if (!finite3(r.x, r.y, r.z)) {
        out_idx[slot] = -1;
        out_d2[slot] = __int_as_float(0x7fc00000);
      } else {
        Best b = make_best(__int_as_float(0x7f800000));
        search<true>(tv, r.x, r.y, r.z, b);
        out_idx[slot] = b.idx() == INT_MAX ? -1 : b.idx();
        out_d2[slot] = b.d2();
      }
    }
    unsigned int next = 0;
    if (lane == 0) next = atomicAdd(chunk_counter, 1u);
    c = chunk_stride() + __shfl_sync(kFull, next, 0);
  }
}

// ------------------------------------------------------------ ICP pass --

// Reduction of the per-thread moments of a pass, in a fixed order: warp
// butterfly in float (lane 0's association order is the same every run), the
// block's 8 warps in a float-float butterfly of 8 lanes, then the last block
// to finish sums the block partials (see below).  Slots: [0] = c0, [1] = c1 (counts),
// [2 + v] = acc[v].  Without kPublish the last block stores them as doubles
// at out; with kPublish it publishes them as tagged words (kResultWords), or,
// in a pass that gave up waiting for its command, stores `seq` in the abort
// word instead and leaves the result untouched.
// The float threshold t with float(e2) <= t exactly when e2 <= limit in
// double: the largest float not above limit (+inf stays +inf).
__device__ __forceinline__ float float_threshold_dev(double limit) {
  if (isinf(limit)) return __int_as_float(0x7f800000);
  if (limit >= static_cast<double>(FLT_MAX)) return FLT_MAX;
  float f = __double2float_rn(limit);
  if (static_cast<double>(f) > limit) f = nextafterf(f, -__int_as_float(0x7f800000));
  return f;
}

// With thr_out, the last block also stores the 3-sigma threshold of the
// residual rejection from this reduction's c1 (pairs) and acc[15] (sum of e2):
// float_threshold(9 * sum_e2 / pairs), 0 pairs giving sigma^2 = 0.
//
// `skipped` (block-uniform) is this block's outcome when the pass waited for a
// command: 0 ran, kSkipStopped found the stop bit or a later seq, kSkipTimedOut
// found no command in time.  counter[1] collects them; the last block
// publishes the result only if every block ran.
//
// Grids of up to kSingleLevelBlocks blocks (every grid of the search kernels:
// at most three blocks per SM) reduce in one level: the last block to finish
// (counter[0]) adds every block's partial: 252 threads, each taking two
// slots of every 28th row in row order, one 16-byte load per row and up to 14
// loads in flight (one round trip for a 391-block grid); then 8 lanes per slot
// add the 28 row groups, lane j groups j, j + 8, ... in order, and an 8-lane
// butterfly adds the lanes (a 28-step chain before: 0.3 us longer).  Partials and sums are
// float-float pairs (see ff_add): with doubles, the last block's 7,000
// additions for a 391-block grid took 3.6-4.1 us of FP64 pipe, the longest
// step of a pass's tail; as float-float they cost a fraction of that (scene
// registration 2.28 -> 2.21 ms, residual iteration 23 -> 16.5 us; the 16-byte
// loads then 2.19 -> 2.16 ms and 16.6 -> 15.0 us).  Larger grids
// reduce in two fixed-order levels: the last block to finish of each group of
// kGroupBlocks consecutive blocks (counter[2 + group]) adds the group's
// partials in block order, one load per thread, and stores the sum over the
// group's first partial; the last group to finish (counter[0]) adds the group
// sums.
constexpr unsigned int kSkipStopped = 1u, kSkipTimedOut = 1u << 16;
// at least every grid of the search kernels (three blocks per SM on 152 SMs)
constexpr unsigned int kSingleLevelBlocks = 462;
static_assert(kGroupBlocks * kMomentSlots <= kThreads, "one thread per partial of a group");

// Release-only increment: orders this thread's earlier stores before the
// increment without the acquire half, which would invalidate the SM's L1 (a
// persistent kernel keeps the tree in L1 from one pass to the next).
__device__ __forceinline__ unsigned int atom_add_release_gpu(unsigned int* a, unsigned int v) {
  unsigned int old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// kPersistent: the block's stores to partials are made by thread 0, which
// then increments the counters with release atomics; only a block that finds
// itself last takes the acquire fence.  The sums are the same in the same
// order either way.  *t_start (if given) is the global time at which the pass
// received its command; the last block publishes its low 32 bits and those of
// the publish time with the result.
// Float-float sums (an unevaluated pair hi + lo of float32 values, about 44
// significant bits): GB300's double-precision rate is a small fraction of its
// float32 rate, and the final sum over every block's partial was the longest
// step of a pass's tail.  TwoSum of the high parts, then the low parts added
// in and the pair renormalised.
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float bb = __fsub_rn(s, a.hi);
  const float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
  const float e = __fadd_rn(err, __fadd_rn(a.lo, b.lo));
  const float hi = __fadd_rn(s, e);
  return FF{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}

// Sum of s over each aligned group of 8 lanes, left in all 8 lanes: a
// three-level butterfly (ff_add is commutative bit for bit: TwoSum's error
// term is exact whichever operand comes first).
__device__ __forceinline__ FF ff_allreduce8(FF s) {
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) {
    const FF o{__shfl_xor_sync(kFull, s.hi, off), __shfl_xor_sync(kFull, s.lo, off)};
    s = ff_add(s, o);
  }
  return s;
}
// Threads that take part in the 8-lane sums: 8 per slot, whole warps.
constexpr int kTreeThreads = (kMomentSlots * 8 + 31) / 32 * 32;
static_assert(kTreeThreads <= kThreads, "8 lanes per slot within the block");

// Shared memory of reduce_moments, one instance per block whichever variants
// of the reduction a kernel uses (a __shared__ array declared inside the
// template would be allocated once per instantiation).
constexpr int kRowGroups = kThreads / (kMomentSlots / 2);
struct ReduceShared {
  FF warp[kThreads / 32][kMomentSlots];
  FF fin[kThreads / kMomentSlots][kMomentSlots];
  FF rows[kRowGroups][kMomentSlots];
  FF res[kMomentSlots];  // the final sums, as float-float pairs
  unsigned long long t_cmd;
  bool last, publish;
};
__device__ __forceinline__ ReduceShared& reduce_shared() {
  __shared__ ReduceShared s;
  return s;
}

// kSigmaOnly: only c1 (slot 1) and acc[15] (slot 17) are reduced -- the first
// residual pass, whose one product is the threshold.  Those two sums take
// exactly the operations, in the same order, that a full reduction of the same
// values takes, so the threshold's sigma^2 is the one the host later reads from
// the second residual pass (which carries the same two sums).  Nothing is
// stored to `out` but the abort word.
template <bool kPublish, bool kPersistent = false, bool kSigmaOnly = false>
__device__ __forceinline__ void reduce_moments(float (&acc)[16], uint32_t c0, uint32_t c1,
                                               double* __restrict__ partials,
                                               unsigned int* __restrict__ counter, double* out,
                                               unsigned long long seq, float* thr_out = nullptr,
                                               unsigned int skipped = 0u,
                                               const unsigned long long* t_start = nullptr,
                                               unsigned long long* thr_word = nullptr) {
  ReduceShared& sh = reduce_shared();
  auto& s_warp = sh.warp;
  auto& s_fin = sh.fin;
  bool& s_last = sh.last;
  float2* const pf = reinterpret_cast<float2*>(partials);
  // the slots this reduction produces
  const auto wanted = [](int slot) { return !kSigmaOnly || slot == 1 || slot == 17; };
#pragma unroll
  for (int v = 0; v < 16; ++v) {
    if (!wanted(2 + v)) continue;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[v] = __fadd_rn(acc[v], __shfl_xor_sync(kFull, acc[v], off));
  }
  if (!kSigmaOnly) c0 = __reduce_add_sync(kFull, c0);
  c1 = __reduce_add_sync(kFull, c1);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    s_warp[warp][0] = FF{static_cast<float>(c0), 0.f};
    s_warp[warp][1] = FF{static_cast<float>(c1), 0.f};
#pragma unroll
    for (int v = 0; v < 16; ++v) s_warp[warp][2 + v] = FF{acc[v], 0.f};
  }
  __syncthreads();
  // every thread of the block is past its search: a kernel launched as a
  // programmatic dependent of this one may start once all blocks are here
  if (!kPersistent) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the block's warps: 8 lanes per slot, lane w holding warp w's value
  static_assert(kThreads / 32 == 8, "one lane of an 8-lane group per warp");
  if (threadIdx.x < kTreeThreads) {
    const int v = threadIdx.x >> 3, w = threadIdx.x & 7;
    const bool mine = v < kMomentSlots && wanted(v);
    FF s = mine ? s_warp[w][v] : FF{0.f, 0.f};
    s = ff_allreduce8(s);
    if (w == 0 && mine) s_fin[0][v] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int v = 0; v < kMomentSlots; ++v)
      if (wanted(v))
        pf[static_cast<int64_t>(blockIdx.x) * kMomentSlots + v] = make_float2(s_fin[0][v].hi, s_fin[0][v].lo);
    if (skipped != 0u) atomicAdd(counter + 1, skipped);
  }
  const int r = threadIdx.x / kMomentSlots, v = threadIdx.x % kMomentSlots;
  // rows of partials the final block adds: every block's (one level) or every
  // group's sum, stored over the group's first partial (two levels)
  unsigned int rows = gridDim.x, row_stride = 1;
  if (gridDim.x > kSingleLevelBlocks) {
    const unsigned int group = blockIdx.x / kGroupBlocks, g0 = group * kGroupBlocks;
    const unsigned int in_group = min(static_cast<unsigned int>(kGroupBlocks), gridDim.x - g0);
    if (threadIdx.x == 0)
      s_last = (atom_add_release_gpu(counter + 2 + group, 1u) == in_group - 1);
    __syncthreads();
    if (!s_last) return;
    if (threadIdx.x == 0) fence_acq_rel_gpu();
    __syncthreads();
    if (threadIdx.x < kGroupBlocks * kMomentSlots && wanted(v)) {
      const float2 x = static_cast<unsigned int>(r) < in_group
                           ? __ldcg(&pf[static_cast<int64_t>(g0 + r) * kMomentSlots + v]) : make_float2(0.f, 0.f);
      s_fin[r][v] = FF{x.x, x.y};
    }
    __syncthreads();
    if (threadIdx.x < kMomentSlots && wanted(threadIdx.x)) {
      FF s{0.f, 0.f};
      for (unsigned int k = 0; k < in_group; ++k) s = ff_add(s, s_fin[k][threadIdx.x]);
      s_warp[0][threadIdx.x] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
#pragma unroll
      for (int u = 0; u < kMomentSlots; ++u)
        if (wanted(u))
          pf[static_cast<int64_t>(g0) * kMomentSlots + u] = make_float2(s_warp[0][u].hi, s_warp[0][u].lo);
      counter[2 + group] = 0u;  // ordered before the next level's release increment
    }
    rows = (gridDim.x + kGroupBlocks - 1) / kGroupBlocks;
    row_stride = kGroupBlocks;
  }
  if (threadIdx.x == 0)
    s_last = (atom_add_release_gpu(counter, 1u) == rows - 1);
  __syncthreads();
  if (!s_last) return;
  // the last block: thread 0 starts the reads it needs at the end (skipped
  // blocks, the pass's start time) now, so that their latency overlaps the
  // sum below
  unsigned int skips = 0u;
  unsigned long long t_cmd = 0ull;
  if (threadIdx.x == 0) {
    fence_acq_rel_gpu();
    skips = atomicExch(counter + 1, 0u);
    if (t_start != nullptr) t_cmd = __ldcg(t_start);
    counter[0] = 0u;
  }
  __syncthreads();
  // rows r, r + 28, ... added in order, two slots per 16-byte load; all of a
  // thread's (up to 14) loads in flight at once
  constexpr int kPairs = kMomentSlots / 2;
  constexpr int kBatch = 14;
  auto& s_rows = sh.rows;
  if (threadIdx.x < kRowGroups * kPairs &&
      (wanted(2 * (threadIdx.x % kPairs)) || wanted(2 * (threadIdx.x % kPairs) + 1))) {
    const int g = threadIdx.x / kPairs, vp = threadIdx.x % kPairs;
    const float4* pf4 = reinterpret_cast<const float4*>(partials);
    FF s0{0.f, 0.f}, s1{0.f, 0.f};
    for (unsigned int j = g; j < rows; j += kBatch * kRowGroups) {
      float4 x[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const unsigned int row = j + u * kRowGroups;
        x[u] = row < rows ? __ldcg(&pf4[static_cast<int64_t>(row) * row_stride * kPairs + vp])
                          : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (j + u * kRowGroups < rows) {
          s0 = ff_add(s0, FF{x[u].x, x[u].y});
          s1 = ff_add(s1, FF{x[u].z, x[u].w});
        }
      }
    }
    s_rows[g][2 * vp] = s0;
    s_rows[g][2 * vp + 1] = s1;
  }
  __syncthreads();
  // the row groups: 8 lanes per slot, lane j adding groups j, j + 8, ... in
  // order, then the 8 lanes' sums together
  if (threadIdx.x < kTreeThreads) {
    const int v = threadIdx.x >> 3, j = threadIdx.x & 7;
    const bool mine = v < kMomentSlots && wanted(v);
    FF s{0.f, 0.f};
    if (mine)
#pragma unroll
      for (int g = j; g < kRowGroups; g += 8) s = ff_add(s, s_rows[g][v]);
    s = ff_allreduce8(s);
    if (j == 0 && mine) sh.res[v] = s;
  }
  __syncthreads();
  unsigned long long* const out_words = reinterpret_cast<unsigned long long*>(out);
  // Thread 0: the abort word of a pass that gave up, the residual threshold,
  // the doubles of a device result; a published result then goes out as
  // tagged words, one 16-byte store by each of the first 19 threads, with no
  // fence (the host checks every word's tag).
  if (threadIdx.x == 0) {
    bool publish = false;
    if (skips != 0u) {
      // The abort marker has a word of its own: the pass queued behind this
      // one may give up too, and its marker must not overwrite this pass's
      // outcome, nor this marker a predecessor's published result.
      if (kPublish && skips >= kSkipTimedOut) {
        __threadfence_system();
        *reinterpret_cast<volatile unsigned long long*>(out_words + kAbortWord) = seq;
      }
    } else {
      publish = kPublish && !kSigmaOnly;
      sh.t_cmd = t_cmd;
    }
    sh.publish = publish;
    if (skips == 0u && (thr_out != nullptr || thr_word != nullptr)) {
      // the slots as doubles, as the host converts them
      const double pairs = static_cast<double>(sh.res[1].hi) + static_cast<double>(sh.res[1].lo);
      const double sum_e2 = static_cast<double>(sh.res[17].hi) + static_cast<double>(sh.res[17].lo);
      const double sigma2 = pairs > 0.0 ? sum_e2 / pairs : 0.0;
      const float thr = float_threshold_dev(9.0 * sigma2);
      if (thr_out != nullptr) *thr_out = thr;
      // release: the counters reset above are in place before any block that
      // reads this word starts the next pass's reduction.  Stored before the
      // result goes to (possibly host-mapped) `out`, so that the release does
      // not wait for those writes to cross to the host.
      if (thr_word != nullptr)
        asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(thr_word),
                     "l"((static_cast<unsigned long long>(static_cast<uint32_t>(seq)) << 32) | __float_as_uint(thr))
                     : "memory");
    }
    if (!kPublish && skips == 0u) {
#pragma unroll
      for (int v = 0; v < kMomentSlots; ++v)
        out[v] = static_cast<double>(sh.res[v].hi) + static_cast<double>(sh.res[v].lo);
    }
  }
  if (kPublish && !kSigmaOnly) {
    __syncthreads();
    const int i = threadIdx.x;
    if (sh.publish && i < kResultWords / 2) {
      const unsigned long long tag = static_cast<unsigned long long>(result_tag(seq)) << 32;
      uint32_t a, b;
      if (i < kMomentSlots) {
        a = __float_as_uint(sh.res[i].hi);
        b = __float_as_uint(sh.res[i].lo);
      } else {
        a = static_cast<uint32_t>(sh.t_cmd);
        b = t_start != nullptr ? static_cast<uint32_t>(global_ns()) : 0u;
      }
      asm volatile("st.relaxed.sys.global.v2.u64 [%0], {%1, %2};" ::"l"(out_words + 2 * i), "l"(tag | a),
                   "l"(tag | b) : "memory");
    }
  }
}

// Accumulate one accepted pair (original source s, matched target q).
//
// Precision of the sums.  Each thread adds its pairs' moments in float32, a
// warp adds its 32 lanes in a five-level float32 butterfly, and everything
// above (warps, blocks, groups) is added as float-float pairs (about 44
// significant bits, converted to double at the end).  A thread sums at most
// k = ceil(n / resident threads) pairs (1 on the 100k scene, 18 on the 2M
// source), so a float32 partial carries an error of at most
// gamma_(k+4) * sum |terms| with gamma_m = m u / (1 - m u), u = 2^-24: for
// k = 18 about 1.3e-6 of the absolute sum, which the float-float levels then
// preserve (each of their additions errs by about 2^-44 of its operands).  The centroids and H are compared with 1e-5 bounds, which this
// meets with room for the cancellation between the shifted second moments
// and the product of the means.  The distance sum (acc[15], whose mean is
// compared at 1e-6) is kept compensated per thread instead: the rounding
// error of each addition is recovered exactly (TwoSum) and carried in a
// second float, folded in before the butterfly, which leaves at most
// about (1 + gamma_5) u ~ 3.6e-7 of it.  (Doubles from the thread level up
// would cost the FP64 pipe, about 4 operations per clock per SM on this part,
// 16 values x 5 butterfly levels per lane on every pass's critical tail.)
__device__ __forceinline__ void add_compensated(float& sum, float& err, float x) {
  const float s = __fadd_rn(sum, x);
  const float xv = __fsub_rn(s, sum);
  const float sv = __fsub_rn(s, xv);
  err = __fadd_rn(err, __fadd_rn(__fsub_rn(sum, sv), __fsub_rn(x, xv)));
  sum = s;
}

__device__ __forceinline__ void add_pair(float (&acc)[16], float sx, float sy, float sz,
                                         const float4& qr, float d2, const IcpPassParams& p) {
  const float ds[3] = {__fsub_rn(sx, p.shift_s[0]), __fsub_rn(sy, p.shift_s[1]),
                       __fsub_rn(sz, p.shift_s[2])};
  const float dq[3] = {__fsub_rn(qr.x, p.shift_q[0]), __fsub_rn(qr.y, p.shift_q[1]),
                       __fsub_rn(qr.z, p.shift_q[2])};
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    acc[a] = __fadd_rn(acc[a], ds[a]);
    acc[3 + a] = __fadd_rn(acc[3 + a], dq[a]);
#pragma unroll
    for (int c = 0; c < 3; ++c) acc[6 + 3 * a + c] = __fadd_rn(acc[6 + 3 * a + c], __fmul_rn(ds[a], dq[c]));
  }
  (void)d2;
}

// p = R s + t, each row ((R_a0 s_x + R_a1 s_y) + R_a2 s_z) + t_a; rt holds R
// (row-major) then t.
__device__ __forceinline__ void transform_point(const float* rt, float sx, float sy, float sz,
                                                float (&q)[3]) {
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    float v = __fadd_rn(__fmul_rn(rt[3 * a], sx), __fmul_rn(rt[3 * a + 1], sy));
    v = __fadd_rn(v, __fmul_rn(rt[3 * a + 2], sz));
    q[a] = __fadd_rn(v, rt[9 + a]);
  }
}
__device__ __forceinline__ void transform_point(const IcpPassParams& p, float sx, float sy, float sz,
                                                float (&q)[3]) {
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    float v = __fadd_rn(__fmul_rn(p.R[3 * a], sx), __fmul_rn(p.R[3 * a + 1], sy));
    v = __fadd_rn(v, __fmul_rn(p.R[3 * a + 2], sz));
    q[a] = __fadd_rn(v, p.t[a]);
  }
}

// Polls use relaxed loads (an acquire load would invalidate the SM's L1 on
// every poll, under the feet of co-resident blocks); the poll that sees the
// awaited word is followed by one acquire fence.
__device__ __forceinline__ unsigned long long load_relaxed_sys(const unsigned long long* a) {
  unsigned long long v;
  asm volatile("ld.relaxed.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long load_relaxed_gpu(const unsigned long long* a) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}

__device__ __forceinline__ void store_release_gpu(unsigned long long* a, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(a), "l"(v) : "memory");
}

// The 12 floats of a command (16-byte aligned) in three vector loads issued
// together: one round trip instead of twelve.
template <bool kSystem>
__device__ __forceinline__ void load_rt(const float* a, float* rt) {
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    if (kSystem)
      asm volatile("ld.relaxed.sys.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(rt[4 * k]), "=f"(rt[4 * k + 1]), "=f"(rt[4 * k + 2]), "=f"(rt[4 * k + 3])
                   : "l"(a + 4 * k) : "memory");
    else
      asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(rt[4 * k]), "=f"(rt[4 * k + 1]), "=f"(rt[4 * k + 2]), "=f"(rt[4 * k + 3])
                   : "l"(a + 4 * k) : "memory");
  }
}

// One thread per block: wait until the host's command names pass `seq` (or
// gives up on it) and copy its R and t to rt.  Returns 0 (run), kSkipStopped
// or kSkipTimedOut.  The first block to arrive polls host memory, for at most
// wait_ns of global time, and forwards the outcome through the device mirror;
// the others wait on the mirror, for at most 2 * wait_ns.
__device__ __forceinline__ unsigned int await_command(const IcpPassParams& p, float* rt) {
  constexpr unsigned long long kRun = 0, kStop = 1, kTimeout = 2;
  const unsigned long long seq = p.seq, t0 = global_ns();
  CommandMirror* m = p.mirror;
  unsigned long long outcome = kTimeout;
  if (atomicMax(&m->elect, seq) < seq) {
    for (;;) {
      const unsigned long long w = load_relaxed_sys(&p.cmd->word);
      if ((w >> 1) == seq) {
        outcome = (w & 1ull) ? kStop : kRun;
        if (outcome == kRun) {
          asm volatile("fence.acq_rel.sys;" ::: "memory");
          float v[12];
          load_rt<true>(p.cmd->rt, v);
#pragma unroll
          for (int k = 0; k < 12; ++k) {
            rt[k] = v[k];
            m->rt[k] = v[k];
          }
        }
        break;
      }
      if ((w >> 1) > seq) {
        outcome = kStop;
        break;
      }
      if (global_ns() - t0 > p.wait_ns) break;
      __nanosleep(200);
    }
    store_release_gpu(&m->word, (seq << 2) | outcome);
  } else {
    for (;;) {
      const unsigned long long w = load_relaxed_gpu(&m->word);
      if ((w >> 2) >= seq) {
        outcome = (w >> 2) == seq ? (w & 3ull) : kStop;
        if (outcome == kRun) {
          asm volatile("fence.acq_rel.gpu;" ::: "memory");
          float v[12];
          load_rt<false>(m->rt, v);
#pragma unroll
          for (int k = 0; k < 12; ++k) rt[k] = v[k];
        }
        break;
      }
      if (global_ns() - t0 > 2 * p.wait_ns) break;
      __nanosleep(100);
    }
  }
  return outcome == kRun ? 0u : outcome == kStop ? kSkipStopped : kSkipTimedOut;
}

// The work of one pass for this thread: its queries (chunks of 32 consecutive
// source records per warp, see first_chunk) transformed by rt, searched,
// tested against the rejection threshold and added to the thread's moments.
// Shared by the per-pass kernel and the persistent registration kernel, so
// both compute the same bits.
template <bool kPerPoint, bool kSlot>
__device__ __forceinline__ void pass_chunks(const TreeView& tv, const float* rt, const float4* __restrict__ src,
                                            int64_t n_run, int64_t n, const IcpPassParams& p,
                                            int32_t* __restrict__ out_idx, float* __restrict__ out_d2,
                                            int32_t* __restrict__ slot_of, uint32_t* __restrict__ leaf_of,
                                            float (&acc)[16], uint32_t& n_acc, uint32_t& n_bad) {
  float d2_err = 0.f;  // compensation of the distance sum acc[15]
  for (int64_t c = first_chunk(); c * 32 < n_run; c += chunk_stride()) {
    const int64_t i = c * 32 + (threadIdx.x & 31);
    if (i >= n) continue;
    const float4 s = src[i];
    const int32_t slot = __float_as_int(s.w);
    int32_t idx = -1, matched = -1;
    float d2 = __int_as_float(0x7fc00000);
    if (!finite3(s.x, s.y, s.z)) {
      ++n_bad;
    } else {
      float q[3];
      transform_point(rt, s.x, s.y, s.z, q);
      if (finite3(q[0], q[1], q[2])) {
        // Without per-point outputs only accepted pairs matter, so the search
        // starts with the rejection radius as its best distance (the page's
        // section 4.4 fuses max_dist into the tree query): it returns the
        // exact nearest point when one lies within the radius, else nothing.
        Best b = make_best(kPerPoint ? __int_as_float(0x7f800000) : p.max_d2);
        if (leaf_of != nullptr) {
          const uint32_t prev = leaf_of[i];
          leaf_of[i] = search_from(tv, q[0], q[1], q[2], b, prev);
        } else {
          search(tv, q[0], q[1], q[2], b);
        }
        idx = b.idx() == INT_MAX ? -1 : b.idx();
        d2 = b.d2();
        if (b.idx() != INT_MAX && b.d2() <= p.max_d2) {
          ++n_acc;
          matched = static_cast<int32_t>(b.slot);
          add_pair(acc, s.x, s.y, s.z, __ldg(&tv.pts[b.slot]), b.d2(), p);
          add_compensated(acc[15], d2_err, b.d2());
        }
      }
    }
    if (kPerPoint) {
      out_idx[slot] = idx;
      out_d2[slot] = d2;
    }
    if (kSlot) slot_of[i] = matched;
  }
  acc[15] = __fadd_rn(acc[15], d2_err);
}

// Three resident blocks per SM: without the bound the command wait makes
// the register allocator settle on 64 registers and spill.
template <bool kPerPoint, bool kSlot>
__global__ void __launch_bounds__(kThreads, 3) icp_pass_kernel(
    const uint2* __restrict__ nodes, const float4* __restrict__ boxes, const float4* __restrict__ pts,
    int smem_slots, const float4* __restrict__ src, int64_t n, IcpPassParams p, double* __restrict__ partials,
    unsigned int* __restrict__ counter, double* out, int32_t* __restrict__ out_idx,
    float* __restrict__ out_d2, int32_t* __restrict__ slot_of, uint32_t* __restrict__ leaf_of) {
  extern __shared__ __align__(16) uint2 s_nodes[];
  __shared__ float s_rt[12];
  __shared__ unsigned int s_skip;
  resolve_shift(p);
  if (p.cmd == nullptr) {
    if (threadIdx.x == 0) {
#pragma unroll
      for (int k = 0; k < 9; ++k) s_rt[k] = p.R[k];
#pragma unroll
      for (int k = 0; k < 3; ++k) s_rt[9 + k] = p.t[k];
      s_skip = 0u;
    }
  } else if (threadIdx.x == 0) {
    s_skip = await_command(p, s_rt);
  }
  stage_top(nodes, s_nodes, smem_slots);  // ends with a block barrier
  const TreeView tv{nodes, boxes, pts, s_nodes, static_cast<uint32_t>(smem_slots)};
  const unsigned int skipped = s_skip;
  const int64_t n_run = skipped == 0u ? n : 0;
  // A pass launched as a programmatic dependent of the previous one may start
  // during that pass's tail: everything above only reads the tree and the
  // command; the warm-start hints, partials and counters below wait for the
  // previous grid to complete (a no-op for an ordinary launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");

  float acc[16];
#pragma unroll
  for (int v = 0; v < 16; ++v) acc[v] = 0.f;
  uint32_t n_acc = 0, n_bad = 0;
  pass_chunks<kPerPoint, kSlot>(tv, s_rt, src, n_run, n, p, out_idx, out_d2, slot_of, leaf_of, acc, n_acc, n_bad);
  reduce_moments<true>(acc, n_acc, n_bad, partials, counter, out, p.seq, nullptr, skipped);
}

// This thread's share of a residual pass: for each of its source records with
// a match (slot_of >= 0), the squared residual e2 of the pair under rt, with
// the search's float arithmetic; every pair is counted in n_pair and its e2
// summed in acc[15]; with kKeep, pairs with e2 <= max_d2 are counted in n_keep
// and their moments accumulated.  Shared by the residual kernel and the
// persistent registration kernel.
template <bool kKeep>
__device__ __forceinline__ void residual_chunks(const float4* __restrict__ pts, const float4* __restrict__ src,
                                                const int32_t* __restrict__ slot_of, int64_t n, const float* rt,
                                                float max_d2, const IcpPassParams& p, float (&acc)[16],
                                                uint32_t& n_keep, uint32_t& n_pair) {
  for (int64_t c = first_chunk(); c * 32 < n; c += chunk_stride()) {
    const int64_t i = c * 32 + (threadIdx.x & 31);
    if (i >= n) continue;
    const int32_t sl = slot_of[i];
    if (sl < 0) continue;
    const float4 s = src[i];
    const float4 r = __ldg(&pts[sl]);
    float q[3];
    transform_point(rt, s.x, s.y, s.z, q);
    const float e2 = dist2(r, q[0], q[1], q[2]);
    ++n_pair;
    const float sum_e2 = __fadd_rn(acc[15], e2);
    if (kKeep && e2 <= max_d2) {
      ++n_keep;
      add_pair(acc, s.x, s.y, s.z, r, 0.f, p);
    }
    acc[15] = sum_e2;
  }
}

// Residual pass of the section 4.4 rejection: for every source record with a
// match from the last correspondence pass (slot_of >= 0), the squared residual
// e2 of the pair under the transform in p (same float arithmetic as the search
// distance).  Counts every pair in c1 and sums its e2 in acc[15].  kSigmaOnly
// (the first pass): only those two sums, reduced to the 3-sigma threshold in
// *thr_out.  Otherwise pairs with e2 <= p.max_d2 (or *thr_in) are counted in c0
// and their moments accumulated in acc[0..14], and the result is published.
template <bool kSigmaOnly>
__global__ void __launch_bounds__(kThreads) residual_pass_kernel(
    const float4* __restrict__ pts, const float4* __restrict__ src, const int32_t* __restrict__ slot_of,
    int64_t n, IcpPassParams p, double* __restrict__ partials, unsigned int* __restrict__ counter,
    double* out, const float* thr_in, float* thr_out) {
  resolve_shift(p);
  if (thr_in != nullptr) p.max_d2 = *thr_in;  // written by the previous pass on this stream
  float rt[12];
#pragma unroll
  for (int k = 0; k < 9; ++k) rt[k] = p.R[k];
#pragma unroll
  for (int k = 0; k < 3; ++k) rt[9 + k] = p.t[k];
  float acc[16];
#pragma unroll
  for (int v = 0; v < 16; ++v) acc[v] = 0.f;
  uint32_t n_keep = 0, n_pair = 0;
  residual_chunks<!kSigmaOnly>(pts, src, slot_of, n, rt, p.max_d2, p, acc, n_keep, n_pair);
  reduce_moments<true, false, kSigmaOnly>(acc, n_keep, n_pair, partials, counter, out, p.seq, thr_out);
}

// ------------------------------------------------ persistent registration

__device__ __forceinline__ void store_relaxed_gpu(unsigned long long* a, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(a), "l"(v) : "memory");
}

// Tag of a command's words: the pass's sequence number and the command's kind,
// with the top bit set so that zeroed memory never carries a valid tag.
__device__ __forceinline__ uint32_t command_tag(unsigned long long seq, unsigned long long kind) {
  return static_cast<uint32_t>((seq << 2) | kind) | 0x80000000u;
}

// Read the 12 tagged words at `a` into rt (all six 16-byte loads in flight at
// once).  Returns the kind of command they name for pass seq (kCmdPass or
// kCmdResidual) when all twelve carry that one tag, else -1.
template <bool kSystem>
__device__ __forceinline__ int load_tagged(const unsigned long long* a, unsigned long long seq, float* rt) {
  unsigned long long w[12];
#pragma unroll
  for (int k = 0; k < 6; ++k) {
    if (kSystem)
      asm volatile("ld.relaxed.sys.global.v2.u64 {%0, %1}, [%2];" : "=l"(w[2 * k]), "=l"(w[2 * k + 1]) : "l"(a + 2 * k) : "memory");
    else
      asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(w[2 * k]), "=l"(w[2 * k + 1]) : "l"(a + 2 * k) : "memory");
  }
  const uint32_t t0 = static_cast<uint32_t>(w[0] >> 32);
  bool same = true;
#pragma unroll
  for (int k = 0; k < 12; ++k) {
    same = same && static_cast<uint32_t>(w[k] >> 32) == t0;
    rt[k] = __uint_as_float(static_cast<uint32_t>(w[k]));
  }
  if (!same) return -1;
  if (t0 == command_tag(seq, kCmdPass)) return static_cast<int>(kCmdPass);
  if (t0 == command_tag(seq, kCmdResidual)) return static_cast<int>(kCmdResidual);
  return -1;
}

// One thread per block: wait until the tagged command names pass `seq` and
// copy its R and t to rt.  Returns kRunPass, kRunResidual, kSkipStopped
// (stop, or a later pass named) or kSkipTimedOut.  The first block to arrive
// polls host memory for at most wait_ns, reading the control word and the
// tagged payload together (one round trip over the CPU link per poll), and
// forwards what it found through the mirror as (seq << 3) | code (codes: the
// host's kinds, or 3 = gave up); the others poll the mirror's control word
// for at most 2 * wait_ns, then read its payload.  No acquire fence: a reader
// accepts the payload once all its tags name the pass and the kind.
constexpr unsigned int kRunPass = 0u, kRunResidual = 2u;
__device__ __forceinline__ unsigned int await_tagged(const TaggedCommand* cmd, TaggedMirror* m,
                                                     unsigned long long seq, unsigned long long wait_ns,
                                                     float* rt) {
  constexpr unsigned long long kRun = kCmdPass, kStop = kCmdStop, kResidual = kCmdResidual, kTimeout = 3;
  const uint32_t tag = static_cast<uint32_t>(seq);
  const unsigned long long t0 = global_ns();
  unsigned long long outcome = kTimeout;
  if (atomicMax(&m->elect, seq) < seq) {
    for (;;) {
      const unsigned long long c = load_relaxed_sys(&cmd->ctrl);
      const int kind = load_tagged<true>(cmd->words, seq, rt);
      const uint32_t ctag = static_cast<uint32_t>(c >> 2);
      if (static_cast<int32_t>(ctag - tag) > 0 || (ctag == tag && (c & 3ull) == kStop)) {
        outcome = kStop;
        break;
      }
      if (kind >= 0) {
        outcome = static_cast<unsigned long long>(kind);
        break;
      }
      if (global_ns() - t0 > wait_ns) break;
      __nanosleep(20);
    }
    if (outcome == kRun || outcome == kResidual) {
      const unsigned long long high = static_cast<unsigned long long>(command_tag(seq, outcome)) << 32;
#pragma unroll
      for (int k = 0; k < 12; ++k) store_relaxed_gpu(&m->words[k], high | __float_as_uint(rt[k]));
    }
    store_relaxed_gpu(&m->t_cmd, global_ns());
    store_relaxed_gpu(&m->ctrl, (seq << 3) | outcome);
  } else {
    // The other blocks poll the control word alone (many of them wait while
    // the last blocks of the previous pass still search), then read the payload.
    for (;;) {
      const unsigned long long c = load_relaxed_gpu(&m->ctrl);
      if ((c >> 3) >= seq) {
        outcome = (c >> 3) == seq ? (c & 7ull) : kStop;
        if (outcome == kRun || outcome == kResidual) {
          while (load_tagged<false>(m->words, seq, rt) != static_cast<int>(outcome)) {
            if (global_ns() - t0 > 2 * wait_ns) {
              outcome = kTimeout;
              break;
            }
          }
        }
        break;
      }
      if (global_ns() - t0 > 2 * wait_ns) break;
      __nanosleep(100);
    }
  }
  return outcome == kRun ? kRunPass : outcome == kResidual ? kRunResidual
                                   : outcome == kStop ? kSkipStopped : kSkipTimedOut;
}

// Every block of the persistent kernel: wait (thread 0, bounded) until the
// residual threshold of pass `seq` has been stored -- one 64-bit word, the
// pass's tag above the float's bits -- and copy it to *out.
__device__ __forceinline__ bool await_threshold(const unsigned long long* word, unsigned long long seq,
                                                unsigned long long wait_ns, float* out) {
  const uint32_t tag = static_cast<uint32_t>(seq);
  const unsigned long long t0 = global_ns();
  for (;;) {
    const unsigned long long w = load_relaxed_gpu(word);
    if (static_cast<uint32_t>(w >> 32) == tag) {
      *out = __uint_as_float(static_cast<uint32_t>(w));
      return true;
    }
    if (global_ns() - t0 > 2 * wait_ns) return false;
    __nanosleep(32);
  }
}

// kSlot: the registration uses the residual rejection -- correspondence
// passes record each source record's matched slot, and a residual command
// runs the two residual passes of the iteration back to back: A (sums e2
// under the command's transform and stores the 3-sigma threshold as a tagged
// word in thr_word; nothing crosses to the host), then, once every block has
// read that threshold, B (the kept pairs' moments, with the pair count and the
// sum of e2 that A reduced, published with seq + 1).  A residual command thus
// uses two sequence numbers; a block that gives up waiting records it in the
// abort word.
template <bool kSlot>
__global__ void __launch_bounds__(kThreads, 3) icp_registration_kernel(
    const uint2* __restrict__ nodes, const float4* __restrict__ boxes, const float4* __restrict__ pts,
    int smem_slots, const float4* __restrict__ src, int64_t n, IcpPassParams p, const TaggedCommand* cmd,
    TaggedMirror* mirror, double* __restrict__ partials, unsigned int* __restrict__ counter, double* out,
    unsigned long long* thr_word, int32_t* __restrict__ slot_of,
    uint32_t* __restrict__ leaf_of) {
  extern __shared__ __align__(16) uint2 s_nodes[];
  __shared__ float s_rt[12];
  __shared__ float s_thr;
  __shared__ unsigned int s_skip;
  resolve_shift(p);
  stage_top(nodes, s_nodes, smem_slots);  // once for the whole registration
  const TreeView tv{nodes, boxes, pts, s_nodes, static_cast<uint32_t>(smem_slots)};
  for (unsigned long long seq = p.seq;;) {
    if (threadIdx.x == 0) s_skip = await_tagged(cmd, mirror, seq, p.wait_ns, s_rt);
    __syncthreads();
    const unsigned int code = s_skip;
    if (code == kSkipStopped) return;
    float acc[16];
#pragma unroll
    for (int v = 0; v < 16; ++v) acc[v] = 0.f;
    if (kSlot && code == kRunResidual) {
      uint32_t n_keep = 0, n_pair = 0;
      residual_chunks<false>(pts, src, slot_of, n, s_rt, 0.f, p, acc, n_keep, n_pair);
      reduce_moments<true, true, true>(acc, n_keep, n_pair, partials, counter, out, seq, nullptr, 0u,
                                       nullptr, thr_word);
      if (threadIdx.x == 0) s_skip = await_threshold(thr_word, seq, p.wait_ns, &s_thr) ? 0u : kSkipTimedOut;
      __syncthreads();
      const unsigned int skipped = s_skip;
#pragma unroll
      for (int v = 0; v < 16; ++v) acc[v] = 0.f;
      n_keep = n_pair = 0;
      if (skipped == 0u) residual_chunks<true>(pts, src, slot_of, n, s_rt, s_thr, p, acc, n_keep, n_pair);
      reduce_moments<true, true>(acc, n_keep, n_pair, partials, counter, out, seq + 1, nullptr, skipped,
                                 &mirror->t_cmd);
      if (skipped != 0u) return;
      seq += 2;
    } else {
      const unsigned int skipped = code == kRunPass ? 0u : kSkipTimedOut;
      uint32_t n_acc = 0, n_bad = 0;
      if (skipped == 0u)
        pass_chunks<false, kSlot>(tv, s_rt, src, n, n, p, nullptr, nullptr, slot_of, leaf_of, acc, n_acc, n_bad);
      reduce_moments<true, true>(acc, n_acc, n_bad, partials, counter, out, seq, nullptr, skipped,
                                 &mirror->t_cmd);
      if (skipped != 0u) return;  // gave up waiting: the pass reports its abort, this block leaves
      seq += 1;
    }
    __syncthreads();  // s_rt, s_thr and s_skip are rewritten for the next command
  }
}

inline int smem_slots_for(const icpnn_tree& t) {
  return static_cast<int>(std::min<int64_t>(t.heap_slots, kSmemSlots));
}

}  // namespace

// ------------------------------------------------------------ launchers --

void decode_bbox(const int32_t bbox6[6], float lo[3], float hi[3]) {
  for (int d = 0; d < 3; ++d) {
    const int32_t a = ordered_from_bits(bbox6[d]);
    const int32_t b = ordered_from_bits(bbox6[3 + d]);
    std::memcpy(&lo[d], &a, sizeof(float));
    std::memcpy(&hi[d], &b, sizeof(float));
    if (bbox6[d] == INT_MAX || bbox6[3 + d] == INT_MIN) lo[d] = hi[d] = 0.f;
  }
}

cudaError_t launch_bbox(const float* xyz, int64_t n, int32_t* bbox6, cudaStream_t s) {
  bbox_init_kernel<<<1, 32, 0, s>>>(bbox6);
  g_launch_count.fetch_add(1, std::memory_order_relaxed);
  if (n > 0) {
    bbox_kernel<<<blocks_for(n, kThreads, 4 * num_sms()), kThreads, 0, s>>>(xyz, n, bbox6);
    g_launch_count.fetch_add(1, std::memory_order_relaxed);
  }
  return cudaGetLastError();
}

cudaError_t launch_morton(const float* xyz, int64_t n, const int32_t* bbox6, uint32_t* keys,
                          uint32_t* vals, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  morton_kernel<<<blocks_for(n, kThreads, 8 * num_sms()), kThreads, 0, s>>>(xyz, n, bbox6, keys, vals);
  g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

int64_t radix_temp_words(int64_t n) {
  const int64_t tiles = (n + kSortTile - 1) / kSortTile;
  return std::max<int64_t>(1, tiles) * kRadix + kRadix;
}

cudaError_t radix_sort(uint32_t* keys, uint32_t* vals, uint32_t* keys_alt, uint32_t* vals_alt,
                       uint32_t* temp, int64_t n, int lo_bit, int hi_bit, cudaStream_t s,
                       uint32_t** sorted_vals, int segments) {
  *sorted_vals = vals;
  if (n <= 1) return cudaSuccess;
  const int tiles = static_cast<int>((n + kSortTile - 1) / kSortTile);
  uint32_t* hist = temp;
  uint32_t* digit_total = temp + static_cast<int64_t>(tiles) * kRadix;
  uint32_t *ki = keys, *vi = vals, *ko = keys_alt, *vo = vals_alt;
  for (int shift = lo_bit; shift < hi_bit; shift += kRadixBits) {
    radix_hist_kernel<<<dim3(tiles, segments), kThreads, 0, s>>>(ki, n, shift, hist, tiles);
    digit_row_scan_kernel<<<dim3(kRadix, segments), kThreads, 0, s>>>(hist, tiles, digit_total);
    radix_scatter_kernel<<<dim3(tiles, segments), kThreads, 0, s>>>(ki, vi, ko, vo, n, shift, hist, digit_total,
                                                                     tiles);
    g_launch_count.fetch_add(3, std::memory_order_relaxed);
    std::swap(ki, ko);
    std::swap(vi, vo);
  }
  *sorted_vals = vi;
  return cudaGetLastError();
}

cudaError_t launch_gather(const float* xyz, int64_t n, const uint32_t* perm, float4* records,
                          cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  gather_kernel<<<blocks_for(n, kThreads, 8 * num_sms()), kThreads, 0, s>>>(xyz, n, perm, records);
  g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

cudaError_t launch_nn(const icpnn_tree& t, const float4* queries, int64_t n, int32_t* idx,
                      float* dist2, uint32_t* chunk_counter, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const cudaError_t ze = cudaMemsetAsync(chunk_counter, 0, sizeof(uint32_t), s);
  if (ze != cudaSuccess) return ze;
  const int slots = smem_slots_for(t);
  const size_t smem = static_cast<size_t>(slots) * sizeof(uint2);
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, nn_kernel, kThreads, smem);
  const int grid = blocks_for(n, kThreads, std::max(1, per_sm) * num_sms());
  nn_kernel<<<grid, kThreads, smem, s>>>(reinterpret_cast<const uint2*>(t.dev.nodes),
                                          reinterpret_cast<const float4*>(t.dev.boxes),
                                          reinterpret_cast<const float4*>(t.dev.points), slots,
                                          queries, n, idx, dist2, chunk_counter);
  g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

int icp_pass_grid(const icpnn_tree& t, int64_t n) {
  const size_t smem = static_cast<size_t>(smem_slots_for(t)) * sizeof(uint2);
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, icp_pass_kernel<false, false>, kThreads, smem);
  return blocks_for(n, kThreads, std::max(1, per_sm) * num_sms());
}

cudaError_t launch_icp_pass(const icpnn_tree& t, const float4* src, int64_t n,
                            const IcpPassParams& p, double* partials, uint32_t* counter,
                            double* out, int32_t* idx, float* dist2, int32_t* slot_of,
                            uint32_t* leaf_of, int grid, cudaStream_t s) {
  const int slots = smem_slots_for(t);
  const uint2* nodes = reinterpret_cast<const uint2*>(t.dev.nodes);
  const float4* boxes = reinterpret_cast<const float4*>(t.dev.boxes);
  const float4* pts = reinterpret_cast<const float4*>(t.dev.points);
  const bool per_point = idx != nullptr || dist2 != nullptr;
  auto kernel = per_point ? (slot_of != nullptr ? icp_pass_kernel<true, true> : icp_pass_kernel<true, false>)
                          : (slot_of != nullptr ? icp_pass_kernel<false, true> : icp_pass_kernel<false, false>);
  // A pass that waits for its command is launched as a programmatic
  // dependent: its blocks may become resident once every block of the
  // previous kernel on the stream has finished its search.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(slots) * sizeof(uint2);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = p.cmd != nullptr ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, nodes, boxes, pts, slots, src, n, p, partials, counter,
                                           out, idx, dist2, slot_of, leaf_of);
  g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e != cudaSuccess ? e : cudaGetLastError();
}

bool registration_kernel_fits(const icpnn_tree& t, int grid) {
  const size_t smem = static_cast<size_t>(smem_slots_for(t)) * sizeof(uint2);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, icp_registration_kernel<false>, kThreads, smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  int per_sm_slot = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_slot, icp_registration_kernel<true>, kThreads, smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return static_cast<int64_t>(std::min(per_sm, per_sm_slot)) * num_sms() >= grid;
}

cudaError_t launch_registration(const icpnn_tree& t, const float4* src, int64_t n, const IcpPassParams& p,
                                const TaggedCommand* cmd, TaggedMirror* mirror, double* partials,
                                uint32_t* counter, double* out, unsigned long long* thr_word,
                                int32_t* slot_of, uint32_t* leaf_of, int grid, cudaStream_t s) {
  const int slots = smem_slots_for(t);
  const uint2* nodes = reinterpret_cast<const uint2*>(t.dev.nodes);
  const float4* boxes = reinterpret_cast<const float4*>(t.dev.boxes);
  const float4* pts = reinterpret_cast<const float4*>(t.dev.points);
  auto kernel = slot_of != nullptr ? icp_registration_kernel<true> : icp_registration_kernel<false>;
  // every block must be resident at once: they wait for the host, which waits
  // for every block's share of each pass
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(slots) * sizeof(uint2);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, nodes, boxes, pts, slots, src, n, p, cmd, mirror,
                                           partials, counter, out, thr_word, slot_of, leaf_of);
  if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_residual_pass(const icpnn_tree& t, const float4* src, const int32_t* slot_of,
                                 int64_t n, const IcpPassParams& p, double* partials,
                                 uint32_t* counter, double* out, int grid, cudaStream_t s,
                                 const float* thr_in, float* thr_out) {
  auto kernel = thr_out != nullptr ? residual_pass_kernel<true> : residual_pass_kernel<false>;
  kernel<<<grid, kThreads, 0, s>>>(reinterpret_cast<const float4*>(t.dev.points), src, slot_of, n, p, partials,
                                   counter, out, thr_in, thr_out);
  g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

// Scratch words: key_lo, key_hi, vals, alt keys, alt vals, gathered hi,
// radix temp, block heads, then (8-byte aligned) the sorted 64-bit keys.
int64_t voxel_key_offset(int64_t n) {
  const int64_t blocks = (n + kThreads - 1) / kThreads;
  const int64_t w = 6 * std::max<int64_t>(n, 1) + radix_temp_words(n) + std::max<int64_t>(blocks, 1) + 64;
  return (w + 1) & ~int64_t{1};
}
int64_t voxel_scratch_words(int64_t n) { return voxel_key_offset(n) + 2 * std::max<int64_t>(n, 1); }

int voxel_downsample(const float* xyz, int64_t n, float v, float* out, int64_t* out_n, uint32_t* scratch,
                     long long* bounds, unsigned long long* total, long long* host_bounds, cudaStream_t s,
                     cudaError_t* err) {
  *err = cudaSuccess;
  *out_n = 0;
  if (n <= 0) return 0;
  const int grid = blocks_for(n, kThreads, 8 * num_sms());
  voxel_bounds_init_kernel<<<1, 32, 0, s>>>(bounds);
  voxel_bounds_kernel<<<grid, kThreads, 0, s>>>(xyz, n, v, bounds);
  g_launch_count.fetch_add(2, std::memory_order_relaxed);
  if ((*err = cudaMemcpyAsync(host_bounds, bounds, 8 * sizeof(long long), cudaMemcpyDeviceToHost, s)) != cudaSuccess) return 0;
  if ((*err = cudaStreamSynchronize(s)) != cudaSuccess) return 0;
  if (host_bounds[7] != 0) return -1;  // an index beyond +-2^40
  const int64_t m = host_bounds[6];
  if (m == 0) return 0;
  VoxelGrid g;
  g.v = v;
  unsigned long long r[3];
  for (int d = 0; d < 3; ++d) {
    g.lo[d] = host_bounds[d];
    r[d] = static_cast<unsigned long long>(host_bounds[3 + d] - host_bounds[d]) + 1ull;
  }
  g.ry = r[1];
  g.rz = r[2];
  // r < 2^41 per axis; the product must stay below 2^63 (it does unless the
  // occupied index box is astronomically large)
  const long double total_keys = static_cast<long double>(r[0]) * r[1] * r[2];
  if (total_keys >= 9.2e18L) return -1;
  g.sentinel = r[0] * r[1] * r[2];
  int bits = 0;
  while (bits < 64 && (g.sentinel >> bits) != 0) ++bits;
  uint32_t* key_lo = scratch;
  uint32_t* key_hi = scratch + n;
  uint32_t* vals = scratch + 2 * n;
  uint32_t* alt_k = scratch + 3 * n;
  uint32_t* alt_v = scratch + 4 * n;
  uint32_t* gath = scratch + 5 * n;
  uint32_t* temp = scratch + 6 * n;
  uint32_t* block_heads = temp + radix_temp_words(n);
  unsigned long long* skey = reinterpret_cast<unsigned long long*>(scratch + voxel_key_offset(n));
  voxel_keys_kernel<<<grid, kThreads, 0, s>>>(xyz, n, g, key_lo, bits > 32 ? key_hi : nullptr, vals);
  g_launch_count.fetch_add(1, std::memory_order_relaxed);
  uint32_t* order = nullptr;
  if ((*err = radix_sort(key_lo, vals, alt_k, alt_v, temp, n, 0, std::min(bits, 32), s, &order)) != cudaSuccess)
    return 0;
  if (bits > 32) {
    // stable LSD over the high word: sort (hi key in the current order, order)
    gather_u32_kernel<<<grid, kThreads, 0, s>>>(key_hi, order, n, gath);
    g_launch_count.fetch_add(1, std::memory_order_relaxed);
    uint32_t* other_v = order == vals ? alt_v : vals;
    uint32_t* other_k = key_lo;  // free now
    if ((*err = radix_sort(gath, order, other_k, other_v, temp, n, 0, bits - 32, s, &order)) != cudaSuccess)
      return 0;
  }
  const int blocks = static_cast<int>((m + kThreads - 1) / kThreads);
  voxel_sorted_keys_kernel<<<grid, kThreads, 0, s>>>(xyz, order, m, g, skey);
  voxel_head_count_kernel<<<blocks, kThreads, 0, s>>>(skey, m, block_heads);
  scan_one_block_kernel<<<1, kThreads, 0, s>>>(block_heads, blocks, total);
  voxel_emit_kernel<<<blocks, kThreads, 0, s>>>(xyz, order, m, skey, block_heads, out);
  g_launch_count.fetch_add(4, std::memory_order_relaxed);
  if ((*err = cudaGetLastError()) != cudaSuccess) return 0;
  unsigned long long h_total = 0;
  if ((*err = cudaMemcpyAsync(&h_total, total, sizeof(h_total), cudaMemcpyDeviceToHost, s)) != cudaSuccess) return 0;
  if ((*err = cudaStreamSynchronize(s)) != cudaSuccess) return 0;
  *out_n = static_cast<int64_t>(h_total);
  return 0;
}

// ------------------------------------------------- allocation-free pass --
// A variant of the fused ICP pass for callers that must not allocate device
// memory.  Instead of Morton-ordered records in pool memory it reads the
// caller's n x 3 source in place (one thread per point), and every piece of
// scratch it needs -- the per-block partial moments, the block counter, the
// bounding box and the final 18-double result -- lives in one file-scope
// device array.  That array is allocated when the module is loaded and stays
// resident on every GPU that loads the library until the process exits.
//
// Layout of g_noalloc_scratch, in doubles:
//   [0, kNoAllocMaxBlocks * kMomentSlots)   partial moments of each block
//   [kNoAllocResult, + kMomentSlots)         the reduced result
//   [kNoAllocCounter, + kNoAllocCounterDoubles)  the reduction's counter words
//   [kNoAllocBbox, + 3)                      six int32 bounding-box words
constexpr int64_t kNoAllocResult = static_cast<int64_t>(kNoAllocMaxBlocks) * kMomentSlots;
constexpr int64_t kNoAllocCounter = kNoAllocResult + kMomentSlots;
constexpr int64_t kNoAllocBbox = kNoAllocCounter + kNoAllocCounterDoubles;
constexpr int64_t kNoAllocDoubles = kNoAllocBbox + 3;
static_assert(static_cast<int64_t>(kNoAllocMaxBlocks) * 256 == ICPNN_NOALLOC_MAX_POINTS,
              "one thread per point, 256 threads per block");
static_assert(kNoAllocResult == noalloc_result_offset() && kNoAllocCounter == noalloc_counter_offset() &&
                  kNoAllocBbox == noalloc_bbox_offset(),
              "scratch layout shared with the host side");

static __device__ __align__(256) double g_noalloc_scratch[kNoAllocDoubles];

namespace {

template <bool kPerPoint>
__global__ void __launch_bounds__(kThreads, 3) icp_pass_inplace_kernel(
    const uint2* __restrict__ nodes, const float4* __restrict__ boxes, const float4* __restrict__ pts,
    int smem_slots, const float* __restrict__ xyz, int64_t n, IcpPassParams p, double* __restrict__ scratch,
    int32_t* __restrict__ out_idx, float* __restrict__ out_d2) {
  extern __shared__ __align__(16) uint2 s_nodes[];
  double* partials = scratch;
  double* result = scratch + kNoAllocResult;
  unsigned int* counter = reinterpret_cast<unsigned int*>(scratch + kNoAllocCounter);
  stage_top(nodes, s_nodes, smem_slots);
  const TreeView tv{nodes, boxes, pts, s_nodes, static_cast<uint32_t>(smem_slots)};

  float acc[16];
#pragma unroll
  for (int v = 0; v < 16; ++v) acc[v] = 0.f;
  uint32_t n_acc = 0, n_bad = 0;

  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) {
    const float sx = xyz[3 * i], sy = xyz[3 * i + 1], sz = xyz[3 * i + 2];
    int32_t idx = -1;
    float d2 = __int_as_float(0x7fc00000);
    if (!finite3(sx, sy, sz)) {
      ++n_bad;
    } else {
      float q[3];
      transform_point(p, sx, sy, sz, q);
      if (finite3(q[0], q[1], q[2])) {
        Best b = make_best(__int_as_float(0x7f800000));
        search(tv, q[0], q[1], q[2], b);
        idx = b.idx();
        d2 = b.d2();
        if (b.d2() <= p.max_d2) {
          ++n_acc;
          add_pair(acc, sx, sy, sz, __ldg(&pts[b.slot]), b.d2(), p);
          acc[15] = __fadd_rn(acc[15], b.d2());  // one point per thread: exact
        }
      }
    }
    if (kPerPoint) {
      out_idx[i] = idx;
      out_d2[i] = d2;
    }
  }
  reduce_moments<false>(acc, n_acc, n_bad, partials, counter, result, 0ull);
}

}  // namespace

cudaError_t noalloc_scratch(double** out) {
  // Host code cannot use the array's name as a device address: it resolves to
  // a host-side shadow.  Look up the real address once per device, with that
  // device current.
  static std::mutex mu;
  static double* addr[kNoAllocMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<double*>(p);
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_icp_pass_inplace(const icpnn_tree& t, const float* xyz, int64_t n,
                                    const IcpPassParams& p, double* scratch, int32_t* idx,
                                    float* dist2, cudaStream_t s) {
  const int slots = smem_slots_for(t);
  const size_t smem = static_cast<size_t>(slots) * sizeof(uint2);
  const int grid = static_cast<int>((n + kThreads - 1) / kThreads);
  const uint2* nodes = reinterpret_cast<const uint2*>(t.dev.nodes);
  const float4* boxes = reinterpret_cast<const float4*>(t.dev.boxes);
  const float4* pts = reinterpret_cast<const float4*>(t.dev.points);
  if (idx != nullptr)
    icp_pass_inplace_kernel<true><<<grid, kThreads, smem, s>>>(nodes, boxes, pts, slots, xyz, n, p, scratch,
                                                               idx, dist2);
  else
    icp_pass_inplace_kernel<false><<<grid, kThreads, smem, s>>>(nodes, boxes, pts, slots, xyz, n, p, scratch,
                                                                nullptr, nullptr);
  g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

}  // namespace icpnn
