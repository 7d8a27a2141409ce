// C ABI of libicpnn: argument checking, device memory, the host ICP loop of
// "Implementing ICP with CUDA-KDTree" section 3.3 with the section 4.6
// stopping rule.  The per-iteration device work is one fused kernel; the only
// per-iteration host crossing is its 18-double moment record, written by the
// kernel straight into mapped pinned memory.
#include <cuda_runtime.h>

#include <atomic>
#include <cfloat>
#include <chrono>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "icpnn_internal.h"
#include "icpnn_probe.h"
#include "kernels.cuh"

namespace icpnn {

// Scratch memory comes from the device's default stream-ordered pool.  By
// default the pool hands freed memory back to the driver at every
// synchronisation, so the next call maps it again; keep up to 1 GiB of it
// per device instead (a setting of this process's pool only).
cudaError_t pool_alloc(void** p, size_t bytes, cudaStream_t s) {
  constexpr int kMaxDev = 64;
  static std::once_flag once[kMaxDev];
  static cudaMemPool_t pools[kMaxDev];
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaMallocAsync(p, bytes, s);
  std::call_once(once[dev], [dev] {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    uint64_t keep = uint64_t{1} << 30;
    int off = 0;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    cudaMemPoolSetAttribute(pool, cudaMemPoolReuseAllowOpportunistic, &off);
    cudaMemPoolSetAttribute(pool, cudaMemPoolReuseAllowInternalDependencies, &off);
    cudaGetLastError();
    pools[dev] = pool;
  });
  if (pools[dev] == nullptr) return cudaMallocAsync(p, bytes, s);  // no pool of our own: the device's default
  return cudaMallocFromPoolAsync(p, bytes, pools[dev], s);
}

extern std::atomic<int64_t> g_launch_count;

namespace {
thread_local std::string tl_error;
}

int fail(int code, const std::string& msg) {
  tl_error = msg;
  return code;
}
void clear_error() { tl_error.clear(); }

namespace {

#define ICPNN_CUDA(call)                                                              \
  do {                                                                                \
    cudaError_t e_ = (call);                                                          \
    if (e_ != cudaSuccess) {                                                          \
      if (e_ == cudaErrorMemoryAllocation) {                                          \
        cudaGetLastError();                                                           \
        return fail(ICPNN_ERR_NO_MEMORY, std::string(#call) + ": " + cudaGetErrorString(e_)); \
      }                                                                               \
      return fail(ICPNN_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
    }                                                                                 \
  } while (0)

bool is_device_pointer(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// Device memory that the current device's kernels may read and write:
// allocated on that device (or managed memory).
bool is_current_device_pointer(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeManaged) return true;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice && a.device == cur;
}

// Device allocations from the stream-ordered pool, returned on the same stream.
class Scratch {
 public:
  explicit Scratch(cudaStream_t s) : s_(s) {}
  ~Scratch() {
    for (void* p : ptrs_) cudaFreeAsync(p, s_);
  }
  template <typename T>
  cudaError_t alloc(T** out, int64_t count) {
    void* p = nullptr;
    const size_t bytes = static_cast<size_t>(std::max<int64_t>(count, 1)) * sizeof(T);
    cudaError_t e = pool_alloc(&p, bytes, s_);
    if (e != cudaSuccess) return e;
    ptrs_.push_back(p);
    *out = static_cast<T*>(p);
    return cudaSuccess;
  }

 private:
  cudaStream_t s_;
  std::vector<void*> ptrs_;
};

// Per-thread pinned, device-mapped buffer for the per-pass moment record and
// other small device->host results.  Kept for the life of the thread.
struct MappedBuffer {
  double* host = nullptr;
  double* dev = nullptr;
  unsigned long long seq = 0;  // last sequence number handed to a pass
};
thread_local MappedBuffer tl_mapped;
// Layout, in doubles, each region on cache lines of its own:
//   [0, kAbortWord]                            a pass's result (tagged words) and its abort word
//   [kCommandOffset, + sizeof(PassCommand))    the host-written command of pre-launched passes
//   [kTaggedOffset, + sizeof(TaggedCommand))   the host-written commands of the persistent kernel
//   [kBboxOffset, + 3)                         the source's box, copied from the device (Source)
// The result is kResultWords tagged words (the 18 moments as float-float
// pairs, then the pass's start and publish times) and the abort word.
constexpr int kCommandOffset = 64;
constexpr int kTaggedOffset = 80;
constexpr int kBboxOffset = 96;  // the source's box, six ordered integers, copied from the device
constexpr int kMappedDoubles = 112;
static_assert(kCommandOffset > kAbortWord, "result words and abort word before the command block");
static_assert(kTaggedOffset * sizeof(double) >= kCommandOffset * sizeof(double) + sizeof(PassCommand) &&
                  kTaggedOffset * sizeof(double) + sizeof(TaggedCommand) <= kMappedDoubles * sizeof(double) &&
                  (kTaggedOffset * sizeof(double)) % 16 == 0,
              "tagged command block must fit the mapped buffer after the pass command");
static_assert(kTaggedOffset * sizeof(double) + sizeof(TaggedCommand) <= kBboxOffset * sizeof(double) &&
                  kBboxOffset + 3 <= kMappedDoubles,
              "the source box's copy must fit after the tagged command");
static_assert(kCommandOffset * sizeof(double) + sizeof(PassCommand) <= kMappedDoubles * sizeof(double),
              "command block must fit the mapped buffer");

int mapped_buffer(MappedBuffer** out) {
  if (tl_mapped.host == nullptr) {
    void* h = nullptr;
    ICPNN_CUDA(cudaHostAlloc(&h, kMappedDoubles * sizeof(double),
                             cudaHostAllocMapped | cudaHostAllocPortable));
    void* d = nullptr;
    const cudaError_t e = cudaHostGetDevicePointer(&d, h, 0);
    if (e != cudaSuccess) {
      cudaFreeHost(h);
      return fail(ICPNN_ERR_CUDA, std::string("cudaHostGetDevicePointer: ") + cudaGetErrorString(e));
    }
    std::memset(h, 0, kMappedDoubles * sizeof(double));
    tl_mapped.host = static_cast<double*>(h);
    tl_mapped.dev = static_cast<double*>(d);
  }
  *out = &tl_mapped;
  return ICPNN_OK;
}

int wait_tree_ready(const icpnn_tree* t, cudaStream_t s);

int check_tree_on_device(const icpnn_tree* t) {
  if (t == nullptr) return fail(ICPNN_ERR_INVALID_ARG, "tree is NULL");
  if (t->dev.nodes == nullptr) return fail(ICPNN_ERR_NOT_UPLOADED, "tree has not been uploaded");
  int cur = -1;
  ICPNN_CUDA(cudaGetDevice(&cur));
  if (cur != t->dev.device)
    return fail(ICPNN_ERR_NOT_UPLOADED, "tree was uploaded to device " + std::to_string(t->dev.device) +
                                            ", current device is " + std::to_string(cur));
  return ICPNN_OK;
}

// Largest float f such that, for every float d, d <= f exactly when
// double(d) <= limit (limit >= 0; +inf -> +inf).
float float_threshold(double limit) {
  if (std::isinf(limit)) return INFINITY;
  if (limit >= static_cast<double>(FLT_MAX)) return FLT_MAX;
  float f = static_cast<float>(limit);
  if (static_cast<double>(f) > limit) f = std::nextafter(f, -INFINITY);
  return f;
}

// Threshold for the maximum-correspondence-distance test: accept iff
// double(d2) <= dmax^2.  No rejection (dmax <= 0 or infinite) -> +inf.
float rejection_threshold(double dmax) {
  if (!(dmax > 0.0) || std::isinf(dmax)) return INFINITY;
  return float_threshold(dmax * dmax);
}

// The source in Morton order as float4 records, plus the float32 centre of
// its bounding box (the shift c_s of the moment sums).  The box is computed on
// the device; the kernels take the centre from it there (bbox6), and the host
// reads its copy in mapped memory only when it first decodes a pass's result
// (shift()), by which time the copy, queued before every pass, has landed.
struct Source {
  float4* recs = nullptr;
  const int32_t* bbox6 = nullptr;                     // device, null without a shift
  const volatile int32_t* bbox6_host = nullptr;       // mapped copy of bbox6
  mutable float shift_[3] = {0, 0, 0};
  mutable bool shift_ready = true;
  const float* shift() const {
    if (!shift_ready) {
      std::atomic_thread_fence(std::memory_order_acquire);
      int32_t h6[6];
      for (int k = 0; k < 6; ++k) h6[k] = bbox6_host[k];
      float lo[3], hi[3];
      decode_bbox(h6, lo, hi);
      for (int d = 0; d < 3; ++d) shift_[d] = 0.5f * (lo[d] + hi[d]);
      shift_ready = true;
    }
    return shift_;
  }
};

int prepare_source(const float* xyz, int64_t n, bool morton, bool want_shift, cudaStream_t s,
                   Scratch& sc, Source* out) {
  const float* d_xyz = xyz;
  if (!is_device_pointer(xyz)) {
    float* tmp = nullptr;
    ICPNN_CUDA(sc.alloc(&tmp, 3 * n));
    ICPNN_CUDA(cudaMemcpyAsync(tmp, xyz, static_cast<size_t>(n) * 3 * sizeof(float),
                               cudaMemcpyHostToDevice, s));
    d_xyz = tmp;
  }
  ICPNN_CUDA(sc.alloc(&out->recs, n));
  const uint32_t* perm = nullptr;
  int32_t* bbox6 = nullptr;
  if (morton || want_shift) {
    ICPNN_CUDA(sc.alloc(&bbox6, 6));
    ICPNN_CUDA(launch_bbox(d_xyz, n, bbox6, s));
  }
  if (morton && n > 1) {
    uint32_t *keys, *vals, *keys2, *vals2, *temp, *sorted;
    ICPNN_CUDA(sc.alloc(&keys, n));
    ICPNN_CUDA(sc.alloc(&vals, n));
    ICPNN_CUDA(sc.alloc(&keys2, n));
    ICPNN_CUDA(sc.alloc(&vals2, n));
    ICPNN_CUDA(sc.alloc(&temp, radix_temp_words(n)));
    ICPNN_CUDA(launch_morton(d_xyz, n, bbox6, keys, vals, s));
    // bits 6..29 of the 30-bit code: cells of 1/256 of the box per axis,
    // ample for warp coherence, in three 8-bit passes (stable, so points of
    // one cell keep their input order)
    ICPNN_CUDA(radix_sort(keys, vals, keys2, vals2, temp, n, 6, 30, s, &sorted));
    perm = sorted;
  }
  ICPNN_CUDA(launch_gather(d_xyz, n, perm, out->recs, s));
  if (want_shift) {
    MappedBuffer* mb = nullptr;
    if (int rc = mapped_buffer(&mb)) return rc;
    int32_t* h6 = reinterpret_cast<int32_t*>(mb->host + kBboxOffset);
    ICPNN_CUDA(cudaMemcpyAsync(h6, bbox6, 6 * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    out->bbox6 = bbox6;
    out->bbox6_host = h6;
    out->shift_ready = false;
  }
  return ICPNN_OK;
}

void decode_moments(const double raw[kMomentSlots], const float cs[3], const float cq[3],
                    icpnn_moments* m) {
  const double N = raw[0];
  m->n_accepted = static_cast<int64_t>(N);
  m->n_nonfinite = static_cast<int64_t>(raw[1]);
  m->sum_d2 = raw[17];
  if (N > 0) {
    for (int a = 0; a < 3; ++a) {
      m->mu_src[a] = static_cast<double>(cs[a]) + raw[2 + a] / N;
      m->mu_tgt[a] = static_cast<double>(cq[a]) + raw[5 + a] / N;
    }
    for (int a = 0; a < 3; ++a)
      for (int b = 0; b < 3; ++b) m->H[3 * a + b] = raw[8 + 3 * a + b] - raw[2 + a] * raw[5 + b] / N;
    m->mse = raw[17] / N;
  } else {
    for (int a = 0; a < 3; ++a) m->mu_src[a] = m->mu_tgt[a] = NAN;
    for (int k = 0; k < 9; ++k) m->H[k] = 0.0;
    m->mse = NAN;
  }
}

// Per-point outputs of a pass or query: the caller's device buffers, or
// staging buffers copied back to the caller's host buffers.
struct PointOutputs {
  int32_t* idx = nullptr;
  float* d2 = nullptr;
  int32_t* host_idx = nullptr;
  float* host_d2 = nullptr;
};

int bind_point_outputs(int32_t* idx, float* d2, int64_t n, Scratch& sc, PointOutputs* po) {
  if (idx == nullptr) return ICPNN_OK;
  if (is_device_pointer(idx)) {
    po->idx = idx;
  } else {
    ICPNN_CUDA(sc.alloc(&po->idx, n));
    po->host_idx = idx;
  }
  if (is_device_pointer(d2)) {
    po->d2 = d2;
  } else {
    ICPNN_CUDA(sc.alloc(&po->d2, n));
    po->host_d2 = d2;
  }
  return ICPNN_OK;
}

int copy_back(const PointOutputs& po, int64_t n, cudaStream_t s) {
  if (po.host_idx)
    ICPNN_CUDA(cudaMemcpyAsync(po.host_idx, po.idx, n * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  if (po.host_d2)
    ICPNN_CUDA(cudaMemcpyAsync(po.host_d2, po.d2, n * sizeof(float), cudaMemcpyDeviceToHost, s));
  if (po.host_idx || po.host_d2) ICPNN_CUDA(cudaStreamSynchronize(s));
  return ICPNN_OK;
}

// Device state of one registration: sorted source, reduction scratch.
struct Pass {
  const icpnn_tree* tree = nullptr;
  Source src;
  int64_t n = 0;
  int grid = 0;
  double* partials = nullptr;
  uint32_t* counter = nullptr;
  CommandMirror* mirror = nullptr;  // device, zeroed: pre-launched passes' command copy
  TaggedMirror* tmirror = nullptr;  // device, zeroed: the persistent kernel's command copy
  MappedBuffer* mb = nullptr;
  int32_t* slot_of = nullptr;  // per Morton-ordered source record: matched slot or -1
  uint32_t* leaf_of = nullptr; // per source record: leaf of the last best match (warm start)
  float shift_q[3] = {0, 0, 0};
  float max_d2 = INFINITY;
  float* thr = nullptr;  // device: the 3-sigma threshold handed from one residual pass to the next
  unsigned long long* thr_word = nullptr;  // device, zeroed: the same, tagged, in the persistent kernel
};

int pass_setup(const icpnn_tree* t, const float* src, int64_t n, double dmax, bool want_slots,
               bool warm_start, cudaStream_t s, Scratch& sc, Pass* ps) {
  if (int rc = wait_tree_ready(t, s)) return rc;
  ps->tree = t;
  ps->n = n;
  if (want_slots) {
    ICPNN_CUDA(sc.alloc(&ps->slot_of, n));
    ICPNN_CUDA(sc.alloc(&ps->thr, 1));
    ICPNN_CUDA(sc.alloc(&ps->thr_word, 1));
    ICPNN_CUDA(cudaMemsetAsync(ps->thr_word, 0, sizeof(unsigned long long), s));
  }
  if (warm_start) {
    ICPNN_CUDA(sc.alloc(&ps->leaf_of, n));
    ICPNN_CUDA(cudaMemsetAsync(ps->leaf_of, 0, static_cast<size_t>(n) * sizeof(uint32_t), s));
  }
  if (int rc = prepare_source(src, n, true, true, s, sc, &ps->src)) return rc;
  ps->grid = icp_pass_grid(*t, n);
  ICPNN_CUDA(sc.alloc(&ps->partials, static_cast<int64_t>(ps->grid) * kMomentSlots));
  const int64_t counter_words = reduction_counter_words(ps->grid);
  ICPNN_CUDA(sc.alloc(&ps->counter, counter_words));
  ICPNN_CUDA(cudaMemsetAsync(ps->counter, 0, static_cast<size_t>(counter_words) * sizeof(uint32_t), s));
  ICPNN_CUDA(sc.alloc(&ps->mirror, 1));
  ICPNN_CUDA(cudaMemsetAsync(ps->mirror, 0, sizeof(CommandMirror), s));
  ICPNN_CUDA(sc.alloc(&ps->tmirror, 1));
  ICPNN_CUDA(cudaMemsetAsync(ps->tmirror, 0, sizeof(TaggedMirror), s));
  if (int rc = mapped_buffer(&ps->mb)) return rc;
  for (int d = 0; d < 3; ++d) ps->shift_q[d] = 0.5f * (t->bbox_lo[d] + t->bbox_hi[d]);
  ps->max_d2 = rejection_threshold(dmax);
  return ICPNN_OK;
}

// Pass `seq`'s result is complete in the mapped words w: every word carries
// the pass's tag (the device stores them with no fence, in any order).  A
// pass that publishes rewrites all the words, so a word is at most one
// published pass stale, and the tag's 31 bits of sequence number tell the two
// apart however long the thread keeps registering.
bool result_published(const volatile unsigned long long* w, unsigned long long seq) {
  const uint32_t tag = result_tag(seq);
  if (static_cast<uint32_t>(w[kResultWords - 1] >> 32) != tag) return false;
  for (int i = 0; i < kResultWords - 1; ++i)
    if (static_cast<uint32_t>(w[i] >> 32) != tag) return false;
  return true;
}

const volatile unsigned long long* result_words(const MappedBuffer* mb) {
  return reinterpret_cast<const volatile unsigned long long*>(mb->host);
}

// A complete published result: the slots as doubles (double(hi) + double(lo),
// the device's own conversion) and, if asked, the pass's device time in ms
// (command seen to publish; 0 when the pass did not record it).
void decode_published(const volatile unsigned long long* w, double raw[kMomentSlots], float* ms = nullptr) {
  for (int v = 0; v < kMomentSlots; ++v) {
    const uint32_t a = static_cast<uint32_t>(w[2 * v]), b = static_cast<uint32_t>(w[2 * v + 1]);
    float hi, lo;
    std::memcpy(&hi, &a, sizeof(float));
    std::memcpy(&lo, &b, sizeof(float));
    raw[v] = static_cast<double>(hi) + static_cast<double>(lo);
  }
  if (ms != nullptr) {
    const uint32_t t0 = static_cast<uint32_t>(w[2 * kMomentSlots]);
    const uint32_t t1 = static_cast<uint32_t>(w[2 * kMomentSlots + 1]);
    *ms = static_cast<float>(static_cast<double>(t1 - t0) * 1e-6);
  }
}

// Wait until the pass with sequence number `seq` has published its result in
// mapped memory, or -- for a pre-launched pass, with `aborted` given -- until
// it is known to have given up waiting for its command.  A pass that gives up
// stores its sequence number in the abort word, so a later pass that gives up
// too (the one queued behind it, say, when launches are serialised or the
// host stalls) cannot hide this pass's outcome: an abort word at or beyond
// `seq` means that pass `seq` has finished, and its tags then tell whether it
// published.  (`abort_from`, if given, is the first sequence number whose
// abort also ends the wait: a residual command's two passes publish only the
// second's result, and either may give up.)  Bounded: the stream is queried
// every few thousand polls, so a failed or finished kernel ends the wait.
int wait_published(const MappedBuffer* mb, unsigned long long seq, cudaStream_t s, bool* aborted = nullptr,
                   unsigned long long abort_from = 0) {
  const volatile unsigned long long* w = result_words(mb);
  const volatile unsigned long long* abort_word = w + kAbortWord;
  if (abort_from == 0) abort_from = seq;
  for (uint64_t spins = 1;; ++spins) {
    if (result_published(w, seq)) break;
    if (aborted != nullptr && *abort_word >= abort_from) {
      std::atomic_thread_fence(std::memory_order_acquire);
      if (result_published(w, seq)) break;
      *aborted = true;
      return ICPNN_OK;
    }
    if ((spins & 4095u) == 0) {
      const cudaError_t e = cudaStreamQuery(s);
      if (result_published(w, seq) || (aborted != nullptr && *abort_word >= abort_from)) continue;
      if (e == cudaSuccess) return fail(ICPNN_ERR_CUDA, "ICP pass finished without publishing its result");
      if (e != cudaErrorNotReady) return fail(ICPNN_ERR_CUDA, std::string("ICP pass: ") + cudaGetErrorString(e));
    }
  }
  std::atomic_thread_fence(std::memory_order_acquire);
  return ICPNN_OK;
}

// The moments of the result that wait_published has just seen (and, if
// asked, the pass's device time).
void read_moments(const Pass& ps, icpnn_moments* m, float* ms = nullptr) {
  double raw[kMomentSlots];
  decode_published(result_words(ps.mb), raw, ms);
  decode_moments(raw, ps.src.shift(), ps.shift_q, m);
}

IcpPassParams pass_params(const Pass& ps) {
  IcpPassParams p{};
  p.src_bbox6 = ps.src.bbox6;
  std::memcpy(p.shift_q, ps.shift_q, sizeof(p.shift_q));
  p.max_d2 = ps.max_d2;
  p.seq = ++ps.mb->seq;
  return p;
}

PassCommand* command_block(const MappedBuffer* mb, bool device) {
  return reinterpret_cast<PassCommand*>((device ? mb->dev : mb->host) + kCommandOffset);
}

// Queue a pass whose transform the host supplies later (pass_command); its
// sequence number goes to *seq.
int pass_prelaunch(const Pass& ps, cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1, unsigned long long* seq) {
  IcpPassParams p = pass_params(ps);
  p.cmd = command_block(ps.mb, true);
  p.mirror = ps.mirror;
  p.wait_ns = kCommandWaitNs;
  if (ev0) ICPNN_CUDA(cudaEventRecord(ev0, s));
  ICPNN_CUDA(launch_icp_pass(*ps.tree, ps.src.recs, ps.n, p, ps.partials, ps.counter, ps.mb->dev, nullptr,
                             nullptr, ps.slot_of, ps.leaf_of, ps.grid, s));
  if (ev1) ICPNN_CUDA(cudaEventRecord(ev1, s));
  *seq = p.seq;
  return ICPNN_OK;
}

// Host-side fault injection for tests (icpnn_probe_delay_commands): the
// calling thread's next commands are written late.
thread_local int64_t tl_cmd_skip = 0, tl_cmd_delayed = 0;
thread_local uint64_t tl_cmd_delay_ns = 0;
// ... and (icpnn_probe_delay_collect) its next reads of a pre-launched pass's
// result start late, after the successor pass has been queued.
thread_local int64_t tl_collect_skip = 0, tl_collect_delayed = 0;
thread_local uint64_t tl_collect_delay_ns = 0;

void injected_collect_delay() {
  if (tl_collect_delayed <= 0) return;
  if (tl_collect_skip > 0) {
    --tl_collect_skip;
    return;
  }
  --tl_collect_delayed;
  std::this_thread::sleep_for(std::chrono::nanoseconds(tl_collect_delay_ns));
}

// Hand pre-launched pass `seq` its transform, or (R == nullptr) tell it to
// return without work.  The values are stored before the word that names
// the pass, with release order.
void pass_command(const Pass& ps, unsigned long long seq, const float* R, const float* tr) {
  if (R != nullptr && tl_cmd_delayed > 0) {
    if (tl_cmd_skip > 0) {
      --tl_cmd_skip;
    } else {
      --tl_cmd_delayed;
      std::this_thread::sleep_for(std::chrono::nanoseconds(tl_cmd_delay_ns));
    }
  }
  PassCommand* c = command_block(ps.mb, false);
  if (R != nullptr) {
    std::memcpy(c->rt, R, 9 * sizeof(float));
    std::memcpy(c->rt + 9, tr, 3 * sizeof(float));
  }
  __atomic_store_n(&c->word, (seq << 1) | (R == nullptr ? 1ull : 0ull), __ATOMIC_RELEASE);
}

TaggedCommand* tagged_block(const MappedBuffer* mb) {
  return reinterpret_cast<TaggedCommand*>(mb->host + kTaggedOffset);
}

// Hand pass `seq` of the persistent kernel its transform (kind kCmdPass, or
// kCmdResidual for the iteration's residual passes), or (R == nullptr) tell
// the kernel to leave.  Every word carries the pass's tag; the control word
// is stored last, with release order.
void tagged_command(const MappedBuffer* mb, unsigned long long seq, const float* R, const float* tr,
                    unsigned long long kind = kCmdPass) {
  if (R != nullptr && tl_cmd_delayed > 0) {
    if (tl_cmd_skip > 0) {
      --tl_cmd_skip;
    } else {
      --tl_cmd_delayed;
      std::this_thread::sleep_for(std::chrono::nanoseconds(tl_cmd_delay_ns));
    }
  }
  TaggedCommand* c = tagged_block(mb);
  if (R != nullptr) {
    const unsigned long long high = static_cast<unsigned long long>(
                                        static_cast<uint32_t>((seq << 2) | kind) | 0x80000000u) << 32;
    for (int j = 0; j < 12; ++j) {
      uint32_t bits;
      std::memcpy(&bits, j < 9 ? &R[j] : &tr[j - 9], sizeof(bits));
      __atomic_store_n(&c->words[j], high | bits, __ATOMIC_RELAXED);
    }
  }
  __atomic_store_n(&c->ctrl, (seq << 2) | (R == nullptr ? kCmdStop : kind), __ATOMIC_RELEASE);
}

// A running persistent kernel; told to leave when the owner leaves early.
// The stop command takes a sequence number of its own: the next registration
// on this thread starts after it, so its kernel can never read this stop,
// still in the command block, as addressed to its own first pass.
struct PersistentRun {
  MappedBuffer* mb = nullptr;
  bool active = false;
  void stop() {
    if (active) tagged_command(mb, ++mb->seq, nullptr, nullptr);
    active = false;
  }
  ~PersistentRun() { stop(); }
};

// A pre-launched pass that has no transform yet; stopped when the owner
// leaves early, so that its blocks return at once.
struct PendingPass {
  const Pass* ps = nullptr;
  unsigned long long seq = 0;
  ~PendingPass() {
    if (seq != 0) pass_command(*ps, seq, nullptr, nullptr);
  }
};

int pass_run(const Pass& ps, const float R[9], const float tr[3], int32_t* idx, float* d2,
             cudaStream_t s, cudaEvent_t ev0, cudaEvent_t ev1, icpnn_moments* m) {
  IcpPassParams p = pass_params(ps);
  std::memcpy(p.R, R, sizeof(p.R));
  std::memcpy(p.t, tr, sizeof(p.t));
  if (ev0) ICPNN_CUDA(cudaEventRecord(ev0, s));
  ICPNN_CUDA(launch_icp_pass(*ps.tree, ps.src.recs, ps.n, p, ps.partials, ps.counter, ps.mb->dev,
                             idx, d2, ps.slot_of, idx == nullptr ? ps.leaf_of : nullptr, ps.grid, s));
  if (ev1) ICPNN_CUDA(cudaEventRecord(ev1, s));
  if (int rc = wait_published(ps.mb, p.seq, s)) return rc;
  read_moments(ps, m);
  return ICPNN_OK;
}

// Per-thread pool of timing events, created on first use and kept, so that
// timing a registration costs two event records per pass and nothing else
// until the elapsed times are read after the loop.
thread_local std::vector<cudaEvent_t> tl_events;

int timing_events(size_t count, cudaEvent_t** out) {
  while (tl_events.size() < count) {
    cudaEvent_t e = nullptr;
    ICPNN_CUDA(cudaEventCreate(&e));
    tl_events.push_back(e);
  }
  *out = tl_events.data();
  return ICPNN_OK;
}

// Residual rejection of one iteration (page section 4.4) under float32 (R, t),
// two passes back to back on the stream: the first sums e2 over all matched
// pairs and leaves the 3-sigma threshold in device memory, the second keeps
// the pairs within it and publishes their moments together with the pair
// count and the sum of e2 (the first pass's sums, bit for bit); the host
// waits once.  Returns sigma^2 and the kept pairs' moments.

int residual_run(const Pass& ps, const float R[9], const float tr[3], cudaStream_t s, double* sigma2,
                 icpnn_moments* kept) {
  IcpPassParams p{};
  std::memcpy(p.R, R, sizeof(p.R));
  std::memcpy(p.t, tr, sizeof(p.t));
  p.src_bbox6 = ps.src.bbox6;
  std::memcpy(p.shift_q, ps.shift_q, sizeof(p.shift_q));
  p.max_d2 = INFINITY;
  p.seq = ++ps.mb->seq;
  ICPNN_CUDA(launch_residual_pass(*ps.tree, ps.src.recs, ps.slot_of, ps.n, p, ps.partials, ps.counter,
                                  ps.mb->dev, ps.grid, s, nullptr, ps.thr));
  const unsigned long long seq_b = ++ps.mb->seq;
  p.seq = seq_b;
  ICPNN_CUDA(launch_residual_pass(*ps.tree, ps.src.recs, ps.slot_of, ps.n, p, ps.partials, ps.counter,
                                  ps.mb->dev, ps.grid, s, ps.thr, nullptr));
  if (int rc = wait_published(ps.mb, seq_b, s)) return rc;
  double raw[kMomentSlots];
  decode_published(result_words(ps.mb), raw);
  const double pairs = raw[1];
  *sigma2 = pairs > 0.0 ? raw[17] / pairs : 0.0;  // the device's threshold came from the same sums
  decode_moments(raw, ps.src.shift(), ps.shift_q, kept);
  kept->n_nonfinite = 0;
  kept->sum_d2 = 0.0;
  kept->mse = NAN;
  return ICPNN_OK;
}

void transform_to_f32(const double T[16], float R[9], float t[3]) {
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 3; ++j) R[3 * i + j] = static_cast<float>(T[4 * i + j]);
    t[i] = static_cast<float>(T[4 * i + 3]);
  }
}

// Device arrays of a tree come from the device's stream-ordered pool.  The
// release waits for all work on the device first, as cudaFree would, then
// hands the arrays back to the pool (kept for the next tree).
void release_device_tree(DeviceTree* d) {
  if (d->nodes == nullptr) return;
  int cur = -1;
  cudaGetDevice(&cur);
  cudaSetDevice(d->device);
  cudaDeviceSynchronize();  // also ends an upload still copying from the host arrays
  cudaFreeAsync(d->nodes, nullptr);
  if (d->points) cudaFreeAsync(d->points, nullptr);
  cudaStreamSynchronize(nullptr);
  if (d->ready) cudaEventDestroy(d->ready);
  cudaGetLastError();
  cudaSetDevice(cur);
  *d = DeviceTree{};
}

// Orders stream s after the tree's upload (see DeviceTree::ready).
int wait_tree_ready(const icpnn_tree* t, cudaStream_t s) {
  if (t->dev.ready != nullptr) ICPNN_CUDA(cudaStreamWaitEvent(s, t->dev.ready, 0));
  return ICPNN_OK;
}

// Host copies of a device-built tree's nodes, boxes and records, made on first
// need.
int ensure_host_copy(icpnn_tree* t) {
  if (!t->host_stale) return ICPNN_OK;
  int cur = -1;
  cudaGetDevice(&cur);
  cudaError_t e = cudaSetDevice(t->dev.device);
  try {
    t->nodes.resize(static_cast<size_t>(t->heap_slots));
    t->boxes.resize(static_cast<size_t>(8 * t->heap_slots));
    t->records.resize(static_cast<size_t>(4 * t->n));
  } catch (const std::bad_alloc&) {
    cudaSetDevice(cur);
    return fail(ICPNN_ERR_NO_MEMORY, "tree: host allocation failed");
  }
  if (e == cudaSuccess)
    e = cudaMemcpy(t->nodes.data(), t->dev.nodes, t->nodes.size() * sizeof(Node), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess)
    e = cudaMemcpy(t->boxes.data(), t->dev.boxes, t->boxes.size() * sizeof(float), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess)
    e = cudaMemcpy(t->records.data(), t->dev.points, t->records.size() * sizeof(float), cudaMemcpyDeviceToHost);
  cudaSetDevice(cur);
  if (e != cudaSuccess) return fail(ICPNN_ERR_CUDA, std::string("tree: copy to the host: ") + cudaGetErrorString(e));
  t->host_stale = false;
  return ICPNN_OK;
}

}  // namespace
}  // namespace icpnn

using namespace icpnn;

extern "C" {

int icpnn_kdtree_build(const float* xyz_host, int64_t n, int32_t leaf_size, int32_t max_depth,
                       uint32_t flags, icpnn_tree** out) {
  clear_error();
  if (out == nullptr) return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build: out is NULL");
  *out = nullptr;
  if (xyz_host == nullptr) return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build: xyz is NULL");
  if (n < 1 || n > INT32_MAX) return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build: n must be in [1, 2^31-1]");
  if (leaf_size < 1 || leaf_size > ICPNN_MAX_LEAF_SIZE)
    return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build: leaf_size must be in [1, 64]");
  if (max_depth == -1) max_depth = ICPNN_MAX_DEPTH;
  if (max_depth < 0 || max_depth > ICPNN_MAX_DEPTH)
    return fail(ICPNN_ERR_TREE_DEPTH, "kdtree_build: max_depth must be in [0, 20] or -1");
  if (flags & ~ICPNN_SPLIT_ROUND_ROBIN) return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build: unknown flag");
  icpnn_tree* t = new (std::nothrow) icpnn_tree();
  if (t == nullptr) return fail(ICPNN_ERR_NO_MEMORY, "kdtree_build: host allocation failed");
  const int rc = build_tree(xyz_host, n, leaf_size, max_depth, (flags & ICPNN_SPLIT_ROUND_ROBIN) != 0, t);
  if (rc != ICPNN_OK) {
    delete t;
    return rc;
  }
  *out = t;
  return ICPNN_OK;
}

int icpnn_kdtree_build_device(const float* xyz, int64_t n, int32_t leaf_size, int32_t max_depth,
                              uint32_t flags, icpnn_tree** out, void* stream) {
  clear_error();
  if (out == nullptr) return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build_device: out is NULL");
  *out = nullptr;
  if (xyz == nullptr) return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build_device: xyz is NULL");
  if (n < 1 || n > INT32_MAX) return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build_device: n must be in [1, 2^31-1]");
  if (leaf_size < 1 || leaf_size > ICPNN_MAX_LEAF_SIZE)
    return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build_device: leaf_size must be in [1, 64]");
  if (max_depth == -1) max_depth = ICPNN_MAX_DEPTH;
  if (max_depth < 0 || max_depth > ICPNN_MAX_DEPTH)
    return fail(ICPNN_ERR_TREE_DEPTH, "kdtree_build_device: max_depth must be in [0, 20] or -1");
  if (flags & ~ICPNN_SPLIT_ROUND_ROBIN) return fail(ICPNN_ERR_INVALID_ARG, "kdtree_build_device: unknown flag");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  icpnn_tree* t = new (std::nothrow) icpnn_tree();
  if (t == nullptr) return fail(ICPNN_ERR_NO_MEMORY, "kdtree_build_device: host allocation failed");
  int rc = ICPNN_OK;
  {
    Scratch sc(s);
    const float* d_xyz = xyz;
    if (!is_device_pointer(xyz)) {
      float* tmp = nullptr;
      cudaError_t e = sc.alloc(&tmp, 3 * n);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(tmp, xyz, static_cast<size_t>(n) * 3 * sizeof(float), cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) rc = fail(ICPNN_ERR_CUDA, std::string("kdtree_build_device: ") + cudaGetErrorString(e));
      d_xyz = tmp;
    }
    if (rc == ICPNN_OK)
      rc = build_tree_device(d_xyz, n, leaf_size, max_depth, (flags & ICPNN_SPLIT_ROUND_ROBIN) != 0, t, s);
  }
  if (rc != ICPNN_OK) {
    delete t;
    return rc;
  }
  *out = t;
  return ICPNN_OK;
}

void icpnn_kdtree_free(icpnn_tree* t) {
  if (t == nullptr) return;
  release_device_tree(&t->dev);
  delete t;
}

int icpnn_kdtree_upload(icpnn_tree* t, void* stream) {
  clear_error();
  if (t == nullptr) return fail(ICPNN_ERR_INVALID_ARG, "kdtree_upload: tree is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int cur = -1;
  ICPNN_CUDA(cudaGetDevice(&cur));
  if (t->dev.nodes != nullptr && t->dev.device == cur) return ICPNN_OK;
  if (int rc = ensure_host_copy(t)) return rc;
  release_device_tree(&t->dev);
  Node* nodes = nullptr;
  float* pts = nullptr;
  // nodes and boxes share one allocation; heap_slots >= 2 is a power of two,
  // so the boxes start 16-byte aligned
  const size_t nb = static_cast<size_t>(t->heap_slots) * sizeof(Node);
  const size_t bb = static_cast<size_t>(t->heap_slots) * 8 * sizeof(float);
  const size_t pb = static_cast<size_t>(t->n) * 4 * sizeof(float);
  cudaError_t e = pool_alloc(reinterpret_cast<void**>(&nodes), nb + bb, s);
  float* boxes = nodes ? reinterpret_cast<float*>(reinterpret_cast<char*>(nodes) + nb) : nullptr;
  if (e == cudaSuccess) e = pool_alloc(reinterpret_cast<void**>(&pts), pb, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(nodes, t->nodes.data(), nb, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(boxes, t->boxes.data(), bb, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(pts, t->records.data(), pb, cudaMemcpyHostToDevice, s);
  // The host arrays are page-locked: the copies are DMAs that run on while
  // the caller goes on; calls that use the tree wait for this event on their
  // own stream, and freeing the tree synchronises the device first.
  cudaEvent_t ready = nullptr;
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventRecord(ready, s);
  if (e != cudaSuccess) {
    if (ready) cudaEventDestroy(ready);
    cudaGetLastError();
    if (nodes) cudaFreeAsync(nodes, s);
    if (pts) cudaFreeAsync(pts, s);
    cudaStreamSynchronize(s);
    cudaGetLastError();
    return fail(e == cudaErrorMemoryAllocation ? ICPNN_ERR_NO_MEMORY : ICPNN_ERR_CUDA,
                std::string("kdtree_upload: ") + cudaGetErrorString(e));
  }
  t->dev.device = cur;
  t->dev.nodes = nodes;
  t->dev.boxes = boxes;
  t->dev.points = pts;
  t->dev.ready = ready;
  return ICPNN_OK;
}

int icpnn_kdtree_info(const icpnn_tree* t, int64_t* n_points, int32_t* leaf_size, int32_t* max_depth,
                      int32_t* depth, int64_t* n_nodes) {
  clear_error();
  if (t == nullptr) return fail(ICPNN_ERR_INVALID_ARG, "kdtree_info: tree is NULL");
  if (n_points) *n_points = t->n;
  if (leaf_size) *leaf_size = t->leaf_size;
  if (max_depth) *max_depth = t->max_depth;
  if (depth) *depth = t->depth;
  if (n_nodes) *n_nodes = t->n_nodes;
  return ICPNN_OK;
}

int icpnn_kdtree_export(const icpnn_tree* t, int64_t node_capacity, float* split_val,
                        int32_t* split_dim, int32_t* left, int32_t* right, int32_t* start,
                        int32_t* end, int32_t* leaf_index) {
  clear_error();
  if (t == nullptr || !split_val || !split_dim || !left || !right || !start || !end || !leaf_index)
    return fail(ICPNN_ERR_INVALID_ARG, "kdtree_export: NULL argument");
  if (node_capacity < t->n_nodes) return fail(ICPNN_ERR_INVALID_ARG, "kdtree_export: node_capacity too small");
  if (int rc = ensure_host_copy(const_cast<icpnn_tree*>(t))) return rc;
  // Walk the heap depth-first, left first: that numbering is the page's
  // recursion order.  Returns [start, end) of the subtree's points.
  struct Frame {
    uint64_t heap;
    int32_t pre;
    int stage;
  };
  std::vector<Frame> stack;
  int32_t next = 0;
  stack.push_back({1, next++, 0});
  while (!stack.empty()) {
    Frame& f = stack.back();
    const Node& nd = t->nodes[f.heap];
    if (node_is_leaf(nd)) {
      split_val[f.pre] = 0.0f;
      split_dim[f.pre] = -1;
      left[f.pre] = right[f.pre] = -1;
      start[f.pre] = static_cast<int32_t>(nd.a);
      end[f.pre] = static_cast<int32_t>(nd.a + (nd.meta >> 2));
      stack.pop_back();
      continue;
    }
    if (f.stage == 0) {
      std::memcpy(&split_val[f.pre], &nd.a, sizeof(float));
      split_dim[f.pre] = static_cast<int32_t>(nd.meta);
      left[f.pre] = next;
      f.stage = 1;
      const uint64_t child = 2 * f.heap;
      stack.push_back({child, next++, 0});
    } else if (f.stage == 1) {
      right[f.pre] = next;
      f.stage = 2;
      const uint64_t child = 2 * f.heap + 1;
      stack.push_back({child, next++, 0});
    } else {
      start[f.pre] = start[left[f.pre]];
      end[f.pre] = end[right[f.pre]];
      stack.pop_back();
    }
  }
  for (int64_t k = 0; k < t->n; ++k) std::memcpy(&leaf_index[k], &t->records[4 * k + 3], sizeof(int32_t));
  return ICPNN_OK;
}

int icpnn_nn_query(const icpnn_tree* t, const float* xyz, int64_t n, int32_t* idx, float* dist2,
                   uint32_t flags, void* stream) {
  clear_error();
  if (n < 0 || n > INT32_MAX) return fail(ICPNN_ERR_INVALID_ARG, "nn_query: n out of range");
  if (flags & ~ICPNN_MORTON_SORT) return fail(ICPNN_ERR_INVALID_ARG, "nn_query: unknown flag");
  if (int rc = check_tree_on_device(t)) return rc;
  if (n == 0) return ICPNN_OK;
  if (!xyz || !idx || !dist2) return fail(ICPNN_ERR_INVALID_ARG, "nn_query: NULL pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = wait_tree_ready(t, s)) return rc;
  PointOutputs po;
  {
    Scratch sc(s);
    Source src;
    if (int rc = prepare_source(xyz, n, (flags & ICPNN_MORTON_SORT) != 0, false, s, sc, &src)) return rc;
    if (int rc = bind_point_outputs(idx, dist2, n, sc, &po)) return rc;
    uint32_t* chunk_counter = nullptr;
    ICPNN_CUDA(sc.alloc(&chunk_counter, 1));
    ICPNN_CUDA(launch_nn(*t, src.recs, n, po.idx, po.d2, chunk_counter, s));
    if (int rc = copy_back(po, n, s)) return rc;
  }
  return ICPNN_OK;
}

int icpnn_icp_step(const icpnn_tree* t, const float* src, int64_t n, const float* R, const float* tr,
                   double max_corr_dist, int32_t* idx, float* dist2, icpnn_moments* out, void* stream) {
  clear_error();
  if (int rc = check_tree_on_device(t)) return rc;
  if (!src || !R || !tr || !out) return fail(ICPNN_ERR_INVALID_ARG, "icp_step: NULL pointer");
  if ((idx == nullptr) != (dist2 == nullptr))
    return fail(ICPNN_ERR_INVALID_ARG, "icp_step: idx and dist2 must both be given or both NULL");
  if (n < 1 || n > INT32_MAX) return fail(ICPNN_ERR_INVALID_ARG, "icp_step: n out of range");
  if (std::isnan(max_corr_dist)) return fail(ICPNN_ERR_INVALID_ARG, "icp_step: max_corr_dist is NaN");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Scratch sc(s);
  Pass ps;
  if (int rc = pass_setup(t, src, n, max_corr_dist, false, false, s, sc, &ps)) return rc;
  PointOutputs po;
  if (int rc = bind_point_outputs(idx, dist2, n, sc, &po)) return rc;
  if (int rc = pass_run(ps, R, tr, po.idx, po.d2, s, nullptr, nullptr, out)) return rc;
  if (int rc = copy_back(po, n, s)) return rc;
  if (out->n_nonfinite > 0)
    return fail(ICPNN_ERR_NONFINITE, "icp_step: " + std::to_string(out->n_nonfinite) +
                                         " source points have non-finite coordinates");
  return ICPNN_OK;
}

// The allocation-free pass: every buffer is the caller's or lives in the
// library's fixed device scratch array; the few bytes that come back to the
// host land in stack buffers.  No cudaMalloc / cudaFree / cudaHostAlloc,
// no stream-ordered pool, no host heap for results.
int icpnn_icp_step_noalloc(const icpnn_tree* t, const float* src, int64_t n, const float* R,
                           const float* tr, double max_corr_dist, int32_t* idx, float* dist2,
                           icpnn_moments* out, void* stream) {
  clear_error();
  if (int rc = check_tree_on_device(t)) return rc;
  if (!src || !R || !tr || !out) return fail(ICPNN_ERR_INVALID_ARG, "icp_step_noalloc: NULL pointer");
  if ((idx == nullptr) != (dist2 == nullptr))
    return fail(ICPNN_ERR_INVALID_ARG, "icp_step_noalloc: idx and dist2 must both be given or both NULL");
  if (n < 1 || n > ICPNN_NOALLOC_MAX_POINTS)
    return fail(ICPNN_ERR_INVALID_ARG,
                "icp_step_noalloc: n = " + std::to_string(n) + " is outside [1, " +
                    std::to_string(ICPNN_NOALLOC_MAX_POINTS) +
                    "], the most points its fixed scratch array can reduce; use icpnn_icp_step");
  if (std::isnan(max_corr_dist)) return fail(ICPNN_ERR_INVALID_ARG, "icp_step_noalloc: max_corr_dist is NaN");
  if (!is_current_device_pointer(src))
    return fail(ICPNN_ERR_INVALID_ARG, "icp_step_noalloc: src must be memory of the current device (a host "
                                       "buffer would need a staging allocation)");
  if (idx != nullptr && (!is_current_device_pointer(idx) || !is_current_device_pointer(dist2)))
    return fail(ICPNN_ERR_INVALID_ARG, "icp_step_noalloc: idx and dist2 must be memory of the current device");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = wait_tree_ready(t, s)) return rc;
  double* scratch = nullptr;
  ICPNN_CUDA(noalloc_scratch(&scratch));
  // the reduction's counters must start at zero; the other words are
  // written before they are read within this call
  ICPNN_CUDA(cudaMemsetAsync(scratch + noalloc_counter_offset(), 0, kNoAllocCounterDoubles * sizeof(double), s));
  int32_t* bbox6 = reinterpret_cast<int32_t*>(scratch + noalloc_bbox_offset());
  ICPNN_CUDA(launch_bbox(src, n, bbox6, s));
  int32_t h6[6];
  ICPNN_CUDA(cudaMemcpyAsync(h6, bbox6, sizeof(h6), cudaMemcpyDeviceToHost, s));
  ICPNN_CUDA(cudaStreamSynchronize(s));
  float lo[3], hi[3];
  decode_bbox(h6, lo, hi);
  IcpPassParams p{};
  std::memcpy(p.R, R, sizeof(p.R));
  std::memcpy(p.t, tr, sizeof(p.t));
  for (int d = 0; d < 3; ++d) {
    p.shift_s[d] = 0.5f * (lo[d] + hi[d]);
    p.shift_q[d] = 0.5f * (t->bbox_lo[d] + t->bbox_hi[d]);
  }
  p.max_d2 = rejection_threshold(max_corr_dist);
  ICPNN_CUDA(launch_icp_pass_inplace(*t, src, n, p, scratch, idx, dist2, s));
  double raw[kMomentSlots];
  ICPNN_CUDA(cudaMemcpyAsync(raw, scratch + noalloc_result_offset(), sizeof(raw), cudaMemcpyDeviceToHost, s));
  ICPNN_CUDA(cudaStreamSynchronize(s));
  decode_moments(raw, p.shift_s, p.shift_q, out);
  if (out->n_nonfinite > 0)
    return fail(ICPNN_ERR_NONFINITE, "icp_step_noalloc: " + std::to_string(out->n_nonfinite) +
                                         " source points have non-finite coordinates");
  return ICPNN_OK;
}

int icpnn_kabsch(const icpnn_moments* m, double* T) {
  clear_error();
  if (m == nullptr || T == nullptr) return fail(ICPNN_ERR_INVALID_ARG, "kabsch: NULL pointer");
  const int rc = kabsch_solve(*m, T);
  if (rc != ICPNN_OK) return fail(rc, "kabsch: fewer than 3 pairs or cross-covariance of rank < 2");
  return ICPNN_OK;
}

int icpnn_icp_align(const icpnn_tree* t, const float* src, int64_t n_src, int32_t max_iter, double eps,
                    double max_corr_dist, const double* init_T, double* out_T, double* final_mse,
                    int32_t* iters, int64_t* final_n_accepted, icpnn_iter_record* trace, int32_t trace_cap,
                    uint32_t flags, void* stream) {
  clear_error();
  if (int rc = check_tree_on_device(t)) return rc;
  if (!src || !out_T || !final_mse || !iters) return fail(ICPNN_ERR_INVALID_ARG, "icp_align: NULL pointer");
  if (n_src < 1 || n_src > INT32_MAX) return fail(ICPNN_ERR_INVALID_ARG, "icp_align: n_src out of range");
  if (max_iter < 1) return fail(ICPNN_ERR_INVALID_ARG, "icp_align: max_iter must be >= 1");
  if (!(eps >= 0.0)) return fail(ICPNN_ERR_INVALID_ARG, "icp_align: eps must be >= 0");
  if (std::isnan(max_corr_dist)) return fail(ICPNN_ERR_INVALID_ARG, "icp_align: max_corr_dist is NaN");
  if (trace_cap < 0 || (trace_cap > 0 && trace == nullptr))
    return fail(ICPNN_ERR_INVALID_ARG, "icp_align: bad trace buffer");
  if (flags & ~(ICPNN_TRACE_TIMING | ICPNN_RESIDUAL_REJECT | ICPNN_NO_PRELAUNCH | ICPNN_NO_PERSISTENT))
    return fail(ICPNN_ERR_INVALID_ARG, "icp_align: unknown flag");
  const bool residual = (flags & ICPNN_RESIDUAL_REJECT) != 0;
  // one-at-a-time pre-launch: the residual passes run between a pass and the
  // next one's transform, so the next pass cannot be queued ahead of them
  // (the persistent kernel runs them itself)
  bool prelaunch = !residual && (flags & ICPNN_NO_PRELAUNCH) == 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  double T[16];
  if (init_T) {
    std::memcpy(T, init_T, sizeof(T));
  } else {
    for (int k = 0; k < 16; ++k) T[k] = (k % 5 == 0) ? 1.0 : 0.0;
  }
  Scratch sc(s);
  Pass ps;
  if (int rc = pass_setup(t, src, n_src, max_corr_dist, residual, true, s, sc, &ps)) return rc;

  // Default: the whole registration as one persistent kernel; else passes
  // pre-launched one at a time (ICPNN_NO_PERSISTENT, or a grid that cannot be
  // resident at once), else ordinary launches.
  PersistentRun run;
  run.mb = ps.mb;
  if ((flags & (ICPNN_NO_PRELAUNCH | ICPNN_NO_PERSISTENT)) == 0 && registration_kernel_fits(*t, ps.grid)) {
    IcpPassParams p = pass_params(ps);
    --ps.mb->seq;  // pass_params took a number; the first pass uses it below
    p.wait_ns = kCommandWaitNs;
    const TaggedCommand* dev_cmd = reinterpret_cast<const TaggedCommand*>(ps.mb->dev + kTaggedOffset);
    const cudaError_t e = launch_registration(*ps.tree, ps.src.recs, ps.n, p, dev_cmd, ps.tmirror, ps.partials,
                                              ps.counter, ps.mb->dev, ps.thr_word, ps.slot_of, ps.leaf_of,
                                              ps.grid, s);
    if (e == cudaSuccess) {
      run.active = true;
      prelaunch = false;
    } else if (e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorNotSupported) {
      cudaGetLastError();
    } else {
      return fail(ICPNN_ERR_CUDA, std::string("icp_align: persistent kernel launch: ") + cudaGetErrorString(e));
    }
  }
  cudaEvent_t* ev = nullptr;
  const int32_t timed = (flags & ICPNN_TRACE_TIMING) ? std::min(trace_cap, max_iter) : 0;
  if (timed > 0 && !run.active)
    if (int rc = timing_events(2 * static_cast<size_t>(timed), &ev)) return rc;

  // Pre-launched passes: `cur` evaluates T; `next` is queued behind it
  // before its result is read and gets the solved transform as its command.
  unsigned long long cur = 0;
  PendingPass next{&ps, 0};
  if (prelaunch) {
    if (int rc = pass_prelaunch(ps, s, timed > 0 ? ev[0] : nullptr, timed > 0 ? ev[1] : nullptr, &cur))
      return rc;
    float R32[9], t32[3];
    transform_to_f32(T, R32, t32);
    pass_command(ps, cur, R32, t32);
  }
  // Result of pass `cur` (already commanded with transform T); queues a
  // successor first when `more` is set.  A pass whose blocks gave up waiting
  // for their transform (a profiler or debugger that serialises launches, a
  // host thread descheduled for the whole wait) is evaluated again by an
  // ordinary launch, and the registration continues with ordinary launches.
  auto collect = [&](bool more, cudaEvent_t ev0, cudaEvent_t ev1, icpnn_moments* m) -> int {
    if (more)
      if (int rc = pass_prelaunch(ps, s, ev0, ev1, &next.seq)) return rc;
    injected_collect_delay();
    bool aborted = false;
    if (int rc = wait_published(ps.mb, cur, s, &aborted)) return rc;
    if (!aborted) {
      read_moments(ps, m);
      return ICPNN_OK;
    }
    if (next.seq != 0) {
      pass_command(ps, next.seq, nullptr, nullptr);
      next.seq = 0;
    }
    prelaunch = false;
    float R32[9], t32[3];
    transform_to_f32(T, R32, t32);
    return pass_run(ps, R32, t32, nullptr, nullptr, s, nullptr, nullptr, m);
  };

  // The persistent kernel's pass under T: command, wait, read.  If the kernel
  // gave up waiting (a profiler that serialises launches, a host thread
  // descheduled for the whole wait) it is told to leave, the counters it may
  // have left behind are cleared, and the pass and the rest of the
  // registration run as ordinary launches.  *pass_ms: the pass's device time
  // (command seen to result published), 0 after a fallback.
  auto persistent_pass = [&](icpnn_moments* m, float* pass_ms) -> int {
    float R32[9], t32[3];
    transform_to_f32(T, R32, t32);
    const unsigned long long seq = ++ps.mb->seq;
    tagged_command(ps.mb, seq, R32, t32);
    injected_collect_delay();
    bool aborted = false;
    if (int rc = wait_published(ps.mb, seq, s, &aborted)) return rc;
    if (!aborted) {
      read_moments(ps, m, pass_ms);
      return ICPNN_OK;
    }
    run.stop();
    ICPNN_CUDA(cudaMemsetAsync(ps.counter, 0, static_cast<size_t>(reduction_counter_words(ps.grid)) * sizeof(uint32_t), s));
    *pass_ms = 0.f;
    return pass_run(ps, R32, t32, nullptr, nullptr, s, nullptr, nullptr, m);
  };

  // The persistent kernel's residual passes of one iteration under (R1, t1):
  // one command, the second pass's result read back (the kept pairs' moments,
  // the pair count and the sum of e2); the same fallback as persistent_pass.
  auto persistent_residual = [&](const float R1[9], const float t1[3], double* sigma2,
                                 icpnn_moments* kept, float* resid_ms) -> int {
    const unsigned long long seq_a = ++ps.mb->seq;
    const unsigned long long seq_b = ++ps.mb->seq;
    tagged_command(ps.mb, seq_a, R1, t1, kCmdResidual);
    // a kernel that gave up -- waiting for this command, or for the threshold
    // between the two passes -- records seq_a or seq_b in the abort word
    bool aborted = false;
    if (int rc = wait_published(ps.mb, seq_b, s, &aborted, seq_a)) return rc;
    if (!aborted) {
      double raw[kMomentSlots];
      // the device time from the residual command's arrival to the second
      // pass's publish
      decode_published(result_words(ps.mb), raw, resid_ms);
      const double pairs = raw[1];
      *sigma2 = pairs > 0.0 ? raw[17] / pairs : 0.0;  // the device's threshold came from the same sums
      decode_moments(raw, ps.src.shift(), ps.shift_q, kept);
      kept->n_nonfinite = 0;
      kept->sum_d2 = 0.0;
      kept->mse = NAN;
      return ICPNN_OK;
    }
    *resid_ms = 0.f;
    run.stop();
    ICPNN_CUDA(cudaMemsetAsync(ps.counter, 0, static_cast<size_t>(reduction_counter_words(ps.grid)) * sizeof(uint32_t), s));
    return residual_run(ps, R1, t1, s, sigma2, kept);
  };

  double mse_hist[3] = {0, 0, 0};
  int32_t done = 0;
  for (int32_t k = 0; k < max_iter; ++k) {
    float R32[9], t32[3];
    transform_to_f32(T, R32, t32);
    icpnn_moments m;
    float pass_ms = 0.f;
    if (run.active) {
      if (int rc = persistent_pass(&m, &pass_ms)) return rc;
    } else if (prelaunch) {
      const bool time_next = k + 1 < timed;
      if (int rc = collect(true, time_next ? ev[2 * k + 2] : nullptr, time_next ? ev[2 * k + 3] : nullptr, &m))
        return rc;
    } else {
      const bool time_it = k < timed;
      if (int rc = pass_run(ps, R32, t32, nullptr, nullptr, s, time_it ? ev[2 * k] : nullptr,
                            time_it ? ev[2 * k + 1] : nullptr, &m))
        return rc;
    }
    if (m.n_nonfinite > 0)
      return fail(ICPNN_ERR_NONFINITE, "icp_align: " + std::to_string(m.n_nonfinite) +
                                           " source points have non-finite coordinates");
    if (m.n_accepted < 3)
      return fail(ICPNN_ERR_DEGENERATE, "icp_align: fewer than 3 correspondences accepted at iteration " +
                                            std::to_string(k));
    double Tn[16];
    if (kabsch_solve(m, Tn) != ICPNN_OK)
      return fail(ICPNN_ERR_DEGENERATE, "icp_align: rank-deficient cross-covariance at iteration " +
                                            std::to_string(k));
    int64_t n_inliers = m.n_accepted;
    double sigma2 = 0.0;
    float resid_ms = 0.f;
    if (residual) {
      // page section 4.4: residuals under the first solve, 3-sigma rule, re-solve
      float R1[9], t1[3];
      transform_to_f32(Tn, R1, t1);
      icpnn_moments kept;
      if (run.active) {
        if (int rc = persistent_residual(R1, t1, &sigma2, &kept, &resid_ms)) return rc;
      } else {
        if (int rc = residual_run(ps, R1, t1, s, &sigma2, &kept)) return rc;
      }
      n_inliers = kept.n_accepted;
      if (n_inliers < 3 || kabsch_solve(kept, Tn) != ICPNN_OK)
        return fail(ICPNN_ERR_DEGENERATE, "icp_align: residual rejection left a degenerate pair set at "
                                          "iteration " + std::to_string(k));
    }
    if (k < trace_cap) {
      icpnn_iter_record& r = trace[k];
      r.iter = k;
      r.flags = 0;
      r.n_accepted = m.n_accepted;
      r.n_inliers = n_inliers;
      r.mse = m.mse;
      r.sigma2 = sigma2;
      std::memcpy(r.T, T, sizeof(T));
      const bool timing = (flags & ICPNN_TRACE_TIMING) != 0;
      r.kernel_ms = timing ? pass_ms : 0.f;
      r.residual_ms = timing ? resid_ms : 0.f;
    }
    std::memcpy(T, Tn, sizeof(T));
    mse_hist[0] = mse_hist[1];
    mse_hist[1] = mse_hist[2];
    mse_hist[2] = m.mse;
    done = k + 1;
    if (prelaunch) {
      // the queued pass evaluates T_{k+1}: the next iteration's pass or the final one
      transform_to_f32(T, R32, t32);
      pass_command(ps, next.seq, R32, t32);
      cur = next.seq;
      next.seq = 0;
    }
    if (k >= 2 && std::fabs(mse_hist[1] - mse_hist[2]) < eps && std::fabs(mse_hist[0] - mse_hist[1]) < eps)
      break;
  }
  if (timed > 0 && ev != nullptr) {
    const int32_t recorded = std::min(timed, done);
    ICPNN_CUDA(cudaEventSynchronize(ev[2 * (recorded - 1) + 1]));
    for (int32_t k = 0; k < recorded; ++k) ICPNN_CUDA(cudaEventElapsedTime(&trace[k].kernel_ms, ev[2 * k], ev[2 * k + 1]));
  }
  float R32[9], t32[3];
  transform_to_f32(T, R32, t32);
  icpnn_moments fin;
  if (run.active) {
    float ms = 0.f;
    if (int rc = persistent_pass(&fin, &ms)) return rc;
    run.stop();
  } else if (prelaunch) {
    if (int rc = collect(false, nullptr, nullptr, &fin)) return rc;
  } else {
    if (int rc = pass_run(ps, R32, t32, nullptr, nullptr, s, nullptr, nullptr, &fin)) return rc;
  }
  std::memcpy(out_T, T, sizeof(T));
  *final_mse = fin.mse;
  *iters = done;
  if (final_n_accepted != nullptr) *final_n_accepted = fin.n_accepted;
  return ICPNN_OK;
}

int icpnn_voxel_downsample(const float* xyz, int64_t n, float voxel_size, float* out_xyz, int64_t* out_n,
                           void* stream) {
  clear_error();
  if (out_n == nullptr) return fail(ICPNN_ERR_INVALID_ARG, "voxel_downsample: out_n is NULL");
  *out_n = 0;
  if (n < 0 || n > INT32_MAX) return fail(ICPNN_ERR_INVALID_ARG, "voxel_downsample: n out of range");
  if (!(voxel_size > 0.0f) || std::isinf(voxel_size))
    return fail(ICPNN_ERR_INVALID_ARG, "voxel_downsample: voxel_size must be positive and finite");
  if (n == 0) return ICPNN_OK;
  if (!xyz || !out_xyz) return fail(ICPNN_ERR_INVALID_ARG, "voxel_downsample: NULL pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int64_t count = 0;
  {
    Scratch sc(s);
    const float* d_xyz = xyz;
    if (!is_device_pointer(xyz)) {
      float* tmp = nullptr;
      ICPNN_CUDA(sc.alloc(&tmp, 3 * n));
      ICPNN_CUDA(cudaMemcpyAsync(tmp, xyz, static_cast<size_t>(n) * 3 * sizeof(float), cudaMemcpyHostToDevice, s));
      d_xyz = tmp;
    }
    const bool host_out = !is_device_pointer(out_xyz);
    float* d_out = out_xyz;
    if (host_out) ICPNN_CUDA(sc.alloc(&d_out, 3 * n));
    uint32_t* scratch = nullptr;
    long long* bounds = nullptr;
    unsigned long long* total = nullptr;
    ICPNN_CUDA(sc.alloc(&scratch, voxel_scratch_words(n)));
    ICPNN_CUDA(sc.alloc(&bounds, 8));
    ICPNN_CUDA(sc.alloc(&total, 1));
    long long host_bounds[8];
    cudaError_t err = cudaSuccess;
    const int rc = voxel_downsample(d_xyz, n, voxel_size, d_out, &count, scratch, bounds, total, host_bounds, s, &err);
    if (err != cudaSuccess) return fail(ICPNN_ERR_CUDA, std::string("voxel_downsample: ") + cudaGetErrorString(err));
    if (rc < 0)
      return fail(ICPNN_ERR_INVALID_ARG, "voxel_downsample: a voxel index exceeds 2^40 (coordinates too large "
                                         "for this voxel size)");
    if (host_out && count > 0) {
      ICPNN_CUDA(cudaMemcpyAsync(out_xyz, d_out, static_cast<size_t>(count) * 3 * sizeof(float),
                                 cudaMemcpyDeviceToHost, s));
      ICPNN_CUDA(cudaStreamSynchronize(s));
    }
  }
  *out_n = count;
  return ICPNN_OK;
}

int icpnn_probe_command_wait(const icpnn_tree* t, const float* src, int64_t n, uint64_t wait_ns, int32_t mode,
                             int32_t* outcome, void* stream) {
  clear_error();
  if (int rc = check_tree_on_device(t)) return rc;
  if (!src || !outcome) return fail(ICPNN_ERR_INVALID_ARG, "probe_command_wait: NULL pointer");
  *outcome = -1;
  if (n < 1 || n > INT32_MAX) return fail(ICPNN_ERR_INVALID_ARG, "probe_command_wait: n out of range");
  if (wait_ns < 1 || wait_ns > 1000000000ull)
    return fail(ICPNN_ERR_INVALID_ARG, "probe_command_wait: wait_ns must be in [1, 1e9]");
  if (mode < 0 || mode > 2) return fail(ICPNN_ERR_INVALID_ARG, "probe_command_wait: mode must be 0, 1 or 2");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Scratch sc(s);
  Pass ps;
  if (int rc = pass_setup(t, src, n, INFINITY, false, false, s, sc, &ps)) return rc;
  IcpPassParams p = pass_params(ps);
  p.cmd = command_block(ps.mb, true);
  p.mirror = ps.mirror;
  p.wait_ns = wait_ns;
  ICPNN_CUDA(launch_icp_pass(*ps.tree, ps.src.recs, ps.n, p, ps.partials, ps.counter, ps.mb->dev, nullptr,
                             nullptr, nullptr, nullptr, ps.grid, s));
  if (mode == 1) pass_command(ps, p.seq, nullptr, nullptr);
  if (mode == 2) {
    const float R[9] = {1, 0, 0, 0, 1, 0, 0, 0, 1}, tr[3] = {0, 0, 0};
    pass_command(ps, p.seq, R, tr);
  }
  ICPNN_CUDA(cudaStreamSynchronize(s));
  const volatile unsigned long long* words = result_words(ps.mb);
  *outcome = result_published(words, p.seq) ? 2 : words[kAbortWord] == p.seq ? 1 : 0;
  return ICPNN_OK;
}

int icpnn_probe_delay_commands(int32_t skip, int32_t count, uint64_t delay_ns) {
  clear_error();
  if (skip < 0 || count < 0 || delay_ns > 10000000000ull)
    return fail(ICPNN_ERR_INVALID_ARG, "probe_delay_commands: skip, count >= 0 and delay_ns <= 1e10");
  tl_cmd_skip = skip;
  tl_cmd_delayed = count;
  tl_cmd_delay_ns = delay_ns;
  return ICPNN_OK;
}

int icpnn_probe_delay_collect(int32_t skip, int32_t count, uint64_t delay_ns) {
  clear_error();
  if (skip < 0 || count < 0 || delay_ns > 10000000000ull)
    return fail(ICPNN_ERR_INVALID_ARG, "probe_delay_collect: skip, count >= 0 and delay_ns <= 1e10");
  tl_collect_skip = skip;
  tl_collect_delayed = count;
  tl_collect_delay_ns = delay_ns;
  return ICPNN_OK;
}

int icpnn_probe_read_result(const uint64_t* words, int64_t n_words, uint64_t seq, double* slots, float* pass_ms,
                            int32_t* complete) {
  clear_error();
  if (words == nullptr || slots == nullptr || pass_ms == nullptr || complete == nullptr)
    return fail(ICPNN_ERR_INVALID_ARG, "probe_read_result: NULL argument");
  if (n_words != kResultWords)
    return fail(ICPNN_ERR_INVALID_ARG, "probe_read_result: n_words must be " + std::to_string(kResultWords));
  const volatile unsigned long long* w = reinterpret_cast<const volatile unsigned long long*>(words);
  *complete = result_published(w, seq) ? 1 : 0;
  if (*complete) decode_published(w, slots, pass_ms);
  return ICPNN_OK;
}

const char* icpnn_last_error(void) { return tl_error.c_str(); }

int64_t icpnn_launch_count(void) { return g_launch_count.load(std::memory_order_relaxed); }

int32_t icpnn_version(void) { return 100; }

}  // extern "C"
