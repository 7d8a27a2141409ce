// Multi-frame registration ("Implementing ICP with CUDA-KDTree", section 3.4:
// with several frames to register, overlap one frame's queries with another
// frame's result copy and solve instead of running frames back to back).
//
// Here every frame is an ordinary icpnn_icp_align run by a host worker on a
// stream of its own; up to `max_concurrent` frames are in flight, handed out
// dynamically.  While one worker waits for its pass or solves on the host,
// the other workers' passes keep the GPU busy, and passes of different frames
// run side by side on the SMs, filling each other's tails.  Each frame's
// result is bit-identical to a single-frame icpnn_icp_align of it: the same
// kernels run with the same grids, only their interleaving changes.
//
// Workers come from the library's process-wide host pool; each worker keeps
// its own non-blocking stream per device and its own mapped result buffer for
// the life of the process.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <condition_variable>
#include <mutex>
#include <string>
#include <vector>

#include "icpnn_internal.h"

namespace icpnn {
namespace {

constexpr int kMaxDevices = 64;
thread_local cudaStream_t tl_stream[kMaxDevices] = {};

int worker_stream(int dev, cudaStream_t* out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(ICPNN_ERR_INVALID_ARG, "icp_align_batch: device id out of range");
  if (tl_stream[dev] == nullptr) {
    const cudaError_t e = cudaStreamCreateWithFlags(&tl_stream[dev], cudaStreamNonBlocking);
    if (e != cudaSuccess) {
      tl_stream[dev] = nullptr;
      return fail(ICPNN_ERR_CUDA, std::string("cudaStreamCreateWithFlags: ") + cudaGetErrorString(e));
    }
  }
  *out = tl_stream[dev];
  return ICPNN_OK;
}

}  // namespace
}  // namespace icpnn

using namespace icpnn;

extern "C" int icpnn_icp_align_batch(const icpnn_tree* target, int32_t n_frames, const float* const* srcs,
                                     const int64_t* n_src, int32_t max_iter, double eps,
                                     double max_corr_dist, const double* init_T, double* out_T,
                                     double* final_mse, int32_t* iters, int64_t* final_n_accepted,
                                     int32_t* status, uint32_t flags, int32_t max_concurrent, void* stream) {
  clear_error();
  if (target == nullptr) return fail(ICPNN_ERR_INVALID_ARG, "icp_align_batch: tree is NULL");
  if (target->dev.nodes == nullptr) return fail(ICPNN_ERR_NOT_UPLOADED, "icp_align_batch: tree has not been uploaded");
  if (n_frames < 1) return fail(ICPNN_ERR_INVALID_ARG, "icp_align_batch: n_frames must be >= 1");
  if (!srcs || !n_src || !out_T || !final_mse || !iters || !status)
    return fail(ICPNN_ERR_INVALID_ARG, "icp_align_batch: NULL pointer");
  for (int32_t f = 0; f < n_frames; ++f)
    if (srcs[f] == nullptr || n_src[f] < 1 || n_src[f] > INT32_MAX)
      return fail(ICPNN_ERR_INVALID_ARG, "icp_align_batch: bad source " + std::to_string(f));
  if (flags & ~(ICPNN_RESIDUAL_REJECT | ICPNN_NO_PRELAUNCH))
    return fail(ICPNN_ERR_INVALID_ARG, "icp_align_batch: unknown flag");
  if (max_concurrent <= 0) max_concurrent = 4;
  const int workers = std::min<int32_t>(max_concurrent, n_frames);
  // With several frames in flight a pass queued ahead of its transform would
  // hold SM slots that other frames' passes can use: launch after the solve.
  const uint32_t frame_flags = flags | (workers > 1 ? ICPNN_NO_PRELAUNCH : 0u);
  const int dev = target->dev.device;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != dev)
    return fail(ICPNN_ERR_NOT_UPLOADED, "icp_align_batch: tree was uploaded to device " + std::to_string(dev) +
                                            ", current device is " + std::to_string(cur));

  // frames start after the work already enqueued on the caller's stream
  cudaEvent_t ready = nullptr;
  cudaError_t e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventRecord(ready, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    if (ready) cudaEventDestroy(ready);
    return fail(ICPNN_ERR_CUDA, std::string("icp_align_batch: ") + cudaGetErrorString(e));
  }

  struct Shared {
    std::atomic<int32_t> next{0};
    std::mutex mu;
    std::condition_variable cv;
    int done = 0;
    std::vector<std::string> msg;
  } sh;
  sh.msg.resize(static_cast<size_t>(n_frames));

  for (int w = 0; w < workers; ++w) {
    pool_submit([&, dev] {
      cudaStream_t ws = nullptr;
      int rc = cudaSetDevice(dev) == cudaSuccess ? worker_stream(dev, &ws)
                                                 : fail(ICPNN_ERR_CUDA, "icp_align_batch: cudaSetDevice failed");
      if (rc == ICPNN_OK && cudaStreamWaitEvent(ws, ready, 0) != cudaSuccess)
        rc = fail(ICPNN_ERR_CUDA, "icp_align_batch: cudaStreamWaitEvent failed");
      const std::string setup_msg = rc == ICPNN_OK ? std::string() : std::string(icpnn_last_error());
      for (;;) {
        const int32_t f = sh.next.fetch_add(1);
        if (f >= n_frames) break;
        int r = rc;
        if (r == ICPNN_OK)
          r = icpnn_icp_align(target, srcs[f], n_src[f], max_iter, eps, max_corr_dist,
                              init_T ? init_T + 16 * static_cast<int64_t>(f) : nullptr,
                              out_T + 16 * static_cast<int64_t>(f), final_mse + f, iters + f,
                              final_n_accepted ? final_n_accepted + f : nullptr, nullptr, 0, frame_flags, ws);
        status[f] = r;
        if (r != ICPNN_OK) sh.msg[static_cast<size_t>(f)] = rc != ICPNN_OK ? setup_msg : icpnn_last_error();
      }
      {
        std::lock_guard<std::mutex> lock(sh.mu);
        ++sh.done;
      }
      sh.cv.notify_all();
    }, workers);
  }
  {
    std::unique_lock<std::mutex> lock(sh.mu);
    sh.cv.wait(lock, [&] { return sh.done == workers; });
  }
  cudaEventDestroy(ready);
  for (int32_t f = 0; f < n_frames; ++f)
    if (status[f] != ICPNN_OK)
      return fail(status[f], "icp_align_batch: frame " + std::to_string(f) + ": " + sh.msg[static_cast<size_t>(f)]);
  return ICPNN_OK;
}
