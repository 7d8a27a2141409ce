// Process-wide pool of host worker threads, shared by the multi-frame
// registration and the tree build.  Created on first use and never torn down:
// the workers are detached and may still be parked on the queue's condition
// variable when the process exits.
//
// The tree build issues short parallel phases back to back, a few tens of
// microseconds each, where waking a parked thread can cost as much as the
// phase.  So an idle worker, and a caller waiting for its tasks, first poll for
// a bounded time (kSpin) before they block.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <deque>
#include <exception>
#include <functional>
#include <memory>
#include <mutex>
#include <thread>

#include "icpnn_internal.h"

namespace icpnn {
namespace {

constexpr auto kSpin = std::chrono::microseconds(200);

// Polls `ready` until it returns true or kSpin has passed; returns its value.
template <class F>
bool spin_until(const F& ready) {
  const auto end = std::chrono::steady_clock::now() + kSpin;
  for (int i = 0;; ++i) {
    if (ready()) return true;
    if ((i & 63) == 63) {
      if (std::chrono::steady_clock::now() >= end) return false;
      std::this_thread::yield();
    }
  }
}

class WorkerPool {
 public:
  void ensure(int n) {
    std::lock_guard<std::mutex> lock(mu_);
    while (threads_ < n) {
      std::thread([this] { loop(); }).detach();
      ++threads_;
    }
  }
  void submit(std::function<void()> job) {
    bool wake;
    {
      std::lock_guard<std::mutex> lock(mu_);
      queue_.push_back(std::move(job));
      queued_.fetch_add(1, std::memory_order_release);
      wake = sleepers_ > 0;
    }
    if (wake) cv_.notify_one();
  }

 private:
  void loop() {
    for (;;) {
      spin_until([this] { return queued_.load(std::memory_order_acquire) > 0; });
      std::function<void()> job;
      {
        std::unique_lock<std::mutex> lock(mu_);
        if (queue_.empty()) {
          ++sleepers_;
          cv_.wait(lock, [this] { return !queue_.empty(); });
          --sleepers_;
        }
        job = std::move(queue_.front());
        queue_.pop_front();
        queued_.fetch_sub(1, std::memory_order_relaxed);
      }
      job();
    }
  }
  std::mutex mu_;
  std::condition_variable cv_;
  std::deque<std::function<void()>> queue_;
  std::atomic<int> queued_{0};  // queue_.size(), readable without the lock
  int sleepers_ = 0;            // workers blocked on cv_, under mu_
  int threads_ = 0;
};

WorkerPool& pool() {
  static WorkerPool* p = new WorkerPool();
  return *p;
}

}  // namespace

void pool_submit(std::function<void()> job, int min_threads) {
  pool().ensure(min_threads);
  pool().submit(std::move(job));
}

void parallel_for(int tasks, const std::function<void(int)>& fn) {
  if (tasks <= 1) {
    if (tasks == 1) fn(0);
    return;
  }
  // Shared state lives on the heap: a helper may still touch it after the
  // caller has seen the last task finish and returned.
  struct Shared {
    std::atomic<int> next{0};
    std::atomic<int> done{0};
    std::mutex mu;
    std::condition_variable cv;
    std::exception_ptr error;  // first exception a task threw, under mu
  };
  auto sh = std::make_shared<Shared>();
  auto run = [sh, tasks, &fn] {
    for (int i; (i = sh->next.fetch_add(1)) < tasks;) {
      try {
        fn(i);
      } catch (...) {
        std::lock_guard<std::mutex> lock(sh->mu);
        if (!sh->error) sh->error = std::current_exception();
      }
      if (sh->done.fetch_add(1) + 1 == tasks) {
        std::lock_guard<std::mutex> lock(sh->mu);
        sh->cv.notify_all();
      }
    }
  };
  const int hw = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  const int helpers = std::min(tasks - 1, hw - 1);
  if (helpers > 0) {
    // one worker per hardware thread besides the caller: nested calls (the
    // tree build's subtrees) each need helpers of their own
    pool().ensure(hw - 1);
    // helpers only start tasks while some remain; `fn` is not touched after
    // the caller's wait below returns, because every started task has ended
    for (int h = 0; h < helpers; ++h) pool().submit(run);
  }
  run();  // the caller takes part, so nested parallel_for cannot deadlock
  if (!spin_until([&] { return sh->done.load() == tasks; })) {
    std::unique_lock<std::mutex> lock(sh->mu);
    sh->cv.wait(lock, [&] { return sh->done.load() == tasks; });
  }
  std::lock_guard<std::mutex> lock(sh->mu);
  if (sh->error) std::rethrow_exception(sh->error);
}

}  // namespace icpnn
