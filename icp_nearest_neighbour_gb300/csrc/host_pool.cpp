// Process-wide pool of host worker threads, shared by the multi-frame
// registration and the tree build.  Created on first use and never torn down:
// the workers are detached and may still be parked on the condition variable
// when the process exits.
//
// Two kinds of work reach the workers:
//   - jobs (pool_submit): long-running closures such as one frame of a batch
//     registration, taken from a mutex-guarded queue;
//   - parallel regions (parallel_for): short phases of the tree build, a few
//     tens of microseconds each, issued back to back.  A region is published
//     on a lock-free board that idle workers scan; a worker joins a region by
//     one compare-and-swap and takes tasks with fetch_add, so a region costs
//     no lock, no allocation and no wake-up while the workers are polling.
//     (Handing each region's tasks out through the job queue cost 18 us for
//     two tasks and 90 us for twelve: the polling workers and the caller
//     convoyed on the queue's mutex.)
// An idle worker polls for a bounded time (kSpin) before it blocks.
//
// Region lifetime.  Regions live in a fixed array and are reused; a board
// entry names a region by (slot, generation).  A worker joins only if the
// region's state still carries that generation, by incrementing the region's
// user count in the same 64-bit word, and the owner reuses a region only
// after its user count has dropped to zero.  So a worker never touches a
// region that has been handed to another caller, and nested or concurrent
// parallel_for calls need no per-thread bookkeeping.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <deque>
#include <exception>
#include <functional>
#include <mutex>
#include <thread>

#include "icpnn_internal.h"

namespace icpnn {
namespace {

constexpr auto kSpin = std::chrono::microseconds(200);
constexpr int kRegions = 128;     // regions alive at once (nesting x callers)
constexpr int kBoardSlots = 64;   // regions published at once

struct Region {
  // generation (high 32 bits) and the number of workers inside (low 32 bits)
  std::atomic<uint64_t> state{0};
  std::atomic<bool> taken{false};  // owned by a parallel_for call
  std::atomic<int> next{0};
  std::atomic<int> done{0};
  std::atomic<int> tasks{0};
  const std::function<void(int)>* fn = nullptr;
  std::mutex error_mu;
  std::exception_ptr error;  // first exception a task threw

  bool open() const {
    return next.load(std::memory_order_relaxed) < tasks.load(std::memory_order_relaxed);
  }
  // Runs unclaimed tasks until none is left; returns how many it ran.
  int run_tasks() {
    const int n = tasks.load(std::memory_order_relaxed);
    int ran = 0;
    for (int i; (i = next.fetch_add(1, std::memory_order_acq_rel)) < n; ++ran) {
      try {
        (*fn)(i);
      } catch (...) {
        std::lock_guard<std::mutex> lock(error_mu);
        if (!error) error = std::current_exception();
      }
      done.fetch_add(1, std::memory_order_acq_rel);
    }
    return ran;
  }
};

class WorkerPool {
 public:
  WorkerPool() {
    for (auto& b : board_) b.store(0, std::memory_order_relaxed);
  }

  void ensure(int n) {
    if (threads_.load(std::memory_order_acquire) >= n) return;
    std::lock_guard<std::mutex> lock(mu_);
    while (threads_.load(std::memory_order_relaxed) < n) {
      std::thread([this] { loop(); }).detach();
      threads_.fetch_add(1, std::memory_order_release);
    }
  }

  void submit(std::function<void()> job) {
    {
      std::lock_guard<std::mutex> lock(mu_);
      queue_.push_back(std::move(job));
      queued_.fetch_add(1, std::memory_order_seq_cst);
    }
    wake();
  }

  // A free region, its generation advanced, or nullptr if all are in use.
  // The generation moves on only while no worker is inside: a worker that
  // read an old board entry and joined after the previous owner released the
  // region leaves at once (no task left) and cannot join the new generation.
  Region* acquire_region(uint32_t* gen) {
    for (int k = 0; k < kRegions; ++k) {
      Region& r = regions_[k];
      bool expected = false;
      if (r.taken.load(std::memory_order_relaxed) ||
          !r.taken.compare_exchange_strong(expected, true, std::memory_order_acquire))
        continue;
      uint64_t s = r.state.load(std::memory_order_acquire);
      for (int i = 0;; ++i) {
        if ((s & 0xffffffffull) == 0) {
          const uint64_t bumped = (((s >> 32) + 1u) & 0xffffffffull) << 32;
          if (r.state.compare_exchange_weak(s, bumped, std::memory_order_acq_rel)) {
            *gen = static_cast<uint32_t>(bumped >> 32);
            return &r;
          }
        } else {
          if ((i & 63) == 63) std::this_thread::yield();
          s = r.state.load(std::memory_order_acquire);
        }
      }
    }
    return nullptr;
  }

  // Publishes region r (generation gen); returns its board slot or -1.
  int publish(Region* r, uint32_t gen) {
    const uint64_t entry = (static_cast<uint64_t>(r - regions_ + 1) << 32) | gen;
    for (int k = 0; k < kBoardSlots; ++k) {
      uint64_t expected = 0;
      if (board_[k].load(std::memory_order_relaxed) == 0 &&
          board_[k].compare_exchange_strong(expected, entry, std::memory_order_seq_cst)) {
        published_.fetch_add(1, std::memory_order_seq_cst);
        wake();
        return k;
      }
    }
    return -1;
  }

  void unpublish(int slot) {
    board_[slot].store(0, std::memory_order_seq_cst);
    published_.fetch_sub(1, std::memory_order_seq_cst);
  }

  // Waits until no worker is inside r, then hands it back.
  void release_region(Region* r) {
    for (int i = 0; (r->state.load(std::memory_order_acquire) & 0xffffffffull) != 0; ++i)
      if ((i & 63) == 63) std::this_thread::yield();
    r->taken.store(false, std::memory_order_release);
  }

 private:
  // Joins a published region with unclaimed tasks and runs them; true if it
  // ran any.
  bool help() {
    if (published_.load(std::memory_order_seq_cst) == 0) return false;
    for (int k = 0; k < kBoardSlots; ++k) {
      const uint64_t entry = board_[k].load(std::memory_order_acquire);
      if (entry == 0) continue;
      Region& r = regions_[(entry >> 32) - 1];
      if (!r.open()) continue;
      const uint32_t gen = static_cast<uint32_t>(entry);
      uint64_t s = r.state.load(std::memory_order_acquire);
      bool joined = false;
      while (static_cast<uint32_t>(s >> 32) == gen) {
        if (r.state.compare_exchange_weak(s, s + 1, std::memory_order_acq_rel)) {
          joined = true;
          break;
        }
      }
      if (!joined) continue;
      const int ran = r.run_tasks();
      r.state.fetch_sub(1, std::memory_order_acq_rel);
      if (ran > 0) return true;
    }
    return false;
  }

  // Some published region still has unclaimed tasks.  (The regions are never
  // freed, so reading one that a new owner is filling in is harmless.)
  bool has_open_region() const {
    if (published_.load(std::memory_order_seq_cst) == 0) return false;
    for (int k = 0; k < kBoardSlots; ++k) {
      const uint64_t entry = board_[k].load(std::memory_order_acquire);
      if (entry != 0 && regions_[(entry >> 32) - 1].open()) return true;
    }
    return false;
  }

  bool take_job() {
    if (queued_.load(std::memory_order_seq_cst) == 0) return false;
    std::function<void()> job;
    {
      std::lock_guard<std::mutex> lock(mu_);
      if (queue_.empty()) return false;
      job = std::move(queue_.front());
      queue_.pop_front();
      queued_.fetch_sub(1, std::memory_order_relaxed);
    }
    job();
    return true;
  }

  void loop() {
    for (;;) {
      auto end = std::chrono::steady_clock::now() + kSpin;
      for (int i = 0;; ++i) {
        if (help() || take_job()) {
          end = std::chrono::steady_clock::now() + kSpin;
          continue;
        }
        if ((i & 63) == 63) {
          // while a parallel region is published (the tree build's upper
          // levels), more are coming: stay ready instead of parking
          const auto now = std::chrono::steady_clock::now();
          if (published_.load(std::memory_order_relaxed) > 0) end = now + kSpin;
          else if (now >= end) break;
          std::this_thread::yield();
        }
      }
      // Park until the next wake-up round, then poll again: a round is
      // announced once (wake), however many regions follow it.
      std::unique_lock<std::mutex> lock(mu_);
      sleepers_.fetch_add(1, std::memory_order_seq_cst);
      const uint64_t round = wake_round_.load(std::memory_order_seq_cst);
      if (queued_.load(std::memory_order_seq_cst) == 0 && !has_open_region())
        cv_.wait(lock, [&] { return wake_round_.load(std::memory_order_seq_cst) != round; });
      sleepers_.fetch_sub(1, std::memory_order_seq_cst);
      wake_pending_.store(false, std::memory_order_seq_cst);
    }
  }

 public:
  // Wakes parked workers after new work became visible (or ahead of it).  A
  // worker about to park counts itself as a sleeper before it checks for
  // work, so either it sees the work or the caller sees the sleeper.  One
  // round at a time: callers that find a round pending skip the mutex.
  void wake() {
    if (sleepers_.load(std::memory_order_seq_cst) == 0) return;
    if (wake_pending_.exchange(true, std::memory_order_seq_cst)) return;
    {
      std::lock_guard<std::mutex> lock(mu_);
      wake_round_.fetch_add(1, std::memory_order_seq_cst);
    }
    cv_.notify_all();
  }

 private:

  std::mutex mu_;
  std::condition_variable cv_;
  std::deque<std::function<void()>> queue_;
  std::atomic<int> queued_{0};     // queue_.size(), readable without the lock
  std::atomic<int> sleepers_{0};   // workers parked on cv_
  std::atomic<uint64_t> wake_round_{0};
  std::atomic<bool> wake_pending_{false};  // a round announced, no worker up yet
  std::atomic<int> threads_{0};
  std::atomic<int> published_{0};  // board entries in use
  std::atomic<uint64_t> board_[kBoardSlots];
  Region regions_[kRegions];
};

WorkerPool& pool() {
  static WorkerPool* p = new WorkerPool();
  return *p;
}

}  // namespace

void pool_wake() { pool().wake(); }

void pool_submit(std::function<void()> job, int min_threads) {
  pool().ensure(min_threads);
  pool().submit(std::move(job));
}

void parallel_for(int tasks, const std::function<void(int)>& fn) {
  if (tasks <= 1) {
    if (tasks == 1) fn(0);
    return;
  }
  const int hw = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  WorkerPool& wp = pool();
  uint32_t gen = 0;
  Region* r = hw > 1 ? wp.acquire_region(&gen) : nullptr;
  if (r == nullptr) {  // no helpers, or every region in use: run here
    for (int i = 0; i < tasks; ++i) fn(i);
    return;
  }
  r->fn = &fn;
  r->next.store(0, std::memory_order_relaxed);
  r->done.store(0, std::memory_order_relaxed);
  r->tasks.store(tasks, std::memory_order_relaxed);
  r->error = nullptr;
  // one worker per hardware thread besides the caller: nested calls (the
  // tree build's subtrees) each need helpers of their own
  wp.ensure(hw - 1);
  const int slot = wp.publish(r, gen);
  r->run_tasks();  // the caller takes part, so nested parallel_for cannot deadlock
  if (slot >= 0) wp.unpublish(slot);
  // every task is claimed; wait for those that workers still run
  for (int i = 0; r->done.load(std::memory_order_acquire) < tasks; ++i)
    if ((i & 63) == 63) std::this_thread::yield();
  std::exception_ptr error = r->error;
  wp.release_region(r);
  if (error) std::rethrow_exception(error);
}

}  // namespace icpnn
