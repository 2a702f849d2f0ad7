// dsa_once.h -- a table of (key, device) pairs on which a one-time set-up step
// has succeeded.  Kernel attributes such as the dynamic shared-memory limit
// apply to the current device only, so they are set once per kernel and per
// device; the table is guarded by a mutex so that host threads driving
// different devices (or the same one) do not race.  Plain C++: no CUDA types,
// so the logic is testable on a machine without a GPU.
#pragma once
#include <mutex>
#include <utility>
#include <vector>

namespace dsa {

class PerDeviceOnce {
 public:
  // Runs `step` (a callable returning true on success) unless it has already
  // succeeded for (key, device); a failed step is retried on the next call.
  // Returns true when the step has succeeded, now or before.
  template <class F>
  bool run(const void* key, int device, F&& step) {
    std::lock_guard<std::mutex> lk(mu_);
    for (const auto& e : done_)
      if (e.first == key && e.second == device) return true;
    if (!step()) return false;
    done_.emplace_back(key, device);
    return true;
  }
  // Number of (key, device) pairs recorded.
  size_t size() {
    std::lock_guard<std::mutex> lk(mu_);
    return done_.size();
  }

 private:
  std::mutex mu_;
  std::vector<std::pair<const void*, int>> done_;
};

}  // namespace dsa
