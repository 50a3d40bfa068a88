// One-time set-up per GPU, safe under concurrent host threads.
//
// Kernel attributes set with cudaFuncSetAttribute (for example a dynamic
// shared-memory size above the 48 KB default) and device properties such as
// the SM count belong to the device that is current when they are set or
// read. A launcher that remembered "done" in one process-wide flag would skip
// the set-up on every other device and its launches there would fail, so each
// launcher keeps one flag per device instead.
//
// Plain C++ (no CUDA types): `setup` returns 0 on success, any other value is
// passed back and leaves the device's flag clear so the next call retries.
#pragma once

#include <atomic>
#include <mutex>

namespace oscar {

constexpr int kMaxDevices = 64;

class PerDeviceOnce {
 public:
  // Runs setup() unless it already succeeded for `device`; 0 when the device is
  // set up, the setup's own non-zero result otherwise, -1 for a device index
  // outside [0, kMaxDevices).
  template <typename F>
  int run_on(int device, F&& setup) {
    if (device < 0 || device >= kMaxDevices) return -1;
    if (done_[device].load(std::memory_order_acquire)) return 0;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[device].load(std::memory_order_relaxed)) return 0;
    const int r = setup();
    if (r == 0) done_[device].store(true, std::memory_order_release);
    return r;
  }

 private:
  std::atomic<bool> done_[kMaxDevices] = {};
  std::mutex mu_;
};

// A value computed once per device (for example the SM count), 0 meaning "not
// yet known"; compute() must return a positive value to be kept.
class PerDeviceValue {
 public:
  template <typename F>
  int get(int device, F&& compute) {
    if (device < 0 || device >= kMaxDevices) return compute();
    int v = val_[device].load(std::memory_order_relaxed);
    if (v > 0) return v;
    v = compute();
    if (v > 0) val_[device].store(v, std::memory_order_relaxed);
    return v;
  }

 private:
  std::atomic<int> val_[kMaxDevices] = {};
};

}  // namespace oscar
