// Per-device, thread-safe memo of one kernel's launch set-up.
//
// A kernel's dynamic shared-memory limit (cudaFuncSetAttribute) and the CTAs
// of it that fit an SM are properties of the (kernel, device) pair: a process
// that calls the library on several GPUs must set the attribute once on each.
// PerDevice keeps one slot per device index, filled by the first call made
// with that device current; concurrent first calls from several host threads
// may each run the set-up (it is idempotent) and store the same value.  No
// CUDA header is needed here, so host tests can drive it with a stub device.
#pragma once

#include <atomic>

namespace pkd {

constexpr int kMaxDevices = 64;

class PerDevice {
  public:
    // The value recorded for `dev` (> 0), computed by make() on first use.
    // make() returns a positive value, or a non-positive error code, which
    // is returned as is and not recorded (the next call tries again).
    // A device index outside [0, kMaxDevices) returns `bad_device`.
    template <class Make>
    int get(int dev, Make make, int bad_device) {
        if (dev < 0 || dev >= kMaxDevices) return bad_device;
        int v = slot_[dev].load(std::memory_order_acquire);
        if (v > 0) return v;
        v = make();
        if (v > 0) slot_[dev].store(v, std::memory_order_release);
        return v;
    }

    // Whether `dev` has a recorded value (for tests).
    bool has(int dev) const {
        return dev >= 0 && dev < kMaxDevices && slot_[dev].load(std::memory_order_acquire) > 0;
    }

  private:
    std::atomic<int> slot_[kMaxDevices] = {};
};

}  // namespace pkd
