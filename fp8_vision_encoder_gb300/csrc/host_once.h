// Per-device, thread-safe one-time set-up on the host (plain C++, no CUDA).
//
// Some CUDA settings belong to the current device, not to the process: the
// opt-in to more than 48 KB of dynamic shared memory (cudaFuncSetAttribute) is
// one.  A process that drives several GPUs, from one or several host threads,
// must make such a call once on each device.  PerDeviceOnce keeps one flag per
// device index under a mutex: run(dev, fn) calls fn() the first time it is
// asked for `dev` and remembers success; a failed fn() is retried by the next
// call.  Device indices outside [0, kMaxDevices) are refused.
#pragma once

#include <mutex>

namespace vitfp8 {

class PerDeviceOnce {
public:
    static constexpr int kMaxDevices = 64;

    template <class Fn>
    bool run(int dev, Fn&& fn) {
        if (dev < 0 || dev >= kMaxDevices) return false;
        std::lock_guard<std::mutex> lock(mu_);
        if (done_[dev]) return true;
        if (!fn()) return false;
        done_[dev] = true;
        return true;
    }

    bool done(int dev) {
        if (dev < 0 || dev >= kMaxDevices) return false;
        std::lock_guard<std::mutex> lock(mu_);
        return done_[dev];
    }

private:
    std::mutex mu_;
    bool done_[kMaxDevices] = {};
};

}  // namespace vitfp8
