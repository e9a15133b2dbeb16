// Host-only check of PerDeviceOnce (per-device, thread-safe one-time set-up):
// many threads asking for many devices at once run each device's set-up
// exactly once; a failed set-up is retried by the next call; device indices
// outside the table are refused without running anything.  Plain C++, no
// CUDA: the set-up functions here only count their calls.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "host_once.h"

int main() {
    using vitfp8::PerDeviceOnce;
    constexpr int kDev = PerDeviceOnce::kMaxDevices;
    PerDeviceOnce once;
    std::atomic<int> calls[kDev];
    for (auto& c : calls) c = 0;

    // 16 threads, each asking for every device 50 times in a different order.
    std::vector<std::thread> th;
    std::atomic<int> failures{0};
    for (int t = 0; t < 16; ++t) {
        th.emplace_back([&, t] {
            for (int rep = 0; rep < 50; ++rep)
                for (int i = 0; i < kDev; ++i) {
                    const int dev = (i * 7 + t * 13 + rep) % kDev;
                    if (!once.run(dev, [&] { ++calls[dev]; return true; })) ++failures;
                }
        });
    }
    for (auto& x : th) x.join();
    if (failures != 0) { std::printf("FAIL: %d refused calls\n", failures.load()); return 1; }
    for (int d = 0; d < kDev; ++d)
        if (calls[d] != 1 || !once.done(d)) { std::printf("FAIL: device %d set up %d times\n", d, calls[d].load()); return 1; }

    // A set-up that fails is not remembered: the next call runs it again.
    PerDeviceOnce retry;
    int attempts = 0;
    if (retry.run(3, [&] { ++attempts; return false; })) { std::puts("FAIL: failed set-up reported ok"); return 1; }
    if (retry.done(3)) { std::puts("FAIL: failed set-up remembered"); return 1; }
    if (!retry.run(3, [&] { ++attempts; return true; }) || attempts != 2) { std::puts("FAIL: no retry"); return 1; }
    if (!retry.run(3, [&] { ++attempts; return true; }) || attempts != 2) { std::puts("FAIL: ran twice"); return 1; }
    if (retry.done(2)) { std::puts("FAIL: another device marked"); return 1; }

    // Out-of-range device indices: refused, set-up never called.
    int ran = 0;
    if (retry.run(-1, [&] { ++ran; return true; }) || retry.run(kDev, [&] { ++ran; return true; }) || ran != 0) {
        std::puts("FAIL: out-of-range device accepted");
        return 1;
    }
    std::puts("host_once ok");
    return 0;
}
