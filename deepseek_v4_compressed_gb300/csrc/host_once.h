// host_once.h -- host set-up done once per device (kernel attributes such as
// the dynamic shared-memory limit), safe with several devices in one process
// and with several host threads calling at once.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

namespace dsv4 {

// One instance per call site.  run(fn) calls fn() the first time it is
// reached with a given device current and returns fn's result; later calls
// on that device return true without calling it.  A failed fn() is retried
// on the next call.  Kernel attributes belong to a device, so a process that
// drives a second GPU sets them again there.
class PerDeviceOnce {
public:
    template <typename F>
    bool run(F&& fn)
    {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
            (void)cudaGetLastError();
            return false;
        }
        std::lock_guard<std::mutex> lock(mu_);
        if (done_[dev]) return true;
        if (!fn()) return false;
        done_[dev] = true;
        return true;
    }

private:
    static constexpr int kMaxDevices = 64;
    std::mutex mu_;
    bool done_[kMaxDevices] = {};
};

}  // namespace dsv4
