// device_once.h -- one-time set-up per device, in plain C++ (no CUDA types),
// so that the host logic can be compiled and checked without a GPU.
//
// Kernel attributes such as the dynamic shared-memory limit belong to one
// device's context: a process that drives several devices has to set them on
// each. once_per_device_with runs `set` once for every device index that
// `get_device` reports as current, keeps its result per device, and returns
// that result on every later call made while the same device is current.
#pragma once

#include <mutex>

namespace fl {

constexpr int kMaxDevices = 64;

// Err is an error-code type whose value-initialised state means success.
// get_device(int*) -> Err reports the current device; bad_device is returned
// for an index outside [0, kMaxDevices).
template <class Err, class GetDevice, class Set>
Err once_per_device_with(std::once_flag (&once)[kMaxDevices], Err (&res)[kMaxDevices], GetDevice &&get_device,
                         Err bad_device, Set &&set) {
    int dev = -1;
    const Err e = get_device(&dev);
    if (e != Err{}) return e;
    if (dev < 0 || dev >= kMaxDevices) return bad_device;
    std::call_once(once[dev], [&] { res[dev] = set(); });
    return res[dev];
}

}  // namespace fl
