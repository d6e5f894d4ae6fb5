// Host-only check of fl::once_per_device_with (csrc/device_once.h) against a
// fake device getter: the set-up runs once per device index, its result is
// kept per device, and indices outside the table are refused. Prints "ok" and
// exits 0 on success; prints the failed check and exits 1 otherwise.
#include <cstdio>
#include <thread>
#include <vector>

#include "device_once.h"

namespace {
int g_current = 0;        // the fake "current device"
int g_get_error = 0;      // error the fake getter reports (0 = success)
int g_calls[fl::kMaxDevices + 8] = {};

int fake_get(int *dev) {
    if (g_get_error) return g_get_error;
    *dev = g_current;
    return 0;
}

int failures = 0;
void check(bool ok, const char *what) {
    if (!ok) {
        std::printf("FAILED: %s\n", what);
        ++failures;
    }
}
}  // namespace

int main() {
    static std::once_flag once[fl::kMaxDevices];
    static int res[fl::kMaxDevices];
    const int kBad = 101;
    // the set-up of device d fails with 7 for d == 3 and succeeds elsewhere
    auto run = [&] {
        return fl::once_per_device_with(once, res, fake_get, kBad, [&] {
            ++g_calls[g_current];
            return g_current == 3 ? 7 : 0;
        });
    };
    g_current = 0;
    check(run() == 0 && run() == 0, "device 0 succeeds");
    check(g_calls[0] == 1, "device 0 set up exactly once");
    g_current = 1;
    check(run() == 0, "device 1 succeeds");
    check(g_calls[1] == 1, "device 1 gets its own set-up");
    g_current = 3;
    check(run() == 7 && run() == 7, "device 3 reports its set-up error on every call");
    check(g_calls[3] == 1, "a failed set-up is not retried");
    g_current = 0;
    check(run() == 0 && g_calls[0] == 1, "device 0 keeps its result after other devices");
    g_current = fl::kMaxDevices;
    check(run() == kBad && g_calls[fl::kMaxDevices] == 0, "index past the table is refused");
    g_current = -1;
    check(run() == kBad, "negative index is refused");
    g_current = 5;
    g_get_error = 9;
    check(run() == 9 && g_calls[5] == 0, "getter error is returned and nothing is set up");
    g_get_error = 0;
    // many threads on one fresh device: still one set-up
    g_current = 6;
    std::vector<std::thread> ts;
    for (int t = 0; t < 16; ++t) ts.emplace_back([&] { run(); });
    for (auto &t : ts) t.join();
    check(g_calls[6] == 1, "concurrent first calls set up once");
    if (failures) return 1;
    std::printf("ok\n");
    return 0;
}
