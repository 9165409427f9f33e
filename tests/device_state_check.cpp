// Host-only check of the library's per-device launch bookkeeping
// (csrc/device_state.h): several host threads make first calls on two stub
// devices at once; each device must end with its own value, a failed set-up
// must not be recorded, and an out-of-range device index must be refused.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "device_state.h"

int main() {
    pkd::PerDevice state;
    std::atomic<int> calls[2] = {};
    std::atomic<int> wrong{0};
    std::vector<std::thread> threads;
    for (int t = 0; t < 8; ++t)
        threads.emplace_back([&, t] {
            for (int i = 0; i < 1000; ++i) {
                const int dev = (t + i) & 1;
                const int v = state.get(dev, [&] { calls[dev].fetch_add(1); return 10 + dev; }, -99);
                if (v != 10 + dev) wrong.fetch_add(1);
            }
        });
    for (auto& th : threads) th.join();
    if (wrong.load()) { std::printf("FAIL: %d wrong values\n", wrong.load()); return 1; }
    if (calls[0].load() < 1 || calls[1].load() < 1 || calls[0].load() > 8 || calls[1].load() > 8) {
        std::printf("FAIL: set-up ran %d / %d times\n", calls[0].load(), calls[1].load());
        return 1;
    }
    if (!state.has(0) || !state.has(1) || state.has(2)) { std::printf("FAIL: has()\n"); return 1; }
    // a failed set-up is returned but not recorded: the next call retries
    int tries = 0;
    if (state.get(5, [&] { ++tries; return -3; }, -99) != -3 || state.has(5)) { std::printf("FAIL: error kept\n"); return 1; }
    if (state.get(5, [&] { ++tries; return 7; }, -99) != 7 || tries != 2) { std::printf("FAIL: retry\n"); return 1; }
    if (state.get(5, [&] { ++tries; return 8; }, -99) != 7 || tries != 2) { std::printf("FAIL: memo\n"); return 1; }
    // device indices outside the table
    if (state.get(-1, [] { return 1; }, -99) != -99 || state.get(pkd::kMaxDevices, [] { return 1; }, -99) != -99) {
        std::printf("FAIL: bad device\n");
        return 1;
    }
    std::printf("ok %d %d\n", calls[0].load(), calls[1].load());
    return 0;
}
