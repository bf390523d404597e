// Host-only check of acnn::PerDeviceSizes (csrc/per_device.h): an action
// recorded for one device does not cover another device, a larger size is
// applied again, a failed action is not recorded, keys are independent, and
// concurrent callers apply an action once.  Exit status 0 on success.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "per_device.h"

static int failures = 0;
#define CHECK(c)                                                         \
    do {                                                                 \
        if (!(c)) {                                                      \
            std::printf("check failed at line %d: %s\n", __LINE__, #c); \
            ++failures;                                                  \
        }                                                                \
    } while (0)

int main() {
    acnn::PerDeviceSizes r;
    int kernel_a = 0, kernel_b = 0;
    int calls = 0;
    auto ok = [&] { ++calls; return true; };
    auto fail = [&] { ++calls; return false; };

    CHECK(r.ensure(&kernel_a, 0, 1000, ok) && calls == 1);   // first use on device 0
    CHECK(r.ensure(&kernel_a, 0, 1000, ok) && calls == 1);   // recorded: no second call
    CHECK(r.ensure(&kernel_a, 0, 500, ok) && calls == 1);    // a smaller size is covered
    CHECK(r.ensure(&kernel_a, 1, 1000, ok) && calls == 2);   // device 1 needs its own
    CHECK(r.ensure(&kernel_a, 1, 1000, ok) && calls == 2);
    CHECK(r.ensure(&kernel_a, 0, 2000, ok) && calls == 3);   // larger on device 0: again
    CHECK(r.ensure(&kernel_a, 1, 1500, ok) && calls == 4);   // ... and on device 1
    CHECK(r.ensure(&kernel_b, 0, 10, ok) && calls == 5);     // another kernel: its own
    CHECK(!r.ensure(&kernel_b, 2, 10, fail) && calls == 6);  // a failure is reported
    CHECK(!r.ensure(&kernel_b, 2, 10, fail) && calls == 7);  // ... and not recorded
    CHECK(r.ensure(&kernel_b, 2, 10, ok) && calls == 8);
    CHECK(r.ensure(&kernel_b, 2, 10, ok) && calls == 8);

    // eight threads asking for the same (key, device): one application
    acnn::PerDeviceSizes shared;
    std::atomic<int> applied{0};
    std::vector<std::thread> ts;
    for (int t = 0; t < 8; ++t)
        ts.emplace_back([&] {
            for (int i = 0; i < 1000; ++i)
                shared.ensure(&kernel_a, 3, 4096, [&] { applied.fetch_add(1); return true; });
        });
    for (auto& t : ts) t.join();
    CHECK(applied.load() == 1);

    std::printf("%s\n", failures ? "FAILED" : "ok");
    return failures ? 1 : 0;
}
