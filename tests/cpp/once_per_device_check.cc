// Host-only check of the per-device "set once" logic that the kernel
// launchers use for their attribute opt-ins (once_on_device in
// da_internal.h): set() runs once per device after it succeeds, again after
// a failure, on every call past device 63, and the bits of different devices
// do not interfere, also with several host threads.  Prints "ok" or the
// first failed check; exits non-zero on failure.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "da_internal.h"

static int fails = 0;
#define CHECK(c)                                              \
    do {                                                      \
        if (!(c)) {                                           \
            std::printf("failed: %s (line %d)\n", #c, __LINE__); \
            ++fails;                                          \
        }                                                     \
    } while (0)

int main() {
    unsigned long long done = 0;
    int calls[66] = {0};
    auto ok_on = [&](int dev) {
        return da::once_on_device(&done, dev, [&] { ++calls[dev < 0 ? 65 : dev]; return cudaSuccess; });
    };
    CHECK(ok_on(0) == cudaSuccess && calls[0] == 1);
    CHECK(ok_on(0) == cudaSuccess && calls[0] == 1);          // cached
    CHECK(ok_on(1) == cudaSuccess && calls[1] == 1);          // another device: its own bit
    CHECK(ok_on(1) == cudaSuccess && calls[1] == 1);
    CHECK(ok_on(63) == cudaSuccess && ok_on(63) == cudaSuccess && calls[63] == 1);
    CHECK(done == ((1ull << 0) | (1ull << 1) | (1ull << 63)));
    CHECK(ok_on(64) == cudaSuccess && ok_on(64) == cudaSuccess && calls[64] == 2);   // no bit: every call
    CHECK(ok_on(-1) == cudaSuccess && calls[65] == 1 && done == ((1ull << 0) | (1ull << 1) | (1ull << 63)));

    // a failing set() leaves the bit clear, so the next call tries again
    int tries = 0;
    cudaError_t next = cudaErrorInvalidValue;
    auto flaky = [&] { ++tries; return next; };
    CHECK(da::once_on_device(&done, 5, flaky) == cudaErrorInvalidValue && tries == 1);
    CHECK((done & (1ull << 5)) == 0);
    next = cudaSuccess;
    CHECK(da::once_on_device(&done, 5, flaky) == cudaSuccess && tries == 2);
    CHECK(da::once_on_device(&done, 5, flaky) == cudaSuccess && tries == 2);

    // several host threads on several devices: every device ends with its bit
    // set, set() ran at least once per device, and never after the bit was seen
    unsigned long long shared = 0;
    std::atomic<int> runs[8];
    for (auto &r : runs) r = 0;
    std::vector<std::thread> th;
    for (int t = 0; t < 16; ++t)
        th.emplace_back([&, t] {
            for (int k = 0; k < 1000; ++k) {
                const int dev = (t + k) % 8;
                da::once_on_device(&shared, dev, [&] { ++runs[dev]; return cudaSuccess; });
            }
        });
    for (auto &x : th) x.join();
    CHECK(shared == 0xffull);
    int before = 0;
    for (auto &r : runs) {
        CHECK(r >= 1 && r <= 16);   // at most one run per thread before the bit is visible
        before += r;
    }
    for (int dev = 0; dev < 8; ++dev) da::once_on_device(&shared, dev, [&] { ++runs[dev]; return cudaSuccess; });
    int after = 0;
    for (auto &r : runs) after += r;
    CHECK(after == before);
    if (fails == 0) std::printf("ok\n");
    return fails == 0 ? 0 : 1;
}
