// Unit test of la::PerDeviceCache (csrc/per_device.h), built with the host
// compiler alone: a value is computed once per (device, key) pair, another
// device gets its own value for the same key, and concurrent first callers
// compute it once.  Prints "ok" and exits 0 on success.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <thread>
#include <vector>

#include "per_device.h"

#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      std::fprintf(stderr, "check failed line %d: %s\n", __LINE__, #c); \
      return 1;                                               \
    }                                                         \
  } while (0)

int main() {
  la::PerDeviceCache<const void *, int> cache;
  int calls = 0;
  static int kernel_a, kernel_b;
  // device 0: computed once, then served from the table
  CHECK(cache.get(0, &kernel_a, [&] { return ++calls; }) == 1);
  CHECK(cache.get(0, &kernel_a, [&] { return ++calls; }) == 1);
  CHECK(calls == 1);
  // the same kernel on device 1 is a separate entry (a device's attribute is per context)
  CHECK(cache.get(1, &kernel_a, [&] { return ++calls; }) == 2);
  CHECK(calls == 2);
  // another kernel on device 0
  CHECK(cache.get(0, &kernel_b, [&] { return ++calls; }) == 3);
  CHECK(cache.get(1, &kernel_a, [&] { return ++calls; }) == 2);
  CHECK(cache.size() == 3);
  // a failure is remembered like any other result (the condition is a property of the device)
  la::PerDeviceCache<int, int> errs;
  int tries = 0;
  CHECK(errs.get(5, 0, [&] { ++tries; return -7; }) == -7);
  CHECK(errs.get(5, 0, [&] { ++tries; return 0; }) == -7);
  CHECK(tries == 1);
  // many threads racing on the first call of several devices: one computation per device
  la::PerDeviceCache<int, int> race;
  std::atomic<int> computed{0};
  std::vector<std::thread> ts;
  for (int t = 0; t < 16; ++t)
    ts.emplace_back([&, t] {
      for (int rep = 0; rep < 100; ++rep) {
        const int dev = (t + rep) % 4;
        const int v = race.get(dev, 0, [&] { computed.fetch_add(1); return 100 + dev; });
        if (v != 100 + dev) std::abort();
      }
    });
  for (auto &th : ts) th.join();
  CHECK(computed.load() == 4);
  CHECK(race.size() == 4);
  std::printf("ok\n");
  return 0;
}
