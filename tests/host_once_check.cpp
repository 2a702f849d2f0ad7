// Host-only check of dsa::PerDeviceOnce (the per-(kernel, device) set-up table):
// a step runs once per (key, device), a failed step is retried, distinct devices
// and keys are independent, and concurrent callers run a step exactly once.
#include <atomic>
#include <cstdio>
#include <thread>
#include <vector>

#include "dsa_once.h"

#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      std::printf("FAILED line %d: %s\n", __LINE__, #c);      \
      return 1;                                               \
    }                                                         \
  } while (0)

int main() {
  dsa::PerDeviceOnce t;
  int kernel_a = 0, kernel_b = 0;  // stand-ins for two kernels' addresses
  int runs = 0;
  auto ok = [&] { ++runs; return true; };
  CHECK(t.run(&kernel_a, 0, ok) && runs == 1);
  CHECK(t.run(&kernel_a, 0, ok) && runs == 1);  // already done on device 0
  CHECK(t.run(&kernel_a, 1, ok) && runs == 2);  // a second device needs its own set-up
  CHECK(t.run(&kernel_b, 1, ok) && runs == 3);  // and so does a second kernel
  CHECK(t.size() == 3);
  int fails = 0;
  auto bad = [&] { ++fails; return false; };
  CHECK(!t.run(&kernel_b, 2, bad) && fails == 1);
  CHECK(!t.run(&kernel_b, 2, bad) && fails == 2);  // not recorded: tried again
  CHECK(t.run(&kernel_b, 2, ok) && runs == 4);
  CHECK(t.run(&kernel_b, 2, bad) && fails == 2);   // recorded after the success
  // 8 threads race on (kernel_a, 7): the step runs once
  std::atomic<int> hits{0};
  std::vector<std::thread> th;
  for (int i = 0; i < 8; ++i)
    th.emplace_back([&] {
      for (int k = 0; k < 1000; ++k) t.run(&kernel_a, 7, [&] { hits.fetch_add(1); return true; });
    });
  for (auto& x : th) x.join();
  CHECK(hits.load() == 1);
  CHECK(t.size() == 5);
  std::printf("ok\n");
  return 0;
}
