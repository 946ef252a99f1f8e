// Drives lcb::DeviceOnce (the per-device-context set-up flags the kernel
// launchers use for their shared-memory limit) with made-up device ordinals and
// context ids, on the host. Prints "ok" and exits 0 when every check holds.
#include <cstdio>

#include "device_once.h"

static int failures = 0;
#define CHECK(cond)                                                 \
  do {                                                              \
    if (!(cond)) {                                                  \
      std::printf("check failed at line %d: %s\n", __LINE__, #cond); \
      ++failures;                                                   \
    }                                                               \
  } while (0)

int main() {
  lcb::DeviceOnce once;
  int calls[4] = {0, 0, 0, 0};
  auto setter = [&](int dev, int rc) {
    return [&calls, dev, rc] {
      ++calls[dev];
      return rc;
    };
  };
  const int kBad = -4;

  // first use on device 0 in context 11 runs the set-up; repeats do not
  CHECK(once.run(0, 11, setter(0, 0), kBad) == 0);
  CHECK(once.run(0, 11, setter(0, 0), kBad) == 0);
  CHECK(calls[0] == 1);
  CHECK(once.done(0, 11));
  // another device has its own flag
  CHECK(!once.done(1, 11));
  CHECK(once.run(1, 12, setter(1, 0), kBad) == 0);
  CHECK(calls[1] == 1);
  CHECK(once.run(0, 11, setter(0, 0), kBad) == 0 && calls[0] == 1);
  // a new context on device 0 (after a reset) runs it again, once
  CHECK(once.run(0, 13, setter(0, 0), kBad) == 0);
  CHECK(once.run(0, 13, setter(0, 0), kBad) == 0);
  CHECK(calls[0] == 2);
  CHECK(!once.done(0, 11) && once.done(0, 13));
  // a failing set-up returns its status and is retried next time
  CHECK(once.run(2, 14, setter(2, -4), kBad) == -4);
  CHECK(!once.done(2, 14));
  CHECK(once.run(2, 14, setter(2, 0), kBad) == 0);
  CHECK(calls[2] == 2 && once.done(2, 14));
  // no context id known: the set-up runs every time and nothing is remembered
  CHECK(once.run(3, 0, setter(3, 0), kBad) == 0);
  CHECK(once.run(3, 0, setter(3, 0), kBad) == 0);
  CHECK(calls[3] == 2 && !once.done(3, 0));
  // ordinals outside the table are refused without running the set-up
  int outside = 0;
  CHECK(once.run(-1, 5, [&] { return ++outside, 0; }, kBad) == kBad);
  CHECK(once.run(lcb::kMaxDeviceOrdinals, 5, [&] { return ++outside, 0; }, kBad) == kBad);
  CHECK(outside == 0);
  if (failures) return 1;
  std::printf("ok\n");
  return 0;
}
