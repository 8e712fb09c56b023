// sv_internal.h -- host-side helpers shared by the libspecverify translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <mutex>

#include "specverify.h"

namespace sv {

// Records a thread-local message and returns `st`.
sv_status fail(sv_status st, const char *fmt, ...);
void clear_error();

bool pdl_enabled();
int device_sm_count();  // SMs of the current device (cached per device)
int current_device();

inline bool aligned(const void *p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}
inline bool overlaps(const void *a, size_t an, const void *b, size_t bn) {
  if (!a || !b || an == 0 || bn == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bn && y < x + an;
}

// Per-device one-time set-up (function attributes): the first call on each
// device runs fn with that device current, later calls (from any host
// thread) return its result.
struct PerDeviceOnce {
  static constexpr int kDevices = 64;
  std::once_flag flag[kDevices];
  cudaError_t result[kDevices] = {};
  template <class F>
  cudaError_t run(F fn) {
    const int d = current_device();
    if (d < 0 || d >= kDevices) return fn();
    std::call_once(flag[d], [&] { result[d] = fn(); });
    return result[d];
  }
};

// Checks cudaPeekAtLastError after a launch.
sv_status check_launch(const char *what);

// Per-translation-unit device error words (bounded-wait give-ups); each
// returns the word and clears it.  Synchronises the device.
unsigned take_device_error_qmv();
unsigned take_device_error_accept();
unsigned take_device_error_gdn();
unsigned take_device_error_plan();
unsigned take_device_error_wide();

}  // namespace sv
