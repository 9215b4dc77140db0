// Bounded mbarrier waits shared by the kernels.
//
// A wait polls the barrier with mbarrier.try_wait (the hardware may suspend
// the thread until the phase completes) and gives up after a time limit: it
// then sets the block's shared abort flag and a bit in the device-wide error
// word, which the host reads with ra_device_error().  The error word is also
// polled now and then, so that every block stops early once one has given up.
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace ra {
namespace {

constexpr uint64_t kWaitTimeoutNs = 4000000000ull;   // ordinary waits: 4 s
constexpr uint64_t kDrainTimeoutNs = 200000000ull;   // draining after an abort: 0.2 s

struct Abort {
  volatile int* flag;     // shared memory: this block gives up
  unsigned int* err;      // global memory: the device error word
};

// Record an error: set `code` in the device error word and, when the host has
// registered a mirror for this device (a word of pinned host memory mapped
// into the device's address space, whose device address sits 8 bytes after
// the error word), raise the mirror too, so that the host's entry points see
// the pending error without synchronising.
__device__ __forceinline__ void raise_error(unsigned int* err, unsigned int code) {
  atomicOr(err, code);
  unsigned int* mirror = *reinterpret_cast<unsigned int* volatile*>(err + 2);
  if (mirror != nullptr) {
    *reinterpret_cast<volatile unsigned int*>(mirror) = 1u;
    __threadfence_system();
  }
}

__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, Abort ab,
                                           unsigned int code, uint64_t limit_ns) {
  const uint64_t t0 = ptx::global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*ab.flag) return false;
    // The device-wide error word and the clock are read only now and then:
    // a global load in the loop would delay noticing the phase change.
    if ((n & 255u) == 0) {
      if (*reinterpret_cast<volatile unsigned int*>(ab.err) != 0) {
        *ab.flag = 1;   // another block already gave up: stop early
        return false;
      }
      if (ptx::global_timer_ns() - t0 > limit_ns) {
        *ab.flag = 1;
        raise_error(ab.err, code);
        return false;
      }
    }
  }
}

// Bounded wait for the phase of `bar` with the given parity.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Abort ab, unsigned int code,
                                         uint64_t limit_ns = kWaitTimeoutNs) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, ab, code, limit_ns);
}

// Wait used on the abort path: ignores the abort flag, shorter limit.
__device__ __noinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::global_timer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::global_timer_ns() - t0 > kDrainTimeoutNs) return false;
  }
  return true;
}

}  // namespace
}  // namespace ra
