// Bounded waits shared by the library's tcgen05 kernels (one copy per
// translation unit: each has its own status word and reads it back with its
// own host function).
//
// No wait on the chip spins forever: each has a time budget, after which the
// kernel records 0x100 | site in the status word, sets the CTA's abort flag
// (the other warps then give up at their next wait) and returns.
#pragma once

#include <stdint.h>

#include "ra_ptx.cuh"

namespace ra {
namespace {

// First failure of a kernel of this translation unit since the last read.
__device__ int g_ra_device_error = 0;

// Wait sites shared by all kernels.
enum : int { kSiteDrain = 9 };

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_ra_device_error, 0, code); }

// Bounded wait on an mbarrier phase. Returns false (and stops the CTA) when the
// budget runs out or another warp already gave up. Each try may sleep up to
// 1 ms until the phase completes, so a waiting warp does not take issue slots
// from the warps that share its scheduler; the clock is read only after an
// unsuccessful try.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned long long budget, int site) {
  if (ptx::mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
  const unsigned long long t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer() - t0 > budget) {
      *abort_flag = 1;
      record_error(0x100 | site);
      return false;
    }
  }
}

// Warp-uniform version: every lane waits, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long budget, int site) {
  const bool ok = wait_bar(bar, parity, abort_flag, budget, site);
  return __all_sync(0xffffffffu, ok);
}

// Polling version of warp_wait: the warp tests the phase without ever
// sleeping, so it sees the completion at once, at the price of the issue slots
// its polls take from the warps that share its scheduler. The clock and the
// abort flag are read every 256 polls.
__device__ __forceinline__ bool warp_wait_spin(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               unsigned long long budget, int site) {
  bool ok = true;
  if (!ptx::mbar_test_wait(bar, parity)) {
    const unsigned long long t0 = ptx::globaltimer();
    for (uint32_t k = 1;; ++k) {
      if (ptx::mbar_test_wait(bar, parity)) break;
      if ((k & 255u) == 0) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (ptx::globaltimer() - t0 > budget) {
          *abort_flag = 1;
          record_error(0x100 | site);
          ok = false;
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// Wait used while tearing down after an abort: ignores the abort flag and
// has its own generous budget (copies and MMAs already issued always finish;
// the CTA must not exit before they do, whatever the normal wait budget is).
constexpr unsigned long long kDrainBudgetNs = 2000000000ull;

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned long long) {
  const unsigned long long t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kDrainBudgetNs) {
      record_error(0x100 | kSiteDrain);
      return;
    }
  }
}

}  // namespace
}  // namespace ra
