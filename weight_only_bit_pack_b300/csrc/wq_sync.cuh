// Bounded waits shared by the kernels that synchronise warps, CTAs or clusters
// through mbarriers and global counters. No wait in this library spins
// forever: after kWaitBudget cycles (about two seconds) the waiting thread
// records WQ_ERR_DEVICE_TIMEOUT and the place that gave up in the workspace
// status word, raises the CTA's abort flag and returns false, so the kernel can
// skip the dependent work and exit with the CUDA context intact.
#pragma once

#include <cstdint>

#include "../../include/wq.h"
#include "wq_sm100.cuh"

namespace wq {

constexpr long long kWaitBudget = 4000000000LL;  // clock64 cycles

__device__ __forceinline__ void record_timeout(uint32_t *status, uint32_t where) {
  atomicOr(status, (uint32_t)WQ_ERR_DEVICE_TIMEOUT | (where << 8));
}

// Bounded wait on an mbarrier phase; gives up when another role aborted or the
// budget ran out (then it aborts the CTA and records where).
// Longest suspension of one wait attempt while draining (1 ms). Waits on the
// critical path poll instead: a suspended warp resumes too late.
constexpr uint32_t kSleepNs = 1000000;

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         uint32_t *status, uint32_t where,
                                         long long budget = kWaitBudget) {
  if (sm100::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (sm100::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      *abort_flag = 1;
      record_timeout(status, where);
      return false;
    }
  }
}

// Warp-collective form: every lane polls (each gets the barrier's acquire) and
// the warp takes one decision, so no lane leaves a loop its warp-mates stay in.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              uint32_t *status, uint32_t where) {
  const bool ok = wait_bar(bar, parity, abort_flag, status, where);
  return __all_sync(0xffffffffu, ok);
}

// Wait used only while draining: ignores the abort flag, bounded budget.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!sm100::mbar_try_wait_sleep(bar, parity, kSleepNs)) {
    if (clock64() - t0 > kWaitBudget) return;
  }
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

}  // namespace wq
