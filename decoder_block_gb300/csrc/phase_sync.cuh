// How a kernel body waits for data that earlier work on the GPU wrote.
//
// The tensor-core kernel bodies (GEMM, decode attention) run either as kernels
// of their own or as phases of the fused decode-step kernel:
//   - kernel of its own (PhaseSync{}, fused() false): the body waits for the
//     previous kernel of the stream (programmatic dependent launch, see
//     grid_dependency_wait in common.cuh) and allocates its own TMEM;
//   - phase of the fused kernel: a cooperative launch, so every CTA is resident
//     at once.  A CTA that has finished phase k adds one arrival to a grid-wide
//     counter; phase k + 1 may read phase k's results once the counter reaches
//     (k + 1) x gridDim.x.  The fused kernel allocates TMEM once for all phases.
// Results of one phase are written with ordinary stores and read by the next
// through TMA (the async proxy), so both sides fence the proxies: the writers
// before their arrival, the reader after its acquire.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace llama {

struct PhaseSync {
  unsigned *arrivals = nullptr;  // fused kernel: [0] phase arrivals, [1] abort word (both zero at launch)
  unsigned target = 0;           // arrivals that complete the phases this one reads
  uint32_t tmem = 0;             // fused kernel: the TMEM columns allocated for every phase
  __host__ __device__ bool fused() const { return arrivals != nullptr; }
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

// One thread.  Returns once the inputs of this phase are complete and visible
// (also to TMA loads issued afterwards by this thread); false if the wait gave
// up (budget spent, recorded as DEV_TIMEOUT_PHASE, or another CTA gave up).
__device__ __forceinline__ bool phase_wait(const PhaseSync &s, int *status) {
  if (!s.fused()) {
    grid_dependency_wait();
    return true;
  }
  const long long t0 = clock64();
  const long long budget = wait_budget(status);
  while (ld_acquire_gpu(s.arrivals) < s.target) {
    if (*(volatile unsigned *)(s.arrivals + 1) != 0u) return false;
    if (clock64() - t0 > budget) {
      report_status(status, DEV_TIMEOUT_PHASE);
      atomicExch(s.arrivals + 1, 1u);
      return false;
    }
    __nanosleep(64);
  }
  fence_proxy_async_all();
  return true;
}

// One warp: lane 0 waits, the warp learns the outcome (and is ordered after the
// acquire through __syncwarp).
__device__ __forceinline__ bool phase_wait_warp(const PhaseSync &s, int *status) {
  if (!s.fused()) {
    grid_dependency_wait();
    return true;
  }
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = phase_wait(s, status) ? 1 : 0;
  __syncwarp();
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Fused kernel, end of a phase: every thread calls this; once the whole CTA is
// done, thread 0 publishes the CTA's arrival.
__device__ __forceinline__ void phase_arrive(const PhaseSync &s) {
  fence_proxy_async_all();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // cumulative over the CTA's writes ordered before it by __syncthreads
    atomicAdd(s.arrivals, 1u);
  }
}

}  // namespace llama
