// chain.cuh -- hand-over of a per-channel value between the tasks of one
// persistent kernel (a sequential chain across chunks inside a parallel prep).
#pragma once

#include "dr_common.cuh"

namespace dr {

// ---- chains between the tasks of one prep kernel: a task hands a per-channel
// value at its chunk end to the next chunk's task through the workspace and
// raises that task's flag (GPU-scope release); the next task waits for it.
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Waits until *flag != 0 or *abort != 0, at most limit_ns of global-timer time.
// Returns false (and raises *abort, so every other waiter returns at once) when
// the flag did not arrive.
__device__ __forceinline__ bool chain_wait(const uint32_t* flag, uint32_t* abort, uint64_t limit_ns) {
  if (ld_acquire_gpu(flag)) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    if (ld_acquire_gpu(flag)) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (ld_acquire_gpu(abort) || t - t0 > limit_ns) {
      atomicExch(abort, 1u);
      return false;
    }
    __nanosleep(64);
  }
}
// Test hooks of the hand-over (set by dr_set_chain_fault_for_testing): the limit of
// a task's wait for its flag, and the index of one flag that is never raised (-1:
// none), so a test can make a wait run out on a flag that nothing sets.
extern __device__ unsigned long long g_chain_wait_ns;
extern __device__ long long g_chain_withhold;

// bytes after the records: one flag per record, the ticket counter, the abort word
__host__ __device__ inline size_t chain_bytes(long nrec) { return ((size_t)(nrec + 2) * 4 + 255) / 256 * 256; }

}  // namespace dr
