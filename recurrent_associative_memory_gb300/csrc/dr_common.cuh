// dr_common.cuh — argument block, device status word and small device helpers
// shared by the libdr kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/dr.h"

namespace dr {

// Everything a forward/decode kernel needs, passed by value.
struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* log_alpha;
  const float* eta;
  const float* alphaP;
  const float* betaP;
  const float* mu;
  const float* omega;
  const float* r;
  const float* S0;        // chunk fwd: init state (nullable)
  float* S;               // chunk fwd: final state (nullable); decode: state in/out
  const float* aux0;      // chunk fwd: aux init (nullable)
  float* aux;             // chunk fwd: aux final (nullable); decode: aux in/out
  void* out;
  int B, T, H, dk, dv, chunk;
  int variant;
  int q_l2norm, k_l2norm;
  int check_finite;
  float eps;
  float ln_x;             // ln(x) of the PGDN bound
  float log_floor;
  float info_scale;
};

// Sticky device status: the first non-OK code written stays until read.
extern __device__ int g_status;

__device__ __forceinline__ void set_status(int code) { atomicCAS(&g_status, 0, code); }

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ bool finite_f(float x) { return isfinite(x); }

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
// bytes after the records: one flag per record, the ticket counter, the abort word
__host__ __device__ inline size_t chain_bytes(long nrec) { return ((size_t)(nrec + 2) * 4 + 255) / 256 * 256; }

}  // namespace dr
