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
  // backward only (null otherwise): the carry of the scalar-decay two-phase path
  // saves the state at every chunk start [B H NC][dk][dv] and the chunk's E
  // [B H NC][64][dv] (fp32), and a null `out` skips the output stores
  float* save_S;
  float* save_E;
  // backward only: the per-channel-decay prep saves every chunk's write vectors
  // w [B H NC][64][dk] (fp32; zero on padding rows)
  float* save_W;
  // segment-parallel carry (scalar-decay two-phase path, few rows and many
  // chunks): 0 = whole rows; 1 = first pass (segment 0 with its outputs, and
  // every middle segment's zero-start state and transition map); 2 = replay of
  // segments 1 .. G-1 from their composed start states.  seg_buf holds per
  // (row, segment) the end state from zero (or segment 0's true end state), the
  // transition map and the start state, each [dk][dv] fp32.
  int seg_pass, seg_G, seg_len;
  float* seg_buf;
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

}  // namespace dr
