// tc_common.cuh — helpers shared by the tensor-core chunkwise kernels: packed
// bf16 conversions and hi/lo splits, TMEM column loads, warp-level TF32x3 tile
// products for the blocks of the triangular inverse, and the TMA tensor-map
// encoder for [B, T, H, d] bf16 tensors.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "umma.cuh"

namespace dr {
namespace tc {

using namespace umma;

// two floats -> packed bf16x2 (round to nearest even), one conversion instruction
static __device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 8 consecutive bf16 (one 16-byte chunk) -> float
static __device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

static __device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                    pack_bf16(f[6], f[7]));
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), 8 values, packed conversions
static __device__ __forceinline__ void split8(const float (&x)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = pack_bf16(x[2 * i], x[2 * i + 1]);
    const float r0 = x[2 * i] - __uint_as_float(h[i] << 16);
    const float r1 = x[2 * i + 1] - __uint_as_float(h[i] & 0xFFFF0000u);
    l[i] = pack_bf16(r0, r1);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// ---- warp-level tensor-core products for the 16/32-row blocks of the triangular
// inverse (below tcgen05's minimum M).  m16n8k8 TF32 with each operand split into
// two TF32 terms (a = a_hi + a_lo) and three products, which keeps fp32 accuracy.
static __device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

static __device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32"
      " {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// D (16 x 8 tile, fp32 fragment) += A[m0.., k0..k0+K) * B[k0.., n0..] over K in steps of 8.
// A, B are fp32 row-major in shared memory with leading dimensions lda, ldb.
template <int KSTEPS>
static __device__ __forceinline__ void tile_mm3(float (&d)[4], const float* A, int lda, const float* B,
                                         int ldb, int lane) {
  const int g = lane >> 2, t = lane & 3;
  float dc[4] = {0.f, 0.f, 0.f, 0.f};   // correction terms, an independent accumulation chain
#pragma unroll
  for (int ks = 0; ks < KSTEPS; ++ks) {
    const float* a = A + 8 * ks;
    const float* bb = B + 8 * ks * ldb;
    const float af[4] = {a[g * lda + t], a[(g + 8) * lda + t], a[g * lda + t + 4],
                         a[(g + 8) * lda + t + 4]};
    const float bf[2] = {bb[t * ldb + g], bb[(t + 4) * ldb + g]};
    uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ah[i] = to_tf32(af[i]);
      al[i] = to_tf32(af[i] - __uint_as_float(ah[i]));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      bh[i] = to_tf32(bf[i]);
      bl[i] = to_tf32(bf[i] - __uint_as_float(bh[i]));
    }
    mma_tf32(dc, al, bh);
    mma_tf32(dc, ah, bl);
    mma_tf32(d, ah, bh);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] += dc[i];
}

// The same 16 x 8 tile product with each operand split into bf16 hi + lo and
// m16n8k16 products (K = 16 per step, half the instructions of the TF32 form;
// KSTEPS8 counts 8-wide steps and is even).  A lane's k slots (2t, 2t+1, 2t+8,
// 2t+9) hold k0 + t + (0, 4, 8, 12) in A and B alike (a sum over k is order-free),
// so it reads the addresses of two 8-wide steps.
static __device__ __forceinline__ void bsplit2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x0, x1);
  lo = pack_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xFFFF0000u));
}
static __device__ __forceinline__ void mma_b16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32"
      " {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
template <int KSTEPS8>
static __device__ __forceinline__ void tile_mm3b(float (&d)[4], const float* A, int lda, const float* B,
                                          int ldb, int lane) {
  static_assert(KSTEPS8 % 2 == 0, "K must be a multiple of 16");
  const int g = lane >> 2, t = lane & 3;
  float dc[4] = {0.f, 0.f, 0.f, 0.f};   // correction terms, an independent accumulation chain
#pragma unroll
  for (int ks = 0; ks < KSTEPS8 / 2; ++ks) {
    const int k0 = 16 * ks + t;
    uint32_t ah[4], al[4], bh[2], bl[2];
    bsplit2(A[g * lda + k0], A[g * lda + k0 + 4], ah[0], al[0]);
    bsplit2(A[(g + 8) * lda + k0], A[(g + 8) * lda + k0 + 4], ah[1], al[1]);
    bsplit2(A[g * lda + k0 + 8], A[g * lda + k0 + 12], ah[2], al[2]);
    bsplit2(A[(g + 8) * lda + k0 + 8], A[(g + 8) * lda + k0 + 12], ah[3], al[3]);
    bsplit2(B[k0 * ldb + g], B[(k0 + 4) * ldb + g], bh[0], bl[0]);
    bsplit2(B[(k0 + 8) * ldb + g], B[(k0 + 12) * ldb + g], bh[1], bl[1]);
    mma_b16816(dc, al, bh);
    mma_b16816(dc, ah, bl);
    mma_b16816(d, ah, bh);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] += dc[i];
}

// store a 16 x 8 fp32 fragment (scaled by s) at C[m0.., n0..]
static __device__ __forceinline__ void tile_store(float* C, int ldc, const float (&d)[4], float s, int lane) {
  const int g = lane >> 2, t = lane & 3;
  C[g * ldc + 2 * t] = s * d[0];
  C[g * ldc + 2 * t + 1] = s * d[1];
  C[(g + 8) * ldc + 2 * t] = s * d[2];
  C[(g + 8) * ldc + 2 * t + 1] = s * d[3];
}

static __device__ __forceinline__ void ld32cols(uint32_t taddr, float (&v)[32]) {
  float t16[16];
  tmem_ld16(taddr, t16);
#pragma unroll
  for (int e = 0; e < 16; ++e) v[e] = t16[e];
  tmem_ld16(taddr + 16, t16);
#pragma unroll
  for (int e = 0; e < 16; ++e) v[16 + e] = t16[e];
}


// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static inline EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [B, T, H, d] bf16 tensor, box of 64 features x 1 head x 64 tokens x 1 batch, 128B swizzle.
static inline bool make_map(CUtensorMap* m, const void* ptr, int B, int T, int H, int d) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, (cuuint64_t)T * H * d * 2};
  cuuint32_t box[4] = {64, 1, 64, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B, T, H, 128] fp32 tensor (per-channel gates), box of 128 features x 1 head x
// 64 tokens x 1 batch without swizzle: lands as a row-major [64][128] fp32 tile
// (32 KB); tokens past the end read as zero.
static inline bool make_map_f32(CUtensorMap* m, const void* ptr, int B, int T, int H) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[4] = {128, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {512, (cuuint64_t)H * 512, (cuuint64_t)T * H * 512};
  cuuint32_t box[4] = {128, 1, 64, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(ptr), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace dr
