// chunk_simt.cu — fused chunkwise forward on fp32 CUDA cores (all variants).
//
// One CTA of 256 threads owns one (b, h, 32-column slice of dv) and walks the
// sequence in 64-token chunks (results are chunk-size invariant), keeping its
// dk x 32 slice of S in shared memory.  Within a chunk (KLA notes section 2.5,
// Eqs. (7)-(9), generalised to a write matrix W as in the PDN notes section 2.6):
//
//   prep   k^, q^ (optional L2 norm, fused into the loads), cumulative log-decay
//          g, write vectors W (GDN/KLA scalars; PGDN statistic scan; KDN
//          variance scan in homogeneous Moebius form, carried across chunks)
//   Gram   L = strict_lower((K W^T) . exp(g_i - g_j)),  P = lower((Q W^T) . exp(...))
//   solve  T = (I + L)^-1: 16x16 diagonal blocks by forward substitution,
//          off-diagonal blocks by recursive doubling (fp32-accurate TF32x3 tiles)
//   carry  R = V - (Gamma.K) S ;  E = T R ;  O = (Gamma.Q) S + P E
//          S <- diag(gamma_C) S + (exp(g_C - g_j).W)^T E
//
// Decay ratios are always formed from log differences (KDN notes section 6,
// numerics).  With per-channel decay (KDN) the Gram cannot factor as a single
// matrix product; the chunk is cut into 16-token sub-chunks and each block
// (I, J) of the Gram uses a reference point with every factor bounded:
//   J < I : k_i exp(g_i - g_b) * w_j exp(g_e(J) - g_j) * exp(g_b - g_e(J)),
//           b = last token of sub-chunk I-1, e(J) = last token of sub-chunk J
//           (all three factors <= 1);
//   J = I : the same with the mid token of the sub-chunk as reference, so the
//           two growing factors stay below exp(decay over 8 tokens).
// This path serves the fp32 mode (tolerance 1e-4), per-channel decay and the
// shapes the tensor-core kernels do not take.
//
// Two-phase per-channel decay with fp32 inputs (dk = dv = 128, chunk 64, with a
// workspace): the same kernel in prep mode (PREP = true) does every chunk's local
// work in parallel and writes an fp32 per-chunk record for kdn_carry_kernel (CUDA
// cores); bf16 inputs take chunk_tc_pc.cu's tensor-core prep and the tcgen05
// carry, with the same chains and variance maps.  Only the variance p at the chunk start is
// sequential across chunks.  With many (b, h) rows the prep chains it itself:
// tasks are taken in chunk-major ticket order and each one hands p at its end to
// the next chunk of its row through the workspace (a release flag; the wait is
// bounded), which costs each CTA only a one-off phase lag.  With few rows the
// chain would serialise the CTAs, so kdn_map_kernel first builds each chunk's
// variance map (a 2x2 Moebius product) and kdn_scan_kernel composes them into p
// at every chunk start.
#include "dr_common.cuh"
#include "tc_common.cuh"
#include "chain.cuh"

namespace dr {

namespace {

using tc::tile_mm3;
using tc::tile_store;

constexpr int kThreads = 256;
constexpr int CM = 64;      // chunk handled on chip
constexpr int NV = 32;      // dv columns per CTA
constexpr int CS = CM + 4;  // row stride of token-minor (transposed) buffers
constexpr int LDL = 68;     // row stride of the row-major L/T buffer
constexpr int LDX = 36;     // row stride of the inverse scratch
constexpr int NSM = CM / 16;

template <int DK>
struct SimtSmem {
  static constexpr int kKt = DK * CS;            // K^T [DK][CS] (k^, then scaled copies)
  static constexpr int kQt = DK * CS;            // Q^T [DK][CS]
  static constexpr int kWt = DK * CS;            // W^T [DK][CS] for the Gram; later T^T [CM][CS]
  static constexpr int kW = CM * DK;             // W   [CM][DK], later exp(g_C - g_j).W
  static constexpr int kS = DK * NV;             // S   [DK][NV]
  static constexpr int kV = CM * NV;             // V, then R, then E  [CM][NV]
  static constexpr int kP = CM * CS;             // P^T [CM][CS]
  static constexpr int kLT = CM * LDL + 32 * LDX;          // L/T row-major + inverse scratch
  static constexpr int kX = (CM * DK > kLT) ? CM * DK : kLT;  // KDN per-channel g | L/T
  static constexpr int kF = (6 + 4 * NSM) * DK;  // KDN decay factor vectors
  static constexpr int kVec = 8 * CM + 2 * DK;
  static constexpr int total = kKt + kQt + kWt + kW + kS + kV + kP + kX + kF + kVec;
  static_assert(kWt >= CM * CS, "T^T aliases W^T");
};

__device__ __forceinline__ long tok_index(const FwdArgs& a, int b, int t, int h) {
  return ((long)b * a.T + t) * a.H + h;
}

// read-only global loads (ld.global.nc), so the compiler may keep many in flight
template <typename Tin>
__device__ __forceinline__ float ldg_in(const void* p, long i);
template <>
__device__ __forceinline__ float ldg_in<float>(const void* p, long i) {
  return __ldg(static_cast<const float*>(p) + i);
}
template <>
__device__ __forceinline__ float ldg_in<__nv_bfloat16>(const void* p, long i) {
  const unsigned short u = __ldg(static_cast<const unsigned short*>(p) + i);
  return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 zero-fills the destination
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}


// m16n8k16 bf16 mma.sync, fp32 accumulate (the bf16-input Gram's split products)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32"
      " {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// (x0, x1) -> packed bf16x2 hi = bf16(x) and lo = bf16(x - hi)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = tc::pack_bf16(x0, x1);
  lo = tc::pack_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xFFFF0000u));
}

// index of the (I, J) pair, J < I, among the 6 strictly lower sub-chunk pairs
__device__ __forceinline__ int pair_index(int I, int J) { return I * (I - 1) / 2 + J; }

// ---- per-chunk record of the two-phase Diagonal KDN path (fp32, bytes; dk = dv = 128)
constexpr uint32_t rkT = 0;          // T = (I + L)^-1, row-major [64][64]
constexpr uint32_t rkP = 16384;      // P^T [64 j][64 i]
constexpr uint32_t rkK = 32768;      // (Gamma.K)^T [128 c][64 i]
constexpr uint32_t rkQ = 65536;      // (Gamma.Q)^T [128 c][64 i]
constexpr uint32_t rkW = 98304;      // (exp(g_C - g_j).w_j) [64 j][128 c]
constexpr uint32_t rkG = 131072;     // gamma_C [128]
constexpr uint32_t rkMap = 132096;   // variance chunk map, 4 floats per channel
constexpr uint32_t rkP0 = 134144;    // variance p at the chunk start [128]
constexpr uint32_t kRecK = 135168;
// (bf16 inputs take the tensor-core prep of chunk_tc_pc.cu, whose records of the
// same size hold bf16 hi/lo tile images for the tcgen05 carry; the variance map
// and the chain fields below are shared.)

// PREP = false: the fused forward, one CTA per (b, h, 32 columns), chunks in order.
// PREP = true (Diagonal KDN, dk = 128): one task per (b, h, chunk), all chunks in
// parallel; the chunk's carry operands are written to the record instead of being
// used.  The variance at the chunk start is read from the record (written by
// kdn_scan_kernel) when chain is null.  Otherwise chain holds one flag per record,
// then the ticket counter and the abort word, all zero at launch: tasks are taken
// by ticket in chunk-major order, a task waits for its flag, reads p from its
// record and hands p at its end to the next chunk's record (then raises that
// chunk's flag); the last chunk of a row writes p to aux.  A task only waits on
// tickets claimed earlier by running CTAs, so the chain needs no co-residency.
// The wait for a flag gives up after g_chain_wait_ns (2 s by default: a lost flag,
// not a slow one), sets DR_ERR_TIMEOUT and the abort word, which releases every
// other waiter at once; the tasks then run to their ends on whatever the record
// holds, so the kernel always finishes.

template <int DK, typename Tin, bool PREP>
__global__ void __launch_bounds__(kThreads, 1) chunk_simt_kernel(FwdArgs a, uint8_t* __restrict__ ws,
                                                                 uint32_t* __restrict__ chain) {
  using SM = SimtSmem<DK>;
  constexpr int TPR = DK / 8;                // threads per token row in the load pass
  constexpr int RPP = kThreads / TPR;        // rows per load pass
  extern __shared__ __align__(16) float sm[];
  float* sKt = sm;
  float* sQt = sKt + SM::kKt;
  float* sWt = sQt + SM::kQt;
  float* sTt = sWt;                          // T^T aliases W^T (dead after the Gram)
  float* sW = sWt + SM::kWt;
  float* sS = sW + SM::kW;
  float* sV = sS + SM::kS;
  float* sPt = sV + SM::kV;
  float* sX = sPt + SM::kP;                  // KDN g [CM][DK], then L/T [CM][LDL] + scratch
  float* sLT = sX;
  float* sXS = sX + CM * LDL;
  float* sF = sX + SM::kX;
  float* sg = sF + SM::kF;        // [CM] scalar cumulative log-decay
  float* sb1 = sg + CM;           // [CM] beta (GDN/KLA), eta (PGDN), r (KDN)
  float* sb2 = sb1 + CM;          // [CM] alphaP
  float* sb3 = sb2 + CM;          // [CM] betaP
  float* sz = sb3 + CM;           // [CM] KDN sum p^ k^2
  float* sgC = sz + CM;           // [DK] gamma_C per channel (scalar: [0])
  float* sOne = sgC + DK;         // [DK] ones (neutral factor vector)

  const int ntile = a.dv / NV;
  const int NCk = (a.T + CM - 1) / CM;
  const int tile = PREP ? 0 : (int)(blockIdx.x % ntile);
  int bh = PREP ? 0 : (int)(blockIdx.x / ntile);
  int b = bh / a.H, h = bh % a.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool kdn = (a.variant == DR_KDN);
  const bool pgdn = (a.variant == DR_PGDN);
  const bool kda = (a.variant == DR_KDA);
  const bool pkda = (a.variant == DR_PKDA);
  const bool ikdn = (a.variant == DR_IKDN);  // isotropic KDN: one variance per head
  const bool perchan = kdn || kda || pkda || ikdn;   // per-channel decay D = diag(alpha)
  const bool pstat = pgdn || pkda;           // the PGDN key statistic and write key
  // W is formed explicitly (not as a per-row multiple of K in the Gram's readout)
  const bool explicit_w = perchan || pgdn;

  // KDN factor vectors inside sF
  float* fOff = sF;                       // [6][DK]   exp(g_b(I) - g_e(J)), J < I
  float* fDa = fOff + 6 * DK;             // [NSM][DK] exp(g_b(I) - g_m(I))
  float* fDb = fDa + NSM * DK;            // [NSM][DK] exp(g_m(I) - g_e(I))
  float* fGb = fDb + NSM * DK;            // [NSM][DK] exp(g_b(I))  (b(0): chunk start)

  if (!PREP) {
    for (int e = tid; e < DK * NV; e += kThreads) {
      const int c = e / NV, n = e % NV;
      sS[e] = a.S0 ? a.S0[((long)bh * DK + c) * a.dv + tile * NV + n] : 0.f;
    }
  }
  if (tid < DK) sOne[tid] = 1.f;
  // per-channel carried gain state (PGDN A / KDN p), held by the thread that
  // scans channel my_c: threads 32.. for PGDN (warp 0 scans the decay), 0.. for KDN
  const int my_c = pgdn ? tid - 32 : tid;
  float carry = 0.f;
  if (my_c >= 0 && my_c < DK) {
    if (pstat) carry = a.aux0 ? a.aux0[(long)bh * DK + my_c] : 0.f;
    if (kdn) carry = a.aux0 ? a.aux0[(long)bh * DK + my_c] : 1.f;
  }
  if (ikdn && tid == DK) carry = a.aux0 ? a.aux0[bh] : 1.f;   // isotropic KDN: thread DK holds b
  const float mu_h = pstat ? a.mu[h] : 0.f;
  bool bad = false;

  const long kIters = PREP ? (long)a.B * a.H * NCk : NCk;
  const bool chained = PREP && chain != nullptr;
  __shared__ long s_ticket;   // chained prep: the task after this one (claimed one ahead)
  long it0 = PREP ? blockIdx.x : 0;
  if (chained) {
    if (tid == 0) s_ticket = atomicAdd(chain + kIters, 1u);
    __syncthreads();
    it0 = s_ticket;
  }
  for (long it = it0; it < kIters; it = chained ? s_ticket : it + (PREP ? gridDim.x : 1)) {
    int t0 = (int)it * CM;
    int ci = 0;       // chunk of a prep task
    long ri = 0;      // its record
    uint8_t* rec = nullptr;
    if (PREP) {   // task (b h, chunk)
      if (chained) {
        ci = (int)(it / (a.B * a.H));
        bh = (int)(it % (a.B * a.H));
      } else {
        bh = (int)(it / NCk);
        ci = (int)(it % NCk);
      }
      b = bh / a.H;
      h = bh % a.H;
      t0 = ci * CM;
      ri = (long)bh * NCk + ci;
      rec = ws + (size_t)ri * kRecK;
      if (!chained && tid < DK) carry = reinterpret_cast<const float*>(rec + rkP0)[tid];
    }
    const int Cc = min(CM, a.T - t0);
    __syncthreads();
    if (chained && tid == 0) s_ticket = atomicAdd(chain + kIters, 1u);

    if (perchan) {   // per-channel log-decay (and KDN process noise), row-major [i][c],
                     // copied asynchronously (16-byte pieces, zero past the end) under the loads
      constexpr int kPieces = CM * DK / 4;   // 16-byte pieces per array
#pragma unroll
      for (int r = 0; r < kPieces / kThreads; ++r) {
        const int e4 = tid + r * kThreads, i = (4 * e4) / DK, c = (4 * e4) % DK;
        const bool real = i < Cc;
        const long ti = (real ? tok_index(a, b, t0 + i, h) : tok_index(a, b, 0, h)) * DK + c;
        cp_async16(sX + 4 * e4, a.log_alpha + ti, real ? 16 : 0);
        if (kdn) cp_async16(sW + 4 * e4, a.omega + ti, real ? 16 : 0);
      }
    }

    // ---- 1. per-token scalars (rows Cc..CM-1 are padding: zero inputs, no decay)
    if (tid < CM) {
      const int i = tid;
      const bool real = i < Cc;
      const long ti = real ? tok_index(a, b, t0 + i, h) : 0;
      if (ikdn) {   // r, omega (scalar per token); ||k^||^2 comes with the key loads
        sb1[i] = real ? a.r[ti] : 1.f;
        sb2[i] = real ? a.omega[ti] : 0.f;
      } else if (!kdn) {
        if (!perchan) sg[i] = real ? a.log_alpha[ti] : 0.f;
        sb1[i] = real ? a.eta[ti] : 0.f;
      } else {
        sb1[i] = real ? a.r[ti] : 1.f;
        sb2[i] = a.info_scale / sb1[i];   // information scale over r, used by the variance scan
      }
      if (pstat) {
        sb2[i] = real ? a.alphaP[ti] : 1.f;
        sb3[i] = real ? a.betaP[ti] : 0.f;
      }
    }
    __syncthreads();

    // ---- 2. loads of K, Q with fused L2 norms; thread (row i, sub) holds channels
    //         sub + TPR e, so the transposed stores hit distinct banks
    {
      const int sub = tid % TPR;
      constexpr int kPasses = CM / RPP;
      float kvp[kPasses][8], qvp[kPasses][8];   // every pass's loads in flight first
#pragma unroll
      for (int pz = 0; pz < kPasses; ++pz) {
        const int i = pz * RPP + tid / TPR;
        const bool real = i < Cc;
        const long base = real ? tok_index(a, b, t0 + i, h) * DK : 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          kvp[pz][e] = real ? ldg_in<Tin>(a.k, base + sub + TPR * e) : 0.f;
          qvp[pz][e] = real ? ldg_in<Tin>(a.q, base + sub + TPR * e) : 0.f;
        }
      }
#pragma unroll
      for (int pz = 0; pz < kPasses; ++pz) {
        const int i = pz * RPP + tid / TPR;
        const bool real = i < Cc;
        const float* kv = kvp[pz];
        const float* qv = qvp[pz];
        float kk = 0.f, qq = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          kk += kv[e] * kv[e];
          qq += qv[e] * qv[e];
        }
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) {
          kk += __shfl_xor_sync(0xffffffffu, kk, o);
          qq += __shfl_xor_sync(0xffffffffu, qq, o);
        }
        const float kn = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
        const float qn = a.q_l2norm ? 1.f / fmaxf(sqrtf(qq), 1e-30f) : 1.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = sub + TPR * e;
          sKt[c * CS + i] = kv[e] * kn;
          sQt[c * CS + i] = qv[e] * qn;
          if (!explicit_w) sW[i * DK + c] = kv[e] * kn;
        }
        if (sub == 0 && real && a.variant == DR_KLA) sb1[i] = sb1[i] / (kk * kn * kn + a.eps);
        if (sub == 0 && ikdn) sb3[i] = kk * kn * kn;   // ||k^||^2 (0 on padding rows)
      }
    }
    if (!PREP) {
      float vv[CM * NV / kThreads];
#pragma unroll
      for (int r = 0; r < CM * NV / kThreads; ++r) {   // all loads in flight, then the stores
        const int e = tid + r * kThreads, i = e / NV, n = e % NV;
        vv[r] = (i < Cc) ? ldg_in<Tin>(a.v, tok_index(a, b, t0 + i, h) * a.dv + tile * NV + n) : 0.f;
      }
#pragma unroll
      for (int r = 0; r < CM * NV / kThreads; ++r) sV[tid + r * kThreads] = vv[r];
    }
    if (perchan) cp_async_wait_all();
    if (chained && ci > 0 && tid == 0 && !chain_wait(chain + ri, chain + kIters + 1, g_chain_wait_ns))
      set_status(DR_ERR_TIMEOUT);
    __syncthreads();
    if (chained && (ikdn ? tid == DK : tid < DK))   // KDN p / PKDA A (thread c) or IKDN b
      // (thread DK) at the chunk start: the row's initial value (default 1 / 0 / 1), or
      // the previous chunk's
      carry = ci == 0 ? (a.aux0 ? a.aux0[ikdn ? (long)bh : (long)bh * DK + tid] : (pkda ? 0.f : 1.f))
                      : __ldcg(reinterpret_cast<const float*>(rec + rkP0) + (ikdn ? 0 : tid));

    // ---- 3. cumulative decay and write vectors
    if (!perchan) {
      if (warp == 0) {  // inclusive scan of log-alpha over 64 tokens, 2 per lane
        const float x0 = sg[2 * lane], x1 = sg[2 * lane + 1];
        float s = x0 + x1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, s, o);
          if (lane >= o) s += y;
        }
        sg[2 * lane] = s - x1;
        sg[2 * lane + 1] = s;
      }
      if (pgdn && my_c >= 0 && my_c < DK) {  // statistic scan for channel c, 8 tokens per step
        const int c = my_c;
        float A = carry;
        for (int i0 = 0; i0 < CM; i0 += 8) {
          float kv[8], Av[8];
          const float4 k0 = *reinterpret_cast<const float4*>(sKt + c * CS + i0);
          const float4 k1 = *reinterpret_cast<const float4*>(sKt + c * CS + i0 + 4);
          kv[0] = k0.x; kv[1] = k0.y; kv[2] = k0.z; kv[3] = k0.w;
          kv[4] = k1.x; kv[5] = k1.y; kv[6] = k1.z; kv[7] = k1.w;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            A = sb2[i0 + e] * A + sb3[i0 + e] * kv[e] * kv[e];
            Av[e] = A;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float rr = logf(fmaxf(Av[e], a.log_floor)) - mu_h;
            const float s = __fdividef(rr, 1.f + fabsf(rr));
            const float w = sb1[i0 + e] * expf(-a.ln_x * s) * kv[e];
            sW[(i0 + e) * DK + c] = w;
            sWt[c * CS + i0 + e] = w;
          }
        }
        carry = A;
      }
      __syncthreads();
    } else if (ikdn) {
      // isotropic KDN (KDN notes section 7, Eq. (40)): the mean squared decay of
      // every token (warp w: tokens 8w .. 8w + 7), then channel c's cumulative
      // log-decay (thread c) while warp DK/32 scans the head's variance, then
      // w = beta k^.  The variance recursion b -> b^/(1 + u b^), b^ = a b + omega
      // is the Moebius map of (n, d) by M = [[a, omega], [u a, 1 + u omega]]
      // (b = n/d; the notes' remark that it is a 2x2 Moebius scan), so the warp
      // forms all 64 prefixes in parallel: two tokens' product per lane, then a
      // shuffle scan of 2x2 products, each rescaled by an exact power of two.
      {
        const int i0 = 8 * warp;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          float s2 = 0.f;
#pragma unroll
          for (int c = lane; c < DK; c += 32) s2 += __expf(2.f * sX[(i0 + r) * DK + c]);
          s2 = warp_sum(s2);
          if (lane == 0) sz[i0 + r] = s2 * (1.f / DK);
        }
      }
      __syncthreads();
      if (tid < DK) {
        const int c = tid;
        float g = 0.f;
        for (int i0 = 0; i0 < CM; i0 += 8) {
          float la[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) la[e] = sX[(i0 + e) * DK + c];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            g += la[e];
            sX[(i0 + e) * DK + c] = g;
          }
        }
      }
      if (warp == DK / 32) {
        auto mmul = [](const float (&A)[4], const float (&B)[4], float (&C)[4]) {
          C[0] = A[0] * B[0] + A[1] * B[2];
          C[1] = A[0] * B[1] + A[1] * B[3];
          C[2] = A[2] * B[0] + A[3] * B[2];
          C[3] = A[2] * B[1] + A[3] * B[3];
        };
        auto renorm = [](float (&C)[4]) {   // exact power-of-two rescale (b = n/d is scale-free)
          int ex;
          frexpf(fmaxf(fmaxf(fabsf(C[0]), fabsf(C[1])), fmaxf(fabsf(C[2]), fabsf(C[3]))), &ex);
#pragma unroll
          for (int z = 0; z < 4; ++z) C[z] = ldexpf(C[z], -ex);
        };
        auto token = [&](int i, float (&M)[4]) {
          const float at = sz[i], om = sb2[i], u = a.info_scale * sb3[i] / (DK * sb1[i]);
          M[0] = at; M[1] = om; M[2] = u * at; M[3] = 1.f + u * om;
        };
        float M0[4], M1[4], Pl[4];
        token(2 * lane, M0);
        token(2 * lane + 1, M1);
        mmul(M1, M0, Pl);   // tokens 2l, 2l + 1 (later factor on the left)
        renorm(Pl);
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {   // inclusive scan over lanes
          float Q[4], R[4];
#pragma unroll
          for (int z = 0; z < 4; ++z) Q[z] = __shfl_up_sync(0xffffffffu, Pl[z], d);
          if (lane >= d) {
            mmul(Pl, Q, R);
#pragma unroll
            for (int z = 0; z < 4; ++z) Pl[z] = R[z];
            renorm(Pl);
          }
        }
        const float b_in = __shfl_sync(0xffffffffu, carry, 0);
        float E[4];   // exclusive prefix: tokens 0 .. 2l - 1
#pragma unroll
        for (int z = 0; z < 4; ++z) E[z] = __shfl_up_sync(0xffffffffu, Pl[z], 1);
        if (lane == 0) { E[0] = 1.f; E[1] = 0.f; E[2] = 0.f; E[3] = 1.f; }
        const float n0 = E[0] * b_in + E[1], d0 = E[2] * b_in + E[3];
        const float b_prev = __fdividef(n0, d0);                    // b before token 2l
        const float bh0 = sz[2 * lane] * b_prev + sb2[2 * lane];
        const float n1 = M0[0] * n0 + M0[1] * d0, d1 = M0[2] * n0 + M0[3] * d0;
        const float b_mid = __fdividef(n1, d1);                     // b before token 2l + 1
        const float bh1 = sz[2 * lane + 1] * b_mid + sb2[2 * lane + 1];
        sz[2 * lane] = __fdividef(bh0, sb1[2 * lane] + bh0 * sb3[2 * lane]);
        sz[2 * lane + 1] = __fdividef(bh1, sb1[2 * lane + 1] + bh1 * sb3[2 * lane + 1]);
        const float nE = Pl[0] * b_in + Pl[1], dE = Pl[2] * b_in + Pl[3];
        const float b_end = __shfl_sync(0xffffffffu, __fdividef(nE, dE), 31);
        if (lane == 0) {
          carry = b_end;
          if (chained) {   // b at the chunk end -> the next chunk's record, or aux after the last
            if (ci + 1 < NCk) {
              __stcg(reinterpret_cast<float*>(rec + kRecK + rkP0), carry);
              __threadfence();
            } else if (a.aux) {
              a.aux[bh] = carry;
            }
          }
        }
      }
      __syncthreads();
      if (tid < DK) {
        const int c = tid;
        for (int i0 = 0; i0 < CM; i0 += 8) {
          const float4 k0 = *reinterpret_cast<const float4*>(sKt + c * CS + i0);
          const float4 k1 = *reinterpret_cast<const float4*>(sKt + c * CS + i0 + 4);
          const float kv[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
          float w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            w[e] = sz[i0 + e] * kv[e];
            sW[(i0 + e) * DK + c] = w[e];
          }
          *reinterpret_cast<float4*>(sWt + c * CS + i0) = make_float4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<float4*>(sWt + c * CS + i0 + 4) = make_float4(w[4], w[5], w[6], w[7]);
        }
      }
      __syncthreads();
    } else if (!kdn) {
      // KDA / PKDA: channel c's cumulative log-decay (thread c), then the write
      // vectors: eta k^ (KDA), or the PGDN statistic scan carried across chunks
      // and w = eta B(A) . k^ (PKDA)
      if (tid < DK) {
        const int c = tid;
        float g = 0.f;
        for (int i0 = 0; i0 < CM; i0 += 8) {
          float la[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) la[e] = sX[(i0 + e) * DK + c];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            g += la[e];
            sX[(i0 + e) * DK + c] = g;
          }
        }
        float A = carry;
        for (int i0 = 0; i0 < CM; i0 += 8) {
          const float4 k0 = *reinterpret_cast<const float4*>(sKt + c * CS + i0);
          const float4 k1 = *reinterpret_cast<const float4*>(sKt + c * CS + i0 + 4);
          const float kv[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
          float w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float scale = 1.f;
            if (pkda) {
              A = sb2[i0 + e] * A + sb3[i0 + e] * kv[e] * kv[e];
              // fast log / exp: ~1e-6 relative in B, far inside either tolerance
              const float rr = __logf(fmaxf(A, a.log_floor)) - (PREP ? a.mu[h] : mu_h);
              scale = __expf(-a.ln_x * __fdividef(rr, 1.f + fabsf(rr)));
            }
            w[e] = sb1[i0 + e] * scale * kv[e];
            sW[(i0 + e) * DK + c] = w[e];
          }
          *reinterpret_cast<float4*>(sWt + c * CS + i0) = make_float4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<float4*>(sWt + c * CS + i0 + 4) = make_float4(w[4], w[5], w[6], w[7]);
        }
        if (pkda) carry = A;
        if (chained) {   // A at the chunk end -> the next chunk's record, or aux after the last
                         // (the flag is raised below, after the barrier)
          if (ci + 1 < NCk) {
            __stcg(reinterpret_cast<float*>(rec + kRecK + rkP0) + c, carry);
            __threadfence();
          } else if (a.aux) {
            a.aux[(long)bh * DK + c] = carry;
          }
        }
      }
      __syncthreads();
    }
    if (perchan) {
      if (kdn && tid < DK) {
        // variance scan of channel c in homogeneous form: (n, d) <- M_t (n, d) with
        // M_t = [[a^2, w], [u a^2, 1 + u w]] (KDN notes section 6); p^_t = n_t / d_{t-1};
        // the pair is rescaled by a power of two (exact) every 8 tokens.
        const int c = tid;
        float n = carry, d = 1.f, g = 0.f;
        for (int i0 = 0; i0 < CM; i0 += 8) {
          const float4 k0 = *reinterpret_cast<const float4*>(sKt + c * CS + i0);
          const float4 k1 = *reinterpret_cast<const float4*>(sKt + c * CS + i0 + 4);
          const float kvs[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int i = i0 + e;
            const float la = sX[i * DK + c];
            const float al = __expf(la);
            const float a2 = al * al;
            const float kk = kvs[e] * kvs[e];
            const float u = sb2[i] * kk;
            const float n1 = a2 * n + sW[i * DK + c] * d;
            sW[i * DK + c] = __fdividef(n1, d);     // p^_i
            d = d + u * n1;
            n = n1;
            g += la;
            sX[i * DK + c] = g;
          }
          int ex;
          frexpf(d, &ex);
          n = ldexpf(n, -ex);
          d = ldexpf(d, -ex);
        }
        carry = n / d;
        if (chained) {   // p at the chunk end -> the next chunk's record, or aux after the last
          if (ci + 1 < NCk) {
            __stcg(reinterpret_cast<float*>(rec + kRecK + rkP0) + c, carry);
            __threadfence();
          } else if (a.aux) {
            a.aux[(long)bh * DK + c] = carry;
          }
        }
      }
      if (kdn) __syncthreads();
      if (chained && tid == 0 && ci + 1 < NCk && ri + 1 != g_chain_withhold)
        st_release_gpu(chain + ri + 1, 1u);
      if (kdn) {   // z_i = sum_c p^_ic k_ic^2: warp w takes rows 8w .. 8w + 7 (keys read as two
          // 16-byte pieces per channel), all partial sums first, then the eight
          // reductions side by side
        constexpr int kRows = CM / (kThreads / 32);
        static_assert(kRows == 8, "eight rows per warp");
        const int i0 = kRows * warp;
        float z[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) z[r] = 0.f;
#pragma unroll
        for (int c = lane; c < DK; c += 32) {
          const float4 k0 = *reinterpret_cast<const float4*>(sKt + c * CS + i0);
          const float4 k1 = *reinterpret_cast<const float4*>(sKt + c * CS + i0 + 4);
          const float kv[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
          for (int r = 0; r < kRows; ++r) z[r] += sW[(i0 + r) * DK + c] * kv[r] * kv[r];
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) z[r] = warp_sum(z[r]);
        if (lane == 0) {
#pragma unroll
          for (int r = 0; r < kRows; ++r)   // gain denominator, inverted once per row
            sz[i0 + r] = 1.f / (sb1[i0 + r] + z[r]);
        }
      }
      if (kdn) __syncthreads();
      // thread (channel c, tokens 4 i4 .. 4 i4 + 3): 16-byte accesses to the token-minor
      // buffers, consecutive channels across lanes in the token-major one
#pragma unroll 2
      for (int e4 = tid; kdn && e4 < CM * DK / 4; e4 += kThreads) {
        const int c = e4 % DK, i0 = 4 * (e4 / DK);
        const float4 k4 = *reinterpret_cast<const float4*>(sKt + c * CS + i0);
        const float kx[4] = {k4.x, k4.y, k4.z, k4.w};
        float w[4];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          w[y] = sW[(i0 + y) * DK + c] * kx[y] * sz[i0 + y];
          sW[(i0 + y) * DK + c] = w[y];
        }
        *reinterpret_cast<float4*>(sWt + c * CS + i0) = make_float4(w[0], w[1], w[2], w[3]);
      }
      __syncthreads();
      // factor vectors from the per-channel g (g_{-1} = 0 at the chunk start); the
      // per-channel exponentials here and below use the fast exp (relative error
      // ~1e-6 at the workloads' decay spans, far inside either tolerance)
      for (int e = tid; e < NSM * DK; e += kThreads) {
        const int I = e / DK, c = e % DK;
        const float gb = (I == 0) ? 0.f : sX[(16 * I - 1) * DK + c];
        const float gm = sX[(16 * I + 7) * DK + c];
        const float ge = sX[(16 * I + 15) * DK + c];
        fDa[I * DK + c] = __expf(gb - gm);
        fDb[I * DK + c] = __expf(gm - ge);
        fGb[I * DK + c] = __expf(gb);
        for (int J = 0; J < I; ++J)
          fOff[pair_index(I, J) * DK + c] = __expf(gb - sX[(16 * J + 15) * DK + c]);
      }
      if (tid < DK) sgC[tid] = __expf(sX[(CM - 1) * DK + tid]);
      // scale K, Q to their sub-chunk's previous boundary and W^T to its own end;
      // the row-major W becomes exp(g_C - g_j) . w_j for the state update
      // (same thread mapping as the gains above: 4 tokens of one sub-chunk per thread)
#pragma unroll 2
      for (int e4 = tid; e4 < CM * DK / 4; e4 += kThreads) {
        const int c = e4 % DK, i0 = 4 * (e4 / DK), I = i0 >> 4;
        const float gb = (I == 0) ? 0.f : sX[(16 * I - 1) * DK + c];
        const float ge = sX[(16 * I + 15) * DK + c];
        const float gC = sX[(CM - 1) * DK + c];
        float4 k4 = *reinterpret_cast<const float4*>(sKt + c * CS + i0);
        float4 q4 = *reinterpret_cast<const float4*>(sQt + c * CS + i0);
        float4 w4 = *reinterpret_cast<const float4*>(sWt + c * CS + i0);
        float* kx = reinterpret_cast<float*>(&k4);
        float* qx = reinterpret_cast<float*>(&q4);
        float* wx = reinterpret_cast<float*>(&w4);
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const float gi = sX[(i0 + y) * DK + c];
          const float fk = __expf(gi - gb);
          kx[y] *= fk;
          qx[y] *= fk;
          wx[y] *= __expf(ge - gi);
          sW[(i0 + y) * DK + c] *= __expf(gC - gi);
        }
        *reinterpret_cast<float4*>(sKt + c * CS + i0) = k4;
        *reinterpret_cast<float4*>(sQt + c * CS + i0) = q4;
        *reinterpret_cast<float4*>(sWt + c * CS + i0) = w4;
      }
      __syncthreads();
    }

    // ---- 4. Gram: L (row-major, into the L/T buffer) and P^T; the per-channel g is dead
    //      Warp-level TF32x3 tensor-core products (fp32-accurate, as in the inverse).
    //      One unit = the 16 x 16 output of sub-chunk pair (I, J <= I) for K (-> L) or
    //      Q (-> P) over all dk channels, as two 16 x 8 halves sharing the A operand;
    //      the pair's per-channel factors scale the W operand before it is split.
    //      Six independent accumulation chains per k-step (hi.hi, lo.hi, hi.lo for each
    //      half) keep the tensor pipe busy.  20 units over 8 warps.
    {
      const int g = lane >> 2, t = lane & 3;
      const float* Wsrc = explicit_w ? sWt : sKt;
      for (int u = warp; u < 20; u += kThreads / 32) {
        const int pr = u >> 1, isq = u & 1;
        int I = 0;
        while ((I + 1) * (I + 2) / 2 <= pr) ++I;           // pair pr -> (I, J), J <= I
        const int J = pr - I * (I + 1) / 2;
        const float* Xt = isq ? sQt : sKt;
        const float* fk = (perchan && J == I) ? fDa + I * DK : sOne;
        const float* fw = perchan ? ((J < I) ? fOff + pair_index(I, J) * DK : fDb + I * DK) : sOne;
        const int ra = 16 * I + g, cb = 16 * J + g;
        float d[2][4], dl[2][4], dr[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int x = 0; x < 4; ++x) d[h][x] = dl[h][x] = dr[h][x] = 0.f;
        if constexpr (sizeof(Tin) == 2) {
          // bf16 inputs (5e-3 bar): m16n8k16 bf16 products of hi/lo splits (~2^-16
          // relative per term), 16 channels per k-step
#pragma unroll 2
          for (int ks = 0; ks < DK / 16; ++ks) {
            const int c0 = 16 * ks + 2 * t, c1 = c0 + 8;   // channels c0, c0+1, c1, c1+1
            const float f00 = fk[c0] * fw[c0], f01 = fk[c0 + 1] * fw[c0 + 1];
            const float f10 = fk[c1] * fw[c1], f11 = fk[c1 + 1] * fw[c1 + 1];
            uint32_t ah[4], al[4];
            split2(Xt[c0 * CS + ra], Xt[(c0 + 1) * CS + ra], ah[0], al[0]);
            split2(Xt[c0 * CS + ra + 8], Xt[(c0 + 1) * CS + ra + 8], ah[1], al[1]);
            split2(Xt[c1 * CS + ra], Xt[(c1 + 1) * CS + ra], ah[2], al[2]);
            split2(Xt[c1 * CS + ra + 8], Xt[(c1 + 1) * CS + ra + 8], ah[3], al[3]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int cc = cb + 8 * h;
              uint32_t bh[2], bl[2];
              split2(Wsrc[c0 * CS + cc] * f00, Wsrc[(c0 + 1) * CS + cc] * f01, bh[0], bl[0]);
              split2(Wsrc[c1 * CS + cc] * f10, Wsrc[(c1 + 1) * CS + cc] * f11, bh[1], bl[1]);
              mma_bf16_16816(dl[h], al, bh);
              mma_bf16_16816(dr[h], ah, bl);
              mma_bf16_16816(d[h], ah, bh);
            }
          }
        } else {
  #pragma unroll 2
          for (int ks = 0; ks < DK / 8; ++ks) {
            const int c0 = 8 * ks + t, c1 = c0 + 4;
            const float af[4] = {Xt[c0 * CS + ra], Xt[c0 * CS + ra + 8], Xt[c1 * CS + ra],
                                 Xt[c1 * CS + ra + 8]};
            const float f0 = fk[c0] * fw[c0], f1 = fk[c1] * fw[c1];
            uint32_t ah[4], al[4];
  #pragma unroll
            for (int x = 0; x < 4; ++x) {
              ah[x] = tc::to_tf32(af[x]);
              al[x] = tc::to_tf32(af[x] - __uint_as_float(ah[x]));
            }
  #pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float bf[2] = {Wsrc[c0 * CS + cb + 8 * h] * f0, Wsrc[c1 * CS + cb + 8 * h] * f1};
              uint32_t bh[2], bl[2];
  #pragma unroll
              for (int x = 0; x < 2; ++x) {
                bh[x] = tc::to_tf32(bf[x]);
                bl[x] = tc::to_tf32(bf[x] - __uint_as_float(bh[x]));
              }
              tc::mma_tf32(dl[h], al, bh);
              tc::mma_tf32(dr[h], ah, bl);
              tc::mma_tf32(d[h], ah, bh);
            }
          }
        }
        // fragment element (row g or g + 8, column 2t or 2t + 1) -> L row-major / P^T
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int i = 16 * I + g + 8 * (x >> 1), j = 16 * J + 8 * h + 2 * t + (x & 1);
            float v = d[h][x] + (dl[h][x] + dr[h][x]);
            if (!perchan) {
              v *= expf(fminf(sg[i] - sg[j], 0.f));
              if (!explicit_w) v *= sb1[j];
            }
            if (isq)
              sPt[j * CS + i] = (j <= i) ? v : 0.f;
            else
              sLT[i * LDL + j] = (j < i) ? v : 0.f;
          }
      }
      // L and P above the diagonal blocks are zero (the inverse's 32 x 32 step reads
      // the upper block of T's top-left quarter)
      for (int e = tid; e < 6 * 256; e += kThreads) {
        const int blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
        const int I = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int J = blk < 3 ? 1 + blk : (blk < 5 ? blk - 1 : 3);
        sPt[(16 * J + cc) * CS + 16 * I + r] = 0.f;
        sLT[(16 * I + r) * LDL + 16 * J + cc] = 0.f;
      }
      __syncthreads();
    }

    // ---- 5. operands of the carry: Gamma.K, Gamma.Q, exp(g_C - g_j).W, gamma_C
    if (perchan) {   // one channel x 4 tokens of a sub-chunk per thread (16-byte accesses)
#pragma unroll 2
      for (int e4 = tid; e4 < CM * DK / 4; e4 += kThreads) {
        const int c = e4 % DK, i0 = 4 * (e4 / DK);
        const float gb = fGb[(i0 >> 4) * DK + c];
        float4 k4 = *reinterpret_cast<const float4*>(sKt + c * CS + i0);
        float4 q4 = *reinterpret_cast<const float4*>(sQt + c * CS + i0);
        k4.x *= gb; k4.y *= gb; k4.z *= gb; k4.w *= gb;
        q4.x *= gb; q4.y *= gb; q4.z *= gb; q4.w *= gb;
        *reinterpret_cast<float4*>(sKt + c * CS + i0) = k4;
        *reinterpret_cast<float4*>(sQt + c * CS + i0) = q4;
      }
    } else {
      const float gC = sg[CM - 1];
#pragma unroll 4
      for (int e = tid; e < CM * DK; e += kThreads) {
        const int i = e / DK, c = e % DK;
        const float gi = expf(sg[i]);
        sKt[c * CS + i] *= gi;
        sQt[c * CS + i] *= gi;
        sW[e] *= expf(gC - sg[i]) * (explicit_w ? 1.f : sb1[i]);
      }
      if (tid == 0) sgC[0] = expf(gC);
    }
    __syncthreads();

    // ---- 6. T = (I + L)^-1 in place (row-major), then T^T for E = T R
    {
      const int j = tid & 15, I = (tid >> 4) & 3, r0 = 16 * I;
      float t[16];
#pragma unroll
      for (int l = 0; l < 16; ++l) t[l] = (l == j) ? 1.f : 0.f;
      if (tid < 64) {
#pragma unroll
        for (int i = 1; i < 16; ++i) {
          float s = 0.f;
#pragma unroll
          for (int l = 0; l < i; ++l) s += sLT[(r0 + i) * LDL + r0 + l] * t[l];
          if (i > j) t[i] = -s;
        }
      }
      __syncthreads();
      if (tid < 64) {
#pragma unroll
        for (int i = 0; i < 16; ++i) sLT[(r0 + i) * LDL + r0 + j] = t[i];
      }
    }
    __syncthreads();
    if (warp < 4) {   // level 1: T_10 = -T_11 (L_10 T_00), T_32 = -T_33 (L_32 T_22)
      const int blk = warp >> 1, nt = warp & 1;
      const int r0 = 32 * blk + 16, c0 = 32 * blk;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      tile_mm3<2>(d, sLT + r0 * LDL + c0, LDL, sLT + c0 * LDL + c0 + 8 * nt, LDL, lane);
      tile_store(sXS + 16 * blk * LDX + 8 * nt, LDX, d, 1.f, lane);
    }
    __syncthreads();
    if (warp < 4) {
      const int blk = warp >> 1, nt = warp & 1;
      const int r0 = 32 * blk + 16, c0 = 32 * blk;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      tile_mm3<2>(d, sLT + r0 * LDL + r0, LDL, sXS + 16 * blk * LDX + 8 * nt, LDX, lane);
      tile_store(sLT + r0 * LDL + c0 + 8 * nt, LDL, d, -1.f, lane);
    }
    __syncthreads();
    {   // level 2: rows 32-63 x cols 0-31: T_C = -T_B (L_C T_A)
      const int mt = warp >> 2, nt = warp & 3;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      tile_mm3<4>(d, sLT + (32 + 16 * mt) * LDL, LDL, sLT + 8 * nt, LDL, lane);
      tile_store(sXS + 16 * mt * LDX + 8 * nt, LDX, d, 1.f, lane);
    }
    __syncthreads();
    {
      const int mt = warp >> 2, nt = warp & 3;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      if (mt == 0)
        tile_mm3<2>(d, sLT + 32 * LDL + 32, LDL, sXS + 8 * nt, LDX, lane);
      else
        tile_mm3<4>(d, sLT + 48 * LDL + 32, LDL, sXS + 8 * nt, LDX, lane);
      tile_store(sLT + (32 + 16 * mt) * LDL + 8 * nt, LDL, d, -1.f, lane);
    }
    __syncthreads();
    if constexpr (PREP) {   // the carry's operands -> the record (float4 stores, coalesced)
      float4* rT = reinterpret_cast<float4*>(rec + rkT);
      float4* rP = reinterpret_cast<float4*>(rec + rkP);
      float4* rK = reinterpret_cast<float4*>(rec + rkK);
      float4* rQ = reinterpret_cast<float4*>(rec + rkQ);
      float4* rW = reinterpret_cast<float4*>(rec + rkW);
#pragma unroll
      for (int r = 0; r < CM * CM / 4 / kThreads; ++r) {
        const int e = tid + r * kThreads, row = e >> 4, c4 = (e & 15) * 4;
        const float4 tv = *reinterpret_cast<const float4*>(sLT + row * LDL + c4);
        rT[e] = make_float4(c4 <= row ? tv.x : 0.f, c4 + 1 <= row ? tv.y : 0.f,
                            c4 + 2 <= row ? tv.z : 0.f, c4 + 3 <= row ? tv.w : 0.f);
        rP[e] = *reinterpret_cast<const float4*>(sPt + row * CS + c4);
      }
#pragma unroll
      for (int r = 0; r < DK * CM / 4 / kThreads; ++r) {
        const int e = tid + r * kThreads, row = e >> 4, c4 = (e & 15) * 4;
        rK[e] = *reinterpret_cast<const float4*>(sKt + row * CS + c4);
        rQ[e] = *reinterpret_cast<const float4*>(sQt + row * CS + c4);
        rW[e] = *reinterpret_cast<const float4*>(sW + 4 * e);
      }
      if (tid < DK / 4)
        reinterpret_cast<float4*>(rec + rkG)[tid] = *reinterpret_cast<const float4*>(sgC + 4 * tid);
      continue;
    }
    for (int e = tid; e < CM * CM; e += kThreads) {   // T^T (upper triangle of T is zero)
      const int i = e >> 6, j = e & 63;
      sTt[j * CS + i] = (j <= i) ? sLT[i * LDL + j] : 0.f;
    }
    __syncthreads();

    // ---- 7. R = V - (Gamma.K) S   (rows i in 4-blocks, columns n in pairs)
    const int ti = tid / 16, tn = tid % 16;  // 16 x 16 thread grid: 4 rows x 2 cols each
    float acc[4][2];
#pragma unroll
    for (int x = 0; x < 4; ++x) acc[x][0] = acc[x][1] = 0.f;
    for (int c = 0; c < DK; ++c) {
      const float4 k4 = *reinterpret_cast<const float4*>(sKt + c * CS + 4 * ti);
      const float2 s2 = *reinterpret_cast<const float2*>(sS + c * NV + 2 * tn);
      const float kx[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        acc[x][0] += kx[x] * s2.x;
        acc[x][1] += kx[x] * s2.y;
      }
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      float2* vp = reinterpret_cast<float2*>(sV + (4 * ti + x) * NV + 2 * tn);
      float2 v2 = *vp;
      v2.x -= acc[x][0];
      v2.y -= acc[x][1];
      *vp = v2;
    }
    __syncthreads();
    // E = T R, written over R once every thread has read it
#pragma unroll
    for (int x = 0; x < 4; ++x) acc[x][0] = acc[x][1] = 0.f;
    for (int j = 0; j < 4 * ti + 4; ++j) {
      const float4 t4 = *reinterpret_cast<const float4*>(sTt + j * CS + 4 * ti);
      const float2 r2 = *reinterpret_cast<const float2*>(sV + j * NV + 2 * tn);
      const float tx[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        acc[x][0] += tx[x] * r2.x;
        acc[x][1] += tx[x] * r2.y;
      }
    }
    __syncthreads();
#pragma unroll
    for (int x = 0; x < 4; ++x)
      *reinterpret_cast<float2*>(sV + (4 * ti + x) * NV + 2 * tn) = make_float2(acc[x][0], acc[x][1]);
    __syncthreads();
    // O = (Gamma.Q) S + P E  -> global
    {
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[x][0] = acc[x][1] = 0.f;
      for (int c = 0; c < DK; ++c) {
        const float4 q4 = *reinterpret_cast<const float4*>(sQt + c * CS + 4 * ti);
        const float2 s2 = *reinterpret_cast<const float2*>(sS + c * NV + 2 * tn);
        const float qx[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          acc[x][0] += qx[x] * s2.x;
          acc[x][1] += qx[x] * s2.y;
        }
      }
      for (int j = 0; j < 4 * ti + 4; ++j) {
        const float4 p4 = *reinterpret_cast<const float4*>(sPt + j * CS + 4 * ti);
        const float2 e2 = *reinterpret_cast<const float2*>(sV + j * NV + 2 * tn);
        const float px[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          acc[x][0] += px[x] * e2.x;
          acc[x][1] += px[x] * e2.y;
        }
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int i = 4 * ti + x;
        if (i < Cc) {
          Tin* op = static_cast<Tin*>(a.out) + tok_index(a, b, t0 + i, h) * a.dv + tile * NV + 2 * tn;
          op[0] = from_f<Tin>(acc[x][0]);
          op[1] = from_f<Tin>(acc[x][1]);
          if (a.check_finite) bad |= !(finite_f(acc[x][0]) && finite_f(acc[x][1]));
        }
      }
    }
    __syncthreads();
    // S <- diag(gamma_C) S + Wbar^T E   (thread: 4 channels x 4 columns)
    {
      const int tc = tid / 8, tv = tid % 8;
      for (int cb = tc; cb < DK / 4; cb += 32) {
        float s4[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int c = 4 * cb + x;
          const float gcf = perchan ? sgC[c] : sgC[0];
          const float4 old = *reinterpret_cast<const float4*>(sS + c * NV + 4 * tv);
          s4[x][0] = gcf * old.x; s4[x][1] = gcf * old.y; s4[x][2] = gcf * old.z; s4[x][3] = gcf * old.w;
        }
        for (int j = 0; j < CM; ++j) {
          const float4 w4 = *reinterpret_cast<const float4*>(sW + j * DK + 4 * cb);
          const float4 e4 = *reinterpret_cast<const float4*>(sV + j * NV + 4 * tv);
          const float wx[4] = {w4.x, w4.y, w4.z, w4.w};
          const float ex[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
          for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) s4[x][y] += wx[x] * ex[y];
        }
#pragma unroll
        for (int x = 0; x < 4; ++x)
          *reinterpret_cast<float4*>(sS + (4 * cb + x) * NV + 4 * tv) =
              make_float4(s4[x][0], s4[x][1], s4[x][2], s4[x][3]);
      }
    }
  }
  __syncthreads();

  // final state and aux
  if (PREP) return;
  if (a.S) {
    for (int e = tid; e < DK * NV; e += kThreads) {
      const int c = e / NV, n = e % NV;
      const float v = sS[e];
      a.S[((long)bh * DK + c) * a.dv + tile * NV + n] = v;
      if (a.check_finite) bad |= !finite_f(v);
    }
  }
  if (a.aux && tile == 0 && (pstat || kdn) && my_c >= 0 && my_c < DK)
    a.aux[(long)bh * DK + my_c] = carry;
  if (a.aux && tile == 0 && ikdn && tid == DK) a.aux[bh] = carry;
  if (bad) set_status(DR_ERR_NONFINITE);
}

// ================================================================= two-phase Diagonal KDN
// The per-channel variance recurrence p^ = a^2 p + w, p = p^ / (1 + u p^) is a
// Moebius map of p, i.e. the linear map (n, d) <- [[a^2, w], [u a^2, 1 + u w]] (n, d)
// in homogeneous coordinates p = n / d (KDN notes section 6); a chunk is the
// product of its tokens' matrices.  With few (b, h) rows (3 B H < SM count) two
// kernels give p at every chunk start before the prep:
//   kdn_map_kernel   one warp per (b, h, chunk), lane = 4 channels (key norm by a
//                    warp reduction); the product is rescaled by a power of two
//                    every 8 tokens (p is scale-free).
//   kdn_scan_kernel  one thread per (b, h, channel) applies the maps in chunk
//                    order and leaves p at every chunk start in the record.
// With more rows the prep chains p itself.  Then chunk_simt_kernel<PREP> does
// every chunk's local work in parallel and kdn_carry_kernel (fp32) or the tcgen05
// carry (bf16) walks the chunks.
constexpr int kKdnMapWarps = 8;   // 4 chunk tasks per block, two warps (token halves) each

__global__ void __launch_bounds__(kKdnMapWarps * 32, 2) kdn_map_kernel(FwdArgs a, uint8_t* __restrict__ ws,
                                                                         int bf16_in) {
  __shared__ float4 part[kKdnMapWarps / 2][128];   // second half's product, per channel
  const int NC = (a.T + CM - 1) / CM;
  const long ntask = (long)a.B * a.H * NC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = warp >> 1, halfw = warp & 1;   // task slot in the block, token half
  const long task = (long)blockIdx.x * (kKdnMapWarps / 2) + slot;
  const bool live = task < ntask;
  const int bh = live ? (int)(task / NC) : 0, c = live ? (int)(task % NC) : 0;
  const int b = bh / a.H, h = bh % a.H;
  float m[4][4];   // per channel [m00, m01, m10, m11]
#pragma unroll
  for (int q = 0; q < 4; ++q) { m[q][0] = 1.f; m[q][1] = 0.f; m[q][2] = 0.f; m[q][3] = 1.f; }
  const int t_lo = halfw * 32, t_hi = live ? min(t_lo + 32, a.T - c * CM) : 0;
  for (int i0 = t_lo; i0 < t_hi; i0 += 4) {
    float kv[4][4], la[4][4], om[4][4], ir[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {   // four tokens' loads in flight at once
      const bool real = i0 + e < t_hi;
      const long ti = ((long)b * a.T + c * CM + (real ? i0 + e : 0)) * a.H + h;
      if (bf16_in) {
        const uint2 raw = real ? *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(a.k) +
                                                                 ti * 128 + 4 * lane)
                               : make_uint2(0u, 0u);
        kv[e][0] = __uint_as_float(raw.x << 16);
        kv[e][1] = __uint_as_float(raw.x & 0xffff0000u);
        kv[e][2] = __uint_as_float(raw.y << 16);
        kv[e][3] = __uint_as_float(raw.y & 0xffff0000u);
      } else {
        const float4 f = real ? *reinterpret_cast<const float4*>(static_cast<const float*>(a.k) +
                                                                 ti * 128 + 4 * lane)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        kv[e][0] = f.x; kv[e][1] = f.y; kv[e][2] = f.z; kv[e][3] = f.w;
      }
      const float4 l4 = real ? *reinterpret_cast<const float4*>(a.log_alpha + ti * 128 + 4 * lane)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 o4 = real ? *reinterpret_cast<const float4*>(a.omega + ti * 128 + 4 * lane)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      la[e][0] = l4.x; la[e][1] = l4.y; la[e][2] = l4.z; la[e][3] = l4.w;
      om[e][0] = o4.x; om[e][1] = o4.y; om[e][2] = o4.z; om[e][3] = o4.w;
      ir[e] = real ? a.info_scale / a.r[ti] : 0.f;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float kk = warp_sum(kv[e][0] * kv[e][0] + kv[e][1] * kv[e][1] + kv[e][2] * kv[e][2] +
                                kv[e][3] * kv[e][3]);
      const float cr = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float al = __expf(la[e][q]), a2 = al * al, w = om[e][q];
        const float kh = kv[e][q] * cr, u = ir[e] * kh * kh;
        // M <- [[a2, w], [u a2, 1 + u w]] M
        const float n0 = a2 * m[q][0] + w * m[q][2], n1 = a2 * m[q][1] + w * m[q][3];
        const float d0 = u * n0 + m[q][2], d1 = u * n1 + m[q][3];
        m[q][0] = n0; m[q][1] = n1; m[q][2] = d0; m[q][3] = d1;
      }
    }
    if (((i0 - t_lo) & 7) == 4 || i0 + 4 >= t_hi) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {   // exact power-of-two rescale
        int ex;
        frexpf(fmaxf(fmaxf(fabsf(m[q][0]), fabsf(m[q][1])), fmaxf(fabsf(m[q][2]), fabsf(m[q][3]))), &ex);
#pragma unroll
        for (int z = 0; z < 4; ++z) m[q][z] = ldexpf(m[q][z], -ex);
      }
    }
  }
  if (halfw == 1) {
#pragma unroll
    for (int q = 0; q < 4; ++q) part[slot][4 * lane + q] = make_float4(m[q][0], m[q][1], m[q][2], m[q][3]);
  }
  __syncthreads();
  if (halfw == 0 && live) {   // M = M_second M_first
    float4* out = reinterpret_cast<float4*>(ws + (size_t)task * kRecK + rkMap);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 s2 = part[slot][4 * lane + q];
      out[4 * lane + q] = make_float4(s2.x * m[q][0] + s2.y * m[q][2], s2.x * m[q][1] + s2.y * m[q][3],
                                      s2.z * m[q][0] + s2.w * m[q][2], s2.z * m[q][1] + s2.w * m[q][3]);
    }
  }
}

__global__ void __launch_bounds__(128) kdn_scan_kernel(FwdArgs a, uint8_t* __restrict__ ws) {
  const int bh = blockIdx.x, ch = threadIdx.x;
  const int NC = (a.T + CM - 1) / CM;
  uint8_t* recs = ws + (size_t)bh * NC * kRecK;
  float n = a.aux0 ? a.aux0[(long)bh * 128 + ch] : 1.f, d = 1.f;
  float4 mc = reinterpret_cast<const float4*>(recs + rkMap)[ch];
  for (int c = 0; c < NC; ++c) {
    const float4 mn = reinterpret_cast<const float4*>(recs + (size_t)min(c + 1, NC - 1) * kRecK + rkMap)[ch];
    reinterpret_cast<float*>(recs + (size_t)c * kRecK + rkP0)[ch] = n / d;
    const float n2 = mc.x * n + mc.y * d, d2 = mc.z * n + mc.w * d;
    int ex;
    frexpf(fmaxf(fabsf(n2), fabsf(d2)), &ex);
    n = ldexpf(n2, -ex);
    d = ldexpf(d2, -ex);
    mc = mn;
  }
  if (a.aux) a.aux[(long)bh * 128 + ch] = n / d;
}

// The carry of the two-phase Diagonal KDN path: one CTA per (b, h, 64 columns).
// Per chunk, from the record (cp.async):
//   R = V - (Gamma.K) S  and  Q S  in one pass over S,  E = T R,  O = (Gamma.Q) S + P E,
//   S <- diag(gamma_C) S + (exp(g_C - g_j).w_j)^T E     (fp32, CUDA cores).
// (Gamma.K)^T of chunk c+1 is copied into a second buffer during chunk c's state
// update; the other operands of chunk c are copied while R is computed.
constexpr int kKcNV = 64;
// shared layout (bytes): K^T x 2 | T | P^T | Q^T | Wbar | gamma | S | V/R/E
constexpr uint32_t kcK = 0;                 // 2 x 32 KB
constexpr uint32_t kcT = 65536;             // 16 KB
constexpr uint32_t kcP = kcT + 16384;       // 16 KB
constexpr uint32_t kcQ = kcP + 16384;       // 32 KB
constexpr uint32_t kcW = kcQ + 32768;       // 32 KB
constexpr uint32_t kcG = kcW + 32768;       // 512 B
constexpr uint32_t kcS = kcG + 512;         // 32 KB
constexpr uint32_t kcV = kcS + 32768;       // 16 KB
constexpr uint32_t kKcSmem = kcV + 16384;


template <typename Tin>
__global__ void __launch_bounds__(kThreads, 1) kdn_carry_kernel(FwdArgs a, const uint8_t* __restrict__ ws) {
  extern __shared__ __align__(16) float smk[];
  __shared__ uint64_t bars[3];   // (Gamma.K)^T buffers 0 / 1, the rest of the record
  __shared__ volatile int s_abort;
  uint8_t* smb = reinterpret_cast<uint8_t*>(smk);
  const float* kT = reinterpret_cast<const float*>(smb + kcT);   // [64][64]
  const float* kPt = reinterpret_cast<const float*>(smb + kcP);  // [64 j][64 i]
  const float* kQt = reinterpret_cast<const float*>(smb + kcQ);  // [128 c][64 i]
  const float* kW = reinterpret_cast<const float*>(smb + kcW);   // [64 j][128 c]
  const float* kG = reinterpret_cast<const float*>(smb + kcG);   // [128]
  float* sS = reinterpret_cast<float*>(smb + kcS);               // [128][64]
  float* sV = reinterpret_cast<float*>(smb + kcV);               // [64][64]: V, R, E
  const int tid = threadIdx.x;
  const int tile = blockIdx.x & 1, bh = blockIdx.x >> 1, b = bh / a.H, h = bh % a.H;
  const int NC = (a.T + CM - 1) / CM;
  const uint8_t* recs = ws + (size_t)bh * NC * kRecK;
  bool bad = false;
  // record pieces arrive by bulk copies (one thread issues, every thread waits,
  // bounded in time; a wait that gives up marks the CTA aborted)
  if (tid == 0) {
    for (int q = 0; q < 3; ++q) umma::mbar_init(&bars[q], 1);
    umma::fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();
  int n_issued[3] = {0, 0, 0};   // copies issued per barrier (thread 0)
  auto load_k = [&](int c) {
    uint64_t* bar = &bars[c & 1];
    ++n_issued[c & 1];
    umma::mbar_expect_tx(bar, 32768);
    umma::bulk_load(smb + kcK + (c & 1) * 32768, recs + (size_t)c * kRecK + rkK, 32768, bar);
  };
  auto wait_bar = [&](int q, uint32_t parity) {
    if (!s_abort && !umma::mbar_wait(&bars[q], parity, 2000000000ull)) s_abort = 1;
  };
  for (int e = tid; e < 128 * kKcNV / 4; e += kThreads) {
    const int c = e >> 4, n4 = (e & 15) * 4;
    reinterpret_cast<float4*>(sS)[e] =
        a.S0 ? *reinterpret_cast<const float4*>(a.S0 + ((long)bh * 128 + c) * a.dv + tile * kKcNV + n4)
             : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (tid == 0) load_k(0);
  const int ti = tid >> 4, tn = tid & 15;   // rows 4 ti.., columns 4 tn..
  for (int c = 0; c < NC; ++c) {
    const int t0 = c * CM, Cc = min(CM, a.T - t0);
    const float* kKt = reinterpret_cast<const float*>(smb + kcK + (c & 1) * 32768);
    __syncthreads();   // previous chunk done with T, P, Q, W, V
    {
      const uint8_t* rec = recs + (size_t)c * kRecK;
      if (tid == 0) {
        ++n_issued[2];
        umma::mbar_expect_tx(&bars[2], 32768 + 32768 * 2 + 512);
        umma::bulk_load(smb + kcT, rec + rkT, 32768, &bars[2]);             // T, P^T
        umma::bulk_load(smb + kcQ, rec + rkQ, 32768 * 2 + 512, &bars[2]);   // Q^T, Wbar, gamma
      }
      // V tile [64 tokens][64 columns] with 16-byte loads
      constexpr int kPer = (int)sizeof(Tin) == 2 ? 8 : 4;   // elements per 16 bytes
      constexpr int kVec = CM * kKcNV / kPer / kThreads;
      uint4 raw[kVec];
#pragma unroll
      for (int r = 0; r < kVec; ++r) {
        const int e = tid + r * kThreads, i = e / (kKcNV / kPer), n0 = (e % (kKcNV / kPer)) * kPer;
        raw[r] = (i < Cc) ? __ldg(reinterpret_cast<const uint4*>(static_cast<const Tin*>(a.v) +
                                  tok_index(a, b, t0 + i, h) * a.dv + tile * kKcNV + n0))
                          : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int r = 0; r < kVec; ++r) {
        const int e = tid + r * kThreads, i = e / (kKcNV / kPer), n0 = (e % (kKcNV / kPer)) * kPer;
        float* dst = sV + i * kKcNV + n0;
        if (kPer == 8) {
          const uint32_t w[4] = {raw[r].x, raw[r].y, raw[r].z, raw[r].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            dst[2 * q] = __uint_as_float(w[q] << 16);
            dst[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
          }
        } else {
          *reinterpret_cast<uint4*>(dst) = raw[r];
        }
      }
      wait_bar(c & 1, (c >> 1) & 1);   // this chunk's (Gamma.K)^T; the rest may still fly
    }
    __syncthreads();
    if (s_abort) break;
    float acc[4][4], aq[4][4];
    // R = V - (Gamma.K) S  and the (Gamma.Q) S part of O, one pass over S; the Q
    // tile is read only after it lands, so the pass waits for it half-way in:
    // first (Gamma.K) S alone over all channels, then (Gamma.Q) S.
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
#pragma unroll 8
    for (int cc = 0; cc < 128; ++cc) {
      const float4 k4 = *reinterpret_cast<const float4*>(kKt + cc * 64 + 4 * ti);
      const float4 s4 = *reinterpret_cast<const float4*>(sS + cc * kKcNV + 4 * tn);
      const float kx[4] = {k4.x, k4.y, k4.z, k4.w}, sx[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] += kx[x] * sx[y];
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      float4* vp = reinterpret_cast<float4*>(sV + (4 * ti + x) * kKcNV + 4 * tn);
      float4 v4 = *vp;
      v4.x -= acc[x][0]; v4.y -= acc[x][1]; v4.z -= acc[x][2]; v4.w -= acc[x][3];
      *vp = v4;
    }
    wait_bar(2, c & 1);
    __syncthreads();   // R complete; T, P, Q, W, gamma landed
    if (s_abort) break;
    // (Gamma.K)^T of chunk c+1 into the other buffer, under the rest of this chunk
    if (tid == 0 && c + 1 < NC) load_k(c + 1);
    // (Gamma.Q) S
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) aq[x][y] = 0.f;
#pragma unroll 8
    for (int cc = 0; cc < 128; ++cc) {
      const float4 q4 = *reinterpret_cast<const float4*>(kQt + cc * 64 + 4 * ti);
      const float4 s4 = *reinterpret_cast<const float4*>(sS + cc * kKcNV + 4 * tn);
      const float qx[4] = {q4.x, q4.y, q4.z, q4.w}, sx[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) aq[x][y] += qx[x] * sx[y];
    }
    // E = T R (T lower triangular), written over R once every thread has read it
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
#pragma unroll 4
    for (int j = 0; j < 4 * ti + 4; ++j) {
      const float4 r4 = *reinterpret_cast<const float4*>(sV + j * kKcNV + 4 * tn);
      const float rx[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float t = kT[(4 * ti + x) * 64 + j];
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] += t * rx[y];
      }
    }
    __syncthreads();
#pragma unroll
    for (int x = 0; x < 4; ++x)
      *reinterpret_cast<float4*>(sV + (4 * ti + x) * kKcNV + 4 * tn) =
          make_float4(acc[x][0], acc[x][1], acc[x][2], acc[x][3]);
    __syncthreads();
    // O = (Gamma.Q) S + P E -> global
#pragma unroll 4
    for (int j = 0; j < 4 * ti + 4; ++j) {
      const float4 p4 = *reinterpret_cast<const float4*>(kPt + j * 64 + 4 * ti);
      const float4 e4 = *reinterpret_cast<const float4*>(sV + j * kKcNV + 4 * tn);
      const float px[4] = {p4.x, p4.y, p4.z, p4.w}, ex[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) aq[x][y] += px[x] * ex[y];
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int i = 4 * ti + x;
      if (i < Cc) {
        Tin* op = static_cast<Tin*>(a.out) + tok_index(a, b, t0 + i, h) * a.dv + tile * kKcNV + 4 * tn;
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          op[y] = from_f<Tin>(aq[x][y]);
          if (a.check_finite) bad |= !finite_f(aq[x][y]);
        }
      }
    }
    // S <- diag(gamma_C) S + Wbar^T E  (thread: 4 channels x 8 columns); S was read
    // above by every thread (R and Q S), so the update waits for all of them
    __syncthreads();
    {
      const int cg = tid >> 3, vg = tid & 7;
      float s8[4][8];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int ch = 4 * cg + x;
        const float gcf = kG[ch];
        const float4 o0 = *reinterpret_cast<const float4*>(sS + ch * kKcNV + 8 * vg);
        const float4 o1 = *reinterpret_cast<const float4*>(sS + ch * kKcNV + 8 * vg + 4);
        s8[x][0] = gcf * o0.x; s8[x][1] = gcf * o0.y; s8[x][2] = gcf * o0.z; s8[x][3] = gcf * o0.w;
        s8[x][4] = gcf * o1.x; s8[x][5] = gcf * o1.y; s8[x][6] = gcf * o1.z; s8[x][7] = gcf * o1.w;
      }
#pragma unroll 8
      for (int j = 0; j < CM; ++j) {
        const float4 w4 = *reinterpret_cast<const float4*>(kW + j * 128 + 4 * cg);
        const float4 e0 = *reinterpret_cast<const float4*>(sV + j * kKcNV + 8 * vg);
        const float4 e1 = *reinterpret_cast<const float4*>(sV + j * kKcNV + 8 * vg + 4);
        const float wx[4] = {w4.x, w4.y, w4.z, w4.w};
        const float ex[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 8; ++y) s8[x][y] += wx[x] * ex[y];
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        float* sp = sS + (4 * cg + x) * kKcNV + 8 * vg;
        *reinterpret_cast<float4*>(sp) = make_float4(s8[x][0], s8[x][1], s8[x][2], s8[x][3]);
        *reinterpret_cast<float4*>(sp + 4) = make_float4(s8[x][4], s8[x][5], s8[x][6], s8[x][7]);
      }
    }
  }
  __syncthreads();
  if (s_abort) {   // drain the copies this CTA may still have in flight, then report
    if (tid == 0) {
      for (int q = 0; q < 3; ++q)
        if (n_issued[q] > 0) umma::mbar_wait(&bars[q], (n_issued[q] - 1) & 1, 500000000ull);
      set_status(DR_ERR_TIMEOUT);
    }
    return;
  }
  if (a.S) {
    for (int e = tid; e < 128 * kKcNV / 4; e += kThreads) {
      const int c = e >> 4, n4 = (e & 15) * 4;
      const float4 v = reinterpret_cast<const float4*>(sS)[e];
      *reinterpret_cast<float4*>(a.S + ((long)bh * 128 + c) * a.dv + tile * kKcNV + n4) = v;
      if (a.check_finite) bad |= !(finite_f(v.x) && finite_f(v.y) && finite_f(v.z) && finite_f(v.w));
    }
  }
  if (bad) set_status(DR_ERR_NONFINITE);
}

int simt_sm_count() {
  static int count[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!count[dev]) cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev);
  return count[dev];
}

}  // namespace

size_t simt_smem_bytes(int dk) {
  return sizeof(float) * (dk == 64 ? SimtSmem<64>::total : SimtSmem<128>::total);
}

cudaError_t launch_chunk_simt(const FwdArgs& a, int dtype, cudaStream_t st) {
  const int grid = a.B * a.H * (a.dv / NV);
  const size_t smem = simt_smem_bytes(a.dk);
#define DR_SIMT(DK_, T_)                                                                   \
  if (a.dk == DK_) {                                                                       \
    cudaError_t err = cudaFuncSetAttribute(chunk_simt_kernel<DK_, T_, false>,              \
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                                           (int)smem);                                     \
    if (err != cudaSuccess) return err;                                                    \
    chunk_simt_kernel<DK_, T_, false><<<grid, kThreads, smem, st>>>(a, nullptr, nullptr);           \
    return cudaGetLastError();                                                             \
  }
  if (dtype == DR_BF16) {
    DR_SIMT(64, __nv_bfloat16) DR_SIMT(128, __nv_bfloat16)
  } else {
    DR_SIMT(64, float) DR_SIMT(128, float)
  }
#undef DR_SIMT
  return cudaErrorInvalidValue;
}

}  // namespace dr

namespace dr {

cudaError_t launch_carry_kdn_tc(const FwdArgs& a, void* workspace, cudaStream_t st);
cudaError_t launch_pc_prep(const FwdArgs& a, void* workspace, uint32_t* chain, int nsm, cudaStream_t st);

bool kdn_split_supported(int variant, int dtype, int dk, int dv, int chunk) {
  return (variant == DR_KDN || variant == DR_KDA || variant == DR_PKDA || variant == DR_IKDN) &&
         (dtype == DR_BF16 || dtype == DR_FP32) && dk == 128 && dv == 128 && chunk == 64;
}

size_t kdn_split_workspace_bytes(int B, int T, int H) {
  const long ntask = (long)B * H * ((T + CM - 1) / CM);
  return (size_t)ntask * kRecK + chain_bytes(ntask);
}

cudaError_t launch_kdn_split(const FwdArgs& a, int dtype, void* workspace, cudaStream_t st) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const long ntask = (long)a.B * a.H * ((a.T + CM - 1) / CM);
  const int nsm = simt_sm_count();
  if (nsm <= 0) return cudaErrorInvalidValue;
  // A row's chunks form a chain of hand-overs (flag latency + the 4.7K-cycle
  // variance scan, ~6K cycles each), which must stay well inside the prep's own
  // time (NC B H / nsm tasks of ~44K cycles per CTA): NC 6K <= 0.4 NC B H 44K / nsm
  // for 3 B H >= nsm.  Fewer rows: map and scan kernels first.
  // KDA has no gain state across chunks: neither the chain nor the map and scan.
  // PKDA (key statistic) and isotropic KDN (one variance per head) chain theirs
  // the same way; with few rows they run the fused kernel instead.
  // The backward's rerun of the forward (a.save_S set) needs the two phases and
  // their records whatever the row count, so PKDA and isotropic KDN chain then.
  const bool kdn = a.variant == DR_KDN;
  const bool chain_only = a.variant == DR_PKDA || a.variant == DR_IKDN;
  const bool chained = (kdn || chain_only) && (3L * a.B * a.H >= nsm || (chain_only && a.save_S));
  if (chain_only && !chained) return launch_chunk_simt(a, dtype, st);
  uint32_t* chain = chained ? reinterpret_cast<uint32_t*>(ws + (size_t)ntask * kRecK) : nullptr;
  cudaError_t err = cudaSuccess;
  if (chained) {
    err = cudaMemsetAsync(chain, 0, chain_bytes(ntask), st);
  } else if (kdn) {
    kdn_map_kernel<<<(int)((ntask + kKdnMapWarps / 2 - 1) / (kKdnMapWarps / 2)), kKdnMapWarps * 32, 0,
                     st>>>(a, ws, dtype == DR_BF16 ? 1 : 0);
    kdn_scan_kernel<<<a.B * a.H, 128, 0, st>>>(a, ws);
    err = cudaGetLastError();
  }
  if (err != cudaSuccess) return err;
  const size_t psmem = simt_smem_bytes(128);
  const int pgrid = (int)(ntask < nsm ? ntask : nsm);
#define DR_KDN_PREP(T_)                                                                    \
  {                                                                                        \
    err = cudaFuncSetAttribute(chunk_simt_kernel<128, T_, true>,                           \
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);   \
    if (err != cudaSuccess) return err;                                                    \
    chunk_simt_kernel<128, T_, true><<<pgrid, kThreads, psmem, st>>>(a, ws, chain);       \
    if ((err = cudaGetLastError()) != cudaSuccess) return err;                             \
  }
  if (dtype == DR_BF16) {   // tensor-core prep, bf16 records -> the tensor-core carry
    if ((err = launch_pc_prep(a, ws, chain, nsm, st)) != cudaSuccess) return err;
    return launch_carry_kdn_tc(a, ws, st);
  }
  DR_KDN_PREP(float)
#undef DR_KDN_PREP
  err = cudaFuncSetAttribute(kdn_carry_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kKcSmem);
  if (err != cudaSuccess) return err;
  kdn_carry_kernel<float><<<a.B * a.H * 2, kThreads, kKcSmem, st>>>(a, ws);
  return cudaGetLastError();
}

}  // namespace dr
