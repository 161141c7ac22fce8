// chunk_tc_pc.cu — tensor-core prep of the two-phase path with per-channel decay
// (Diagonal KDN, KDA, PKDA, isotropic KDN; bf16 inputs, dk = dv = 128, chunk 64).
//
// One persistent CTA per SM takes one task (b, h, chunk) at a time and writes the
// chunk's record for the tcgen05 carry of chunk_tc_split.cu (KLA notes section
// 2.5, Eqs. (7)-(9), with the per-channel decay D_t = diag(alpha_t) of the KDN
// notes section 1 and the write vectors of each variant):
//
//   loads   K, Q (bf16, 128B-swizzled) and the per-channel log-decay (fp32; KDN
//           also its process noise) arrive by TMA, zero past the end of the row.
//   scans   a thread per channel: the cumulative log-decay g and the variant's
//           carried gain state (KDN variance in homogeneous Moebius form, KDN
//           notes section 6; PKDA key statistic and bound, PDN notes Eq. (9));
//           isotropic KDN scans its head variance on one warp (KDN notes Eq. (40)).
//   Gram    L_ij = sum_c k^_ic w_jc exp(g_ic - g_jc) (j < i) and P (j <= i) on one
//           tcgen05 MMA group.  Each 16-token sub-chunk I takes its middle token
//           m(I) as reference (decay ratios from log differences, KDN notes
//           section 6): A rows = [k^_i ; q^_i] exp(g_i - g_m(I)); the B operand
//           holds, for each I, the write vectors of tokens j < 16 (I + 1) scaled by
//           exp(g_m(I) - g_j) (160 rows); every factor is <= 1 except inside a
//           sub-chunk, where it is bounded by the decay over 8 tokens.  bf16 hi/lo
//           splits of both operands and three products keep fp32 accuracy.
//   inverse T = (I + L)^-1: 16 x 16 diagonal blocks by substitution, the rest by
//           recursive doubling (bf16 hi/lo mma.sync: the blocks are below tcgen05's M).
//   W'      W' = T (Gamma.K) on tcgen05 (Gamma.K = k^_i exp(g_i), hi/lo), read out
//           transposed.
//   record  T, W'^T, P, (Gamma.Q), Wbar = exp(g_C - g_j) w_j (bf16 hi/lo images),
//           gamma_C = exp(g_C) per channel; images go straight to global memory.
//
// The gain state is sequential across chunks.  With many rows the tasks are taken
// in chunk-major ticket order and each hands its state at the chunk end to the
// next chunk's record through a release flag (the wait is bounded: on a lost flag
// it sets DR_ERR_TIMEOUT and the abort word, and the task runs on); with few rows
// (Diagonal KDN only) kdn_map / kdn_scan have left the state at every chunk start
// in the records.
#include <cuda.h>
#include <cuda_bf16.h>

#include "chain.cuh"
#include "dr_common.cuh"
#include "tc_common.cuh"
#include "umma.cuh"

namespace dr {
namespace {

using namespace umma;
using namespace tc;

constexpr uint64_t kWait = 2000000000ull;   // 2 s per bounded wait
constexpr int LDL = 68;                     // fp32 L/T row stride
constexpr int LDX = 36;                     // fp32 scratch row stride
constexpr int kThreads = 512;              // 16 warps: two per scheduler in every phase
constexpr int kUnits = 1024 / kThreads;     // (token, 8-channel) units per thread
constexpr int kWarps = kThreads / 32;

// ---- record of one chunk (bytes; read by the carry's per-channel mode)
constexpr uint32_t rbT = 0;          // T hi | T lo [64 i][64 j]
constexpr uint32_t rbWp = 16384;     // W'^T hi [128 c][64 i], then lo
constexpr uint32_t rbP = 49152;      // P hi | P lo [64 i][64 j]
constexpr uint32_t rbVec = 65536;    // fp32: [0,128) ones, [128,256) gamma_C per channel
constexpr uint32_t rbQ = 66560;      // (Gamma.Q) [64 tok][128] hi (two 64-column blocks), then lo
constexpr uint32_t rbW = 99328;      // Wbar, same layout
constexpr uint32_t rkP0 = 134144;    // gain state at the chunk start (chains, map and scan)
constexpr uint32_t kRec = 135168;

// ---- shared memory (bytes from a 1024-aligned base)
constexpr uint32_t sKQ = 0;          // K kb0 | Q kb0 | K kb1 | Q kb1 (8 KB bf16 tiles); later
                                     //   (Gamma.K) hi in the K places, lo in the Q places
constexpr uint32_t sG = 32768;       // fp32 [64][128]: log-decay, then cumulative g
constexpr uint32_t sA = 65536;       // Gram A image: [K~ ; Q~] hi (32 KB) | lo (32 KB); before
                                     //   it fp32 [64][128]: KDN omega -> p^, PKDA bound B(A)
constexpr uint32_t sB = 131072;      // Gram B image: 160 rows x 128, hi (40 KB) | lo (40 KB)
constexpr uint32_t sLT = sB;                    // after the Gram: L/T fp32 [64][LDL]
constexpr uint32_t sXS = sB + 64 * LDL * 4;     //   inverse scratch [64][LDX]
constexpr uint32_t sTi = sB + 32768;            //   T hi | T lo (the W' MMA's B operand)
constexpr uint32_t sGK = sB + 49152;            //   (Gamma.K) hi [64 tok][128] (two 8 KB
                                                //   channel blocks), then lo at +16 KB
constexpr uint32_t sVec = 212992;    // vectors below
constexpr int kTokVecs = 13;         // per-token vectors of 64 floats
constexpr int kChVecs = 15;          // per-channel vectors of 128 floats
constexpr uint32_t kSmem = sVec + (kTokVecs * 64 + kChVecs * 128) * 4 + 1024;
static_assert(kSmem <= 232448, "shared memory per block");
constexpr uint32_t kBBlk = 20480;    // one 64-channel block of the B image (160 rows)
constexpr uint32_t kBLo = 40960;

constexpr uint32_t tGram = 0;        // TMEM: Gram, M = 128 x N = 160
constexpr uint32_t tW = 256;         // W', M = 128 x N = 128 (T hi | T lo products)
constexpr uint32_t kTmem = 512;
constexpr uint32_t I_GR = idesc_bf16(128, 160, 0, 0);
constexpr uint32_t I_WT = idesc_bf16(128, 128, 1, 0);    // A = Gamma.K (MN-major), B = T (K-major)
constexpr uint32_t I_WT64 = idesc_bf16(128, 64, 1, 0);

enum { B_KQ, B_LA, B_OM, B_GRAM, B_WP, B_COUNT };

// B-operand row of token j in sub-chunk I's block (blocks of 16, 32, 48, 64 rows)
__device__ __forceinline__ int brow(int I, int j) { return 8 * I * (I + 1) + j; }
// index of the pair (I, J), J < I, among the 6 strictly lower sub-chunk pairs
__device__ __forceinline__ int pair_index(int I, int J) { return I * (I - 1) / 2 + J; }

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ void st_global16(uint8_t* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}

template <int VARIANT>
__global__ void __launch_bounds__(kThreads, 1)
    pc_prep_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmLA, const __grid_constant__ CUtensorMap tmOM,
                   FwdArgs a, uint8_t* __restrict__ ws, uint32_t* __restrict__ chain) {
  constexpr bool kKdn = VARIANT == DR_KDN;
  constexpr bool kPkda = VARIANT == DR_PKDA;
  constexpr bool kIkdn = VARIANT == DR_IKDN;
  constexpr bool kF = kKdn || kPkda;   // a per-element factor of w in the fp32 buffer at sA
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  __shared__ uint64_t bars[B_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ int s_ok;
  __shared__ long s_next;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NC = (a.T + 63) / 64;
  const long nrow = (long)a.B * a.H;
  const long ntask = nrow * NC;
  const bool chained = chain != nullptr;

  float* fG_ = reinterpret_cast<float*>(sm + sG);   // [64][128]
  float* fA_ = reinterpret_cast<float*>(sm + sA);   // [64][128] (before the A image)
  float* vcr = reinterpret_cast<float*>(sm + sVec); // key normalisation
  float* vqn = vcr + 64;    // query normalisation
  float* vkn = vqn + 64;    // ||k^||^2
  float* vsc = vkn + 64;    // per-token scale of w
  float* vr = vsc + 64;     // observation noise r (KDN, isotropic KDN)
  float* vus = vr + 64;     // information scale / r (KDN)
  float* veta = vus + 64;   // eta (KDA, PKDA)
  float* vaP = veta + 64;   // PKDA statistic decay and gain
  float* vbP = vaP + 64;
  float* vom = vbP + 64;    // isotropic KDN process noise (per token)
  float* vaa = vom + 64;    // isotropic KDN mean squared decay
  float* vkk = vaa + 64;    // raw ||k||^2, ||q||^2
  float* vqq = vkk + 64;
  float* fEm = vqq + 64;            // [4][128] exp(g_m(I))
  float* fF = fEm + 4 * 128;        // [6][128] exp(g_m(I) - g_m(J)), J < I
  float* fGm = fF + 6 * 128;        // [4][128] exp(g_C - g_m(J))
  float* fgC = fGm + 4 * 128;       // [128]    exp(g_C)

  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmLA);
    if (kKdn) tma_prefetch_desc(&tmOM);
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, kTmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;

  // task -> (row b h, chunk); tickets are chunk-major when chained (32-bit: a
  // launch has fewer than 2^31 tasks)
  const int nrow_i = (int)nrow;
  auto decode = [&](long it, int& bh, int& ci) {
    const int t = (int)it;
    if (chained) {
      ci = t / nrow_i;
      bh = t - ci * nrow_i;
    } else {
      bh = t / NC;
      ci = t - bh * NC;
    }
  };
  // issue counts per barrier (thread 0), for the drain after an abort
  int c_kq = 0, c_la = 0, c_om = 0, c_gram = 0, c_wp = 0;
  auto load_kq = [&](int bh, int ci) {
    const int b = bh / a.H, h = bh % a.H;
    uint8_t* base = sm + sKQ;
    mbar_expect_tx(&bars[B_KQ], 32768);
    tma_load_4d(base, &tmK, &bars[B_KQ], 0, h, ci * 64, b);
    tma_load_4d(base + 16384, &tmK, &bars[B_KQ], 64, h, ci * 64, b);
    tma_load_4d(base + 8192, &tmQ, &bars[B_KQ], 0, h, ci * 64, b);
    tma_load_4d(base + 24576, &tmQ, &bars[B_KQ], 64, h, ci * 64, b);
    ++c_kq;
  };
  auto load_la = [&](int bh, int ci) {
    mbar_expect_tx(&bars[B_LA], 32768);
    tma_load_4d(sm + sG, &tmLA, &bars[B_LA], 0, bh % a.H, ci * 64, bh / a.H);
    ++c_la;
  };
  auto load_om = [&](int bh, int ci) {
    mbar_expect_tx(&bars[B_OM], 32768);
    tma_load_4d(sm + sA, &tmOM, &bars[B_OM], 0, bh % a.H, ci * 64, bh / a.H);
    ++c_om;
  };
  // every thread waits for a barrier phase: thread 0 polls (bounded), the others
  // take its verdict
  auto cta_wait = [&](int id, uint32_t parity) -> bool {
    if (tid == 0) s_ok = mbar_wait(&bars[id], parity, kWait) ? 1 : 0;
    __syncthreads();
    const bool ok = s_ok != 0;
    __syncthreads();
    return ok;
  };

  // per-token gates of the next task, held in registers by threads 0..63
  float n_r = 1.f, n_eta = 0.f, n_aP = 1.f, n_bP = 0.f, n_om = 0.f;
  auto prefetch_gates = [&](int bh, int ci) {
    const int i = tid, tok = ci * 64 + i;
    const bool real = i < 64 && tok < a.T;
    const long ti = real ? ((long)(bh / a.H) * a.T + tok) * a.H + (bh % a.H) : 0;
    n_r = 1.f;
    n_eta = 0.f;
    n_aP = 1.f;
    n_bP = 0.f;
    n_om = 0.f;
    if (real) {
      if (kKdn || kIkdn) n_r = a.r[ti];
      if (!kKdn && !kIkdn) n_eta = a.eta[ti];
      if (kPkda) {
        n_aP = a.alphaP[ti];
        n_bP = a.betaP[ti];
      }
      if (kIkdn) n_om = a.omega[ti];
    }
  };

  long it;
  if (chained) {
    if (tid == 0) s_next = atomicAdd(chain + ntask, 1u);
    __syncthreads();
    it = s_next;
    __syncthreads();
  } else {
    it = blockIdx.x;
  }
  if (it < ntask) {
    int bh0, ci0;
    decode(it, bh0, ci0);
    if (tid == 0) {
      load_kq(bh0, ci0);
      load_la(bh0, ci0);
      if (kKdn) load_om(bh0, ci0);
    }
    if (tid < 64) prefetch_gates(bh0, ci0);
  }
  bool abort = false;

  for (int k = 0; it < ntask; ++k) {
    int bh, ci;
    decode(it, bh, ci);
    const int h = bh % a.H;
    const long ri = (long)bh * NC + ci;
    uint8_t* rec = ws + (size_t)ri * kRec;
    if (chained && tid == 0) s_next = atomicAdd(chain + ntask, 1u);
    if (!cta_wait(B_KQ, k & 1) || !cta_wait(B_LA, k & 1) || (kKdn && !cta_wait(B_OM, k & 1))) {
      abort = true;
      break;
    }
    const long nxt = chained ? s_next : it + gridDim.x;
    const bool has_next = nxt < ntask;
    int nbh = 0, nci = 0;
    if (has_next) decode(nxt, nbh, nci);

    // ---- 1. per-token gates and norms
    if (tid < 64) {
      vr[tid] = n_r;
      vus[tid] = a.info_scale / n_r;
      veta[tid] = n_eta;
      vaP[tid] = n_aP;
      vbP[tid] = n_bP;
      vom[tid] = n_om;
      if (has_next) prefetch_gates(nbh, nci);
    }
    if (tid < 256) {
      const uint8_t* KQ = sm + sKQ;
      const int i = tid >> 2, part = tid & 3, kb = part >> 1, c0 = (part & 1) * 32;
      float kk = 0.f, qq = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float fk[8], fq[8];
        unpack8(*reinterpret_cast<const uint4*>(KQ + kb * 16384 + sw128_offset(i, c0 + 8 * m)), fk);
        unpack8(*reinterpret_cast<const uint4*>(KQ + kb * 16384 + sw128_offset(64 + i, c0 + 8 * m)), fq);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          kk += fk[e] * fk[e];
          qq += fq[e] * fq[e];
        }
      }
      kk += __shfl_xor_sync(0xffffffffu, kk, 1);
      kk += __shfl_xor_sync(0xffffffffu, kk, 2);
      qq += __shfl_xor_sync(0xffffffffu, qq, 1);
      qq += __shfl_xor_sync(0xffffffffu, qq, 2);
      if (part == 0) {
        const float cr = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
        vcr[i] = cr;
        vqn[i] = a.q_l2norm ? 1.f / fmaxf(sqrtf(qq), 1e-30f) : 1.f;
        vkn[i] = kk * cr * cr;
      }
    }
    // ---- 2. scans.  First every term off the recurrences' chains, for all (token,
    //         channel) at once in the B-image region (free until the B pass): KDN
    //         a^2 and u = (information scale / r) k^2, PKDA betaP k^2.  Then the
    //         channels' recurrences: cumulative log-decay g, KDN variance, PKDA
    //         statistic; isotropic KDN: warp 4 scans the head variance.
    float* fX_ = reinterpret_cast<float*>(sm + sB);   // [64][128] KDN a^2
    float* fY_ = fX_ + 64 * 128;                      // [64][128] KDN u, PKDA betaP k^2
    float st = 0.f;   // the gain state at the chunk start
    if (kKdn || kPkda) {
      // Four threads per channel (part = tid / 128 takes tokens 16 part .. + 15).  Each
      // first composes its tokens' maps of (n, d) — KDN M = [[a^2, w], [u a^2, 1 + u w]],
      // PKDA n <- alphaP n + betaP k^2 (d = 1) — and its log-decay sum, before the
      // hand-over wait; after it, the chunk-start state through the parts' maps gives
      // each part its start and the chunk's end state (handed over at once), and only
      // then does each part walk its tokens.
      __syncthreads();   // the norms
#pragma unroll 2
      for (int r = 0; r < kUnits; ++r) {
        const int u = tid + r * kThreads, i = u >> 4, cg = u & 15, kb = cg >> 3, c8 = (cg & 7) * 8;
        const int cc = 64 * kb + c8;
        float k8[8], y[8];
        unpack8(*reinterpret_cast<const uint4*>(sm + sKQ + kb * 16384 + sw128_offset(i, c8)), k8);
        const float cr = vcr[i], sc = kKdn ? vus[i] : vbP[i];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float kh = k8[e] * cr;   // normalised first: cr is 1e30 on padding rows
          y[e] = sc * kh * kh;
        }
        float4* yp = reinterpret_cast<float4*>(fY_ + i * 128 + cc);
        yp[0] = make_float4(y[0], y[1], y[2], y[3]);
        yp[1] = make_float4(y[4], y[5], y[6], y[7]);
        if (kKdn) {
          const float4* lp = reinterpret_cast<const float4*>(fG_ + i * 128 + cc);
          const float4 l0 = lp[0], l1 = lp[1];
          float4* xp = reinterpret_cast<float4*>(fX_ + i * 128 + cc);
          xp[0] = make_float4(__expf(2.f * l0.x), __expf(2.f * l0.y), __expf(2.f * l0.z), __expf(2.f * l0.w));
          xp[1] = make_float4(__expf(2.f * l1.x), __expf(2.f * l1.y), __expf(2.f * l1.z), __expf(2.f * l1.w));
        }
      }
      __syncthreads();
      const int c = tid & 127, part = tid >> 7, i0 = 16 * part;
      float P0 = 1.f, P1 = 0.f, P2 = 0.f, P3 = 1.f, gs = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int o = (i0 + e) * 128 + c;
        gs += fG_[o];
        const float y = fY_[o];
        if (kKdn) {
          const float x = fX_[o], om = fA_[o];
          const float q0 = fmaf(x, P0, om * P2), q1 = fmaf(x, P1, om * P3);
          P2 = fmaf(y, q0, P2);
          P3 = fmaf(y, q1, P3);
          P0 = q0;
          P1 = q1;
          if ((e & 7) == 7) {   // exact power-of-two rescale (the map acts projectively)
            const float sc = __uint_as_float(0x7f000000u - (__float_as_uint(fmaxf(P3, P2)) & 0x7f800000u));
            P0 *= sc;
            P1 *= sc;
            P2 *= sc;
            P3 *= sc;
          }
        } else {
          const float x = vaP[i0 + e];
          P0 *= x;
          P1 = fmaf(x, P1, y);
        }
      }
      float4* sMap = reinterpret_cast<float4*>(sm + sB + 65536);       // [4][128] part maps
      float* sGs = reinterpret_cast<float*>(sm + sB + 65536 + 8192);   // [4][128] part sums
      sMap[part * 128 + c] = make_float4(P0, P1, P2, P3);
      sGs[part * 128 + c] = gs;
      // the chained gain state: wait for the previous chunk's hand-over
      if (chained && ci > 0 && tid == 0 && !chain_wait(chain + ri, chain + ntask + 1, g_chain_wait_ns))
        set_status(DR_ERR_TIMEOUT);
      __syncthreads();
      if (chained)
        st = ci == 0 ? (a.aux0 ? a.aux0[(long)bh * 128 + c] : (kKdn ? 1.f : 0.f))
                     : __ldcg(reinterpret_cast<const float*>(rec + rkP0) + c);
      else
        st = reinterpret_cast<const float*>(rec + rkP0)[c];
      float g = 0.f, n = st, d = 1.f;
      auto apply = [&](const float4& Q) {
        const float n1 = fmaf(Q.x, n, Q.y * d), d1 = fmaf(Q.z, n, Q.w * d);
        const float sc = kKdn ? __uint_as_float(0x7f000000u - (__float_as_uint(d1) & 0x7f800000u)) : 1.f;
        n = n1 * sc;
        d = d1 * sc;
      };
      for (int q = 0; q < part; ++q) {
        g += sGs[q * 128 + c];
        apply(sMap[q * 128 + c]);
      }
      if (chained && part == 3) {   // state at the chunk end -> next record, or aux
        const float ns = n, ds = d;
        apply(make_float4(P0, P1, P2, P3));
        const float end = kKdn ? n / d : n;
        n = ns;
        d = ds;
        if (ci + 1 < NC)   // published by thread 0's release after the barrier below
          __stcg(reinterpret_cast<float*>(rec + kRec + rkP0) + c, end);
        else if (a.aux)
          a.aux[(long)bh * 128 + c] = end;
      }
      __syncthreads();
      // every thread's hand-over store precedes the barrier; thread 0's release store
      // publishes them at GPU scope (release semantics are cumulative over the barrier)
      if (chained && tid == 0 && ci + 1 < NC && ri + 1 != g_chain_withhold)
        st_release_gpu(chain + ri + 1, 1u);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int o = (i0 + e) * 128 + c;
        g += fG_[o];
        fG_[o] = g;
        const float y = fY_[o];
        if (kKdn) {   // p^_i = n_i / d_{i-1}
          const float n1 = fmaf(fX_[o], n, fA_[o] * d);
          fA_[o] = __fdividef(n1, d);
          d = fmaf(y, n1, d);
          n = n1;
          if ((e & 7) == 7) {   // exact power-of-two rescale to d in [1, 2) (d >= 1)
            const float sc = __uint_as_float(0x7f000000u - (__float_as_uint(d) & 0x7f800000u));
            n *= sc;
            d *= sc;
          }
        } else {   // A_t = alphaP A + betaP k^2 (the bound follows below)
          n = fmaf(vaP[i0 + e], n, y);
          fA_[o] = n;
        }
      }
      __syncthreads();
    } else {
      // the chained gain state (isotropic KDN): wait for the previous chunk's hand-over
      if (chained && ci > 0 && kIkdn && tid == 0 && !chain_wait(chain + ri, chain + ntask + 1, g_chain_wait_ns))
        set_status(DR_ERR_TIMEOUT);
      __syncthreads();
      if (kIkdn && warp == 4) {
        st = 1.f;
        if (chained)
          st = ci == 0 ? (a.aux0 ? a.aux0[bh] : 1.f) : __ldcg(reinterpret_cast<const float*>(rec + rkP0));
      }
      if (kIkdn) {   // mean squared decay of every token (warp w: tokens 8w .. 8w + 7)
#pragma unroll
        for (int rr = 0; rr < 64 / kWarps; ++rr) {
          const int i = (64 / kWarps) * warp + rr;
          float s2 = 0.f;
#pragma unroll
          for (int c = lane; c < 128; c += 32) s2 += __expf(2.f * fG_[i * 128 + c]);
          s2 = warp_sum(s2);
          if (lane == 0) vaa[i] = s2 * (1.f / 128.f);
        }
        __syncthreads();
      }

      if (tid < 128) {   // the cumulative log-decay, channel tid
        const int c = tid;
        float g = 0.f;
#pragma unroll 8
        for (int i = 0; i < 64; ++i) {
          g += fG_[i * 128 + c];
          fG_[i * 128 + c] = g;
        }
      }
      if (kIkdn && warp == 4) {
        // b -> b^ / (1 + u b^), b^ = a b + omega is the Moebius map of (n, d) by
        // M = [[a, omega], [u a, 1 + u omega]]: two tokens' product per lane, a shuffle
        // scan of 2x2 products (each rescaled by an exact power of two), then b^ of
        // every token and beta = b^ / (r + b^ ||k^||^2) (KDN notes Eq. (40))
        auto mmul = [](const float (&A)[4], const float (&B)[4], float (&C)[4]) {
          C[0] = A[0] * B[0] + A[1] * B[2];
          C[1] = A[0] * B[1] + A[1] * B[3];
          C[2] = A[2] * B[0] + A[3] * B[2];
          C[3] = A[2] * B[1] + A[3] * B[3];
        };
        auto renorm = [](float (&C)[4]) {
          int ex;
          frexpf(fmaxf(fmaxf(fabsf(C[0]), fabsf(C[1])), fmaxf(fabsf(C[2]), fabsf(C[3]))), &ex);
#pragma unroll
          for (int z = 0; z < 4; ++z) C[z] = ldexpf(C[z], -ex);
        };
        auto token = [&](int i, float (&M)[4]) {
          const float at = vaa[i], om = vom[i], u = a.info_scale * vkn[i] / (128.f * vr[i]);
          M[0] = at;
          M[1] = om;
          M[2] = u * at;
          M[3] = 1.f + u * om;
        };
        const float b_in = st;
        float M0[4], M1[4], Pl[4];
        token(2 * lane, M0);
        token(2 * lane + 1, M1);
        mmul(M1, M0, Pl);
        renorm(Pl);
#pragma unroll
        for (int dd = 1; dd < 32; dd <<= 1) {
          float Q[4], R[4];
#pragma unroll
          for (int z = 0; z < 4; ++z) Q[z] = __shfl_up_sync(0xffffffffu, Pl[z], dd);
          if (lane >= dd) {
            mmul(Pl, Q, R);
#pragma unroll
            for (int z = 0; z < 4; ++z) Pl[z] = R[z];
            renorm(Pl);
          }
        }
        float E[4];
#pragma unroll
        for (int z = 0; z < 4; ++z) E[z] = __shfl_up_sync(0xffffffffu, Pl[z], 1);
        if (lane == 0) {
          E[0] = 1.f;
          E[1] = 0.f;
          E[2] = 0.f;
          E[3] = 1.f;
        }
        const float n0 = E[0] * b_in + E[1], d0 = E[2] * b_in + E[3];
        const float bh0 = vaa[2 * lane] * __fdividef(n0, d0) + vom[2 * lane];
        const float n1 = M0[0] * n0 + M0[1] * d0, d1 = M0[2] * n0 + M0[3] * d0;
        const float bh1 = vaa[2 * lane + 1] * __fdividef(n1, d1) + vom[2 * lane + 1];
        vsc[2 * lane] = __fdividef(bh0, vr[2 * lane] + bh0 * vkn[2 * lane]);
        vsc[2 * lane + 1] = __fdividef(bh1, vr[2 * lane + 1] + bh1 * vkn[2 * lane + 1]);
        const float nE = Pl[0] * b_in + Pl[1], dE = Pl[2] * b_in + Pl[3];
        const float b_end = __shfl_sync(0xffffffffu, __fdividef(nE, dE), 31);
        if (lane == 0 && chained) {
          if (ci + 1 < NC)
            __stcg(reinterpret_cast<float*>(rec + kRec + rkP0), b_end);
          else if (a.aux)
            a.aux[bh] = b_end;
        }
      }
      __syncthreads();
      // every thread's hand-over store precedes the barrier; thread 0's release store
      // publishes them at GPU scope (release semantics are cumulative over the barrier)
      if (chained && (kKdn || kPkda || kIkdn) && tid == 0 && ci + 1 < NC && ri + 1 != g_chain_withhold)
        st_release_gpu(chain + ri + 1, 1u);
    }
    if (kPkda) {   // the bound B(A) = exp(-ln(x) r / (1 + |r|)), r = log max(A, floor) - mu
                   // (PDN notes Eq. (9); fast log / exp), in place
      const float mu_h = a.mu[h];
      float4* f4 = reinterpret_cast<float4*>(fA_);
#pragma unroll 2
      for (int e4 = tid; e4 < 64 * 128 / 4; e4 += kThreads) {
        float4 v = f4[e4];
        float* x = reinterpret_cast<float*>(&v);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float rr = __logf(fmaxf(x[e], a.log_floor)) - mu_h;
          x[e] = __expf(-a.ln_x * __fdividef(rr, 1.f + fabsf(rr)));
        }
        f4[e4] = v;
      }
    }

    // ---- 3. per-token write scale; per-channel factors of the sub-chunk references
    if (kKdn && tid < 256) {   // 1 / (r_i + sum_c p^_ic k^_ic^2): four threads per token
      const int i = tid >> 2, part = tid & 3, kb = part >> 1, c0 = (part & 1) * 32;
      const uint8_t* KQ = sm + sKQ;
      float z = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float k8[8];
        unpack8(*reinterpret_cast<const uint4*>(KQ + kb * 16384 + sw128_offset(i, c0 + 8 * m)), k8);
        const float4* pp = reinterpret_cast<const float4*>(fA_ + i * 128 + 64 * kb + c0 + 8 * m);
        const float4 p0 = pp[0], p1 = pp[1];
        const float p8[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) z += p8[e] * k8[e] * k8[e];
      }
      z += __shfl_xor_sync(0xffffffffu, z, 1);
      z += __shfl_xor_sync(0xffffffffu, z, 2);
      if (part == 0) vsc[i] = 1.f / (vr[i] + z * vcr[i] * vcr[i]);
    } else if (!kIkdn) {
      if (tid < 64) vsc[tid] = veta[tid];
    }
    for (int e = tid; e < kChVecs * 128; e += kThreads) {
      const int v = e >> 7, c = e & 127;
      const float gC = fG_[63 * 128 + c];
      float x;
      if (v < 4) {
        x = fG_[(16 * v + 7) * 128 + c];
      } else if (v < 10) {
        const int p = v - 4, I = p < 1 ? 1 : (p < 3 ? 2 : 3), J = p - I * (I - 1) / 2;
        x = fG_[(16 * I + 7) * 128 + c] - fG_[(16 * J + 7) * 128 + c];
      } else if (v < 14) {
        x = gC - fG_[(16 * (v - 10) + 7) * 128 + c];
      } else {
        x = gC;
      }
      fEm[e] = __expf(x);   // fEm, fF, fGm, fgC are consecutive
    }
    __syncthreads();

    // ---- 4. B image: for token j of sub-chunk J, w~_j = w_j exp(g_m(J) - g_j), then
    //         block I >= J gets w~_j exp(g_m(I) - g_m(J)).  Unit = (token, 8 channels).
#pragma unroll 2
    for (int r = 0; r < kUnits; ++r) {
      const int u = tid + r * kThreads, j = u >> 4, cg = u & 15, kb = cg >> 3, c8 = (cg & 7) * 8;
      const int cc = 64 * kb + c8, J = j >> 4;
      float k8[8];
      unpack8(*reinterpret_cast<const uint4*>(sm + sKQ + kb * 16384 + sw128_offset(j, c8)), k8);
      const float4* gp = reinterpret_cast<const float4*>(fG_ + j * 128 + cc);
      const float4* mp = reinterpret_cast<const float4*>(fG_ + (16 * J + 7) * 128 + cc);
      const float4 g0 = gp[0], g1 = gp[1], m0 = mp[0], m1 = mp[1];
      const float gj[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const float gm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
      float f8[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
      if (kF) {
        const float4* fp = reinterpret_cast<const float4*>(fA_ + j * 128 + cc);
        const float4 f0 = fp[0], f1 = fp[1];
        f8[0] = f0.x; f8[1] = f0.y; f8[2] = f0.z; f8[3] = f0.w;
        f8[4] = f1.x; f8[5] = f1.y; f8[6] = f1.z; f8[7] = f1.w;
      }
      const float s = vsc[j] * vcr[j];
      float w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = s * k8[e] * f8[e];
      if (a.save_W) {   // backward: the write vectors themselves
        float4* sw = reinterpret_cast<float4*>(a.save_W + ((size_t)ri * 64 + j) * 128 + cc);
        sw[0] = make_float4(w[0], w[1], w[2], w[3]);
        sw[1] = make_float4(w[4], w[5], w[6], w[7]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] *= __expf(gm[e] - gj[e]);
      uint4 hi, lo;
#pragma unroll 1
      for (int I = J; I < 4; ++I) {
        float x[8];
        if (I == J) {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = w[e];
        } else {   // two 16-byte loads (8 scalar loads of a channel vector conflict 4 ways)
          const float4* F = reinterpret_cast<const float4*>(fF + pair_index(I, J) * 128 + cc);
          const float4 f0 = F[0], f1 = F[1];
          const float ff[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = w[e] * ff[e];
        }
        split8(x, hi, lo);
        const uint32_t off = sB + kb * kBBlk + sw128_offset(brow(I, j), c8);
        *reinterpret_cast<uint4*>(sm + off) = hi;
        *reinterpret_cast<uint4*>(sm + off + kBLo) = lo;
      }
    }
    __syncthreads();

    // ---- 5. A image [K~ ; Q~] = [k^_i ; q^_i] exp(g_i - g_m(I))
#pragma unroll 2
    for (int r = 0; r < kUnits; ++r) {
      const int u = tid + r * kThreads, i = u >> 4, cg = u & 15, kb = cg >> 3, c8 = (cg & 7) * 8;
      const int cc = 64 * kb + c8, I = i >> 4;
      const uint8_t* kp = sm + sKQ + kb * 16384 + sw128_offset(i, c8);
      const uint8_t* qp = sm + sKQ + kb * 16384 + sw128_offset(64 + i, c8);
      float k8[8], q8[8];
      unpack8(*reinterpret_cast<const uint4*>(kp), k8);
      unpack8(*reinterpret_cast<const uint4*>(qp), q8);
      const float4* gp = reinterpret_cast<const float4*>(fG_ + i * 128 + cc);
      const float4* mp = reinterpret_cast<const float4*>(fG_ + (16 * I + 7) * 128 + cc);
      const float4 g0 = gp[0], g1 = gp[1], m0 = mp[0], m1 = mp[1];
      const float gi[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      const float gm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
      const float cr = vcr[i], qn = vqn[i];
      float xk[8], xq[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float f = __expf(gi[e] - gm[e]);
        xk[e] = k8[e] * cr * f;
        xq[e] = q8[e] * qn * f;
      }
      uint4 hi, lo;
      split8(xk, hi, lo);
      const uint32_t ok = sA + kb * 16384 + sw128_offset(i, c8);
      *reinterpret_cast<uint4*>(sm + ok) = hi;
      *reinterpret_cast<uint4*>(sm + ok + 32768) = lo;
      split8(xq, hi, lo);
      const uint32_t oq = sA + kb * 16384 + sw128_offset(64 + i, c8);
      *reinterpret_cast<uint4*>(sm + oq) = hi;
      *reinterpret_cast<uint4*>(sm + oq + 32768) = lo;
    }
    if (tid < 128) {
      float* rv = reinterpret_cast<float*>(rec + rbVec);
      rv[tid] = 1.f;           // e^g qn and u slots: folded into (Gamma.Q) and Wbar
      rv[128 + tid] = fgC[tid];
    }
    fence_proxy_async();
    __syncthreads();

    // ---- 6. the Gram [K~ ; Q~] B^T (three hi/lo products); the next task's K / Q and
    //         log-decay tiles may load now
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ab = smem_u32(sm + sA), bb = smem_u32(sm + sB);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
        const uint64_t dah = desc_sw128(ab + kb * 16384 + ko, 16, 1024);
        const uint64_t dal = desc_sw128(ab + 32768 + kb * 16384 + ko, 16, 1024);
        const uint64_t dbh = desc_sw128(bb + kb * kBBlk + ko, 16, 1024);
        const uint64_t dbl = desc_sw128(bb + kBLo + kb * kBBlk + ko, 16, 1024);
        mma_bf16(tmem + tGram, dah, dbh, I_GR, ks > 0);
        mma_bf16(tmem + tGram, dah, dbl, I_GR, true);
        mma_bf16(tmem + tGram, dal, dbh, I_GR, true);
      }
      mma_commit(&bars[B_GRAM]);
      ++c_gram;
      if (has_next) {
        load_kq(nbh, nci);
        load_la(nbh, nci);
      }
    }
    // While the Gram runs (its operands are only read): (Gamma.Q) = Q~ exp(g_m(I)) and
    // Wbar = B_3 exp(g_C - g_m(3)) (block 3 of the B image holds every token's
    // w_j exp(g_m(3) - g_j)) to the record from the images' hi + lo, and (Gamma.K) =
    // K~ exp(g_m(I)) into registers, stored once the B image is free.
    uint4 gk_hi[kUnits], gk_lo[kUnits];
#pragma unroll
    for (int r = 0; r < kUnits; ++r) {
      const int u = tid + r * kThreads, i = u >> 4, cg = u & 15, kb = cg >> 3, c8 = (cg & 7) * 8;
      const int cc = 64 * kb + c8;
      float Em[8], G3[8];
      {
        const float4* ep = reinterpret_cast<const float4*>(fEm + (i >> 4) * 128 + cc);
        const float4* gp = reinterpret_cast<const float4*>(fGm + 3 * 128 + cc);
        const float4 e0 = ep[0], e1 = ep[1], g0 = gp[0], g1 = gp[1];
        Em[0] = e0.x; Em[1] = e0.y; Em[2] = e0.z; Em[3] = e0.w;
        Em[4] = e1.x; Em[5] = e1.y; Em[6] = e1.z; Em[7] = e1.w;
        G3[0] = g0.x; G3[1] = g0.y; G3[2] = g0.z; G3[3] = g0.w;
        G3[4] = g1.x; G3[5] = g1.y; G3[6] = g1.z; G3[7] = g1.w;
      }
      const uint32_t ok = sA + kb * 16384 + sw128_offset(i, c8);
      const uint32_t oq = sA + kb * 16384 + sw128_offset(64 + i, c8);
      const uint32_t ob = sB + kb * kBBlk + sw128_offset(brow(3, i), c8);
      float xh[8], xl[8], y[8];
      uint4 hi, lo;
      unpack8(*reinterpret_cast<const uint4*>(sm + oq), xh);
      unpack8(*reinterpret_cast<const uint4*>(sm + oq + 32768), xl);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = (xh[e] + xl[e]) * Em[e];
      split8(y, hi, lo);
      const uint32_t og = kb * 8192 + sw128_offset(i, c8);
      st_global16(rec + rbQ + og, hi);
      st_global16(rec + rbQ + 16384 + og, lo);
      unpack8(*reinterpret_cast<const uint4*>(sm + ob), xh);
      unpack8(*reinterpret_cast<const uint4*>(sm + ob + kBLo), xl);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = (xh[e] + xl[e]) * G3[e];
      split8(y, hi, lo);
      st_global16(rec + rbW + og, hi);
      st_global16(rec + rbW + 16384 + og, lo);
      unpack8(*reinterpret_cast<const uint4*>(sm + ok), xh);
      unpack8(*reinterpret_cast<const uint4*>(sm + ok + 32768), xl);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = (xh[e] + xl[e]) * Em[e];
      split8(y, gk_hi[r], gk_lo[r]);
    }
    if (!cta_wait(B_GRAM, k & 1)) {
      abort = true;
      break;
    }
    tc_fence_after();

    // ---- 7. Gram readout: row r < 64 -> L (fp32, j < i), r >= 64 -> P (j <= i) as a
    //         bf16 hi/lo image in the record.  Row i of sub-chunk I finds its columns
    //         j = 0 .. 16 I + 15 at brow(I, j); warps of a TMEM quadrant split its
    //         16-column pieces.
    {
      const int q = warp & 3, pch = warp >> 2, npch = kWarps / 4;
      const int row = 32 * q + lane, i = row & 63, I = i >> 4;
      const bool isq = row >= 64;
      float* LT = reinterpret_cast<float*>(sm + sLT);
      const int pb = (q & 1) ? 3 : 0, pe = (q & 1) ? 10 : 3;
      const int p0 = I * (I + 1) / 2;   // first piece of this row's block
      for (int p = pb + pch; p < pe; p += npch) {
        float v[16];
        tmem_ld16(tmem + lane_off + tGram + 16 * p, v);
        tmem_ld_wait();
        const int jc = p - p0;
        if (jc >= 0 && jc <= I) {
          const int j0 = 16 * jc;
          float x[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = j0 + e;
            x[e] = (isq ? j <= i : j < i) ? v[e] : 0.f;
          }
          if (!isq) {
#pragma unroll
            for (int e = 0; e < 16; e += 4)
              *reinterpret_cast<float4*>(LT + i * LDL + j0 + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
          } else {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              float y[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) y[e] = x[8 * hh + e];
              uint4 hi, lo;
              split8(y, hi, lo);
              const uint32_t off = sw128_offset(i, j0 + 8 * hh);
              st_global16(rec + rbP + off, hi);
              st_global16(rec + rbP + 8192 + off, lo);
            }
          }
        }
      }
      for (int jc = I + 1 + pch; jc < 4; jc += npch) {   // above the row's block: zero
        if (!isq) {
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(LT + i * LDL + 16 * jc + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t off = sw128_offset(i, 16 * jc + 8 * hh);
            st_global16(rec + rbP + off, z);
            st_global16(rec + rbP + 8192 + off, z);
          }
        }
      }
    }
    // (Gamma.K) as the W' MMA's A operand [64 tok][128] (MN-major, two 64-channel
    // blocks 8 KB apart)
#pragma unroll
    for (int r = 0; r < kUnits; ++r) {
      const int u = tid + r * kThreads, i = u >> 4, cg = u & 15, kb = cg >> 3, c8 = (cg & 7) * 8;
      const uint32_t og = sGK + kb * 8192 + sw128_offset(i, c8);
      *reinterpret_cast<uint4*>(sm + og) = gk_hi[r];
      *reinterpret_cast<uint4*>(sm + og + 16384) = gk_lo[r];
    }
    tc_fence_before();
    __syncthreads();
    if (kKdn && tid == 0 && has_next) load_om(nbh, nci);   // the A image has been read

    // ---- 8. T = (I + L)^-1 in place: diagonal 16x16 blocks (threads 0-63, a column each)
    float* LT = reinterpret_cast<float*>(sm + sLT);
    float* XS = reinterpret_cast<float*>(sm + sXS);
    {
      const int j = tid & 15, I = (tid >> 4) & 3, r0 = 16 * I;
      float tt[16];
#pragma unroll
      for (int l = 0; l < 16; ++l) tt[l] = (l == j) ? 1.f : 0.f;
      if (tid < 64) {
#pragma unroll
        for (int i = 1; i < 16; ++i) {
          float s = 0.f;
#pragma unroll
          for (int l = 0; l < i; ++l) s += LT[(r0 + i) * LDL + r0 + l] * tt[l];
          if (i > j) tt[i] = -s;
        }
      }
      __syncthreads();
      if (tid < 64) {
#pragma unroll
        for (int i = 0; i < 16; ++i) LT[(r0 + i) * LDL + r0 + j] = tt[i];
      }
    }
    __syncthreads();
    // level 1: T_10, T_32; level 2: the 32 x 32 lower-left block
    if (warp < 4) {
      const int blk = warp >> 1, nt = warp & 1;
      const int r0 = 32 * blk + 16, c0 = 32 * blk;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      tile_mm3b<2>(d, LT + r0 * LDL + c0, LDL, LT + c0 * LDL + c0 + 8 * nt, LDL, lane);
      tile_store(XS + 16 * blk * LDX + 8 * nt, LDX, d, 1.f, lane);
    }
    __syncthreads();
    if (warp < 4) {
      const int blk = warp >> 1, nt = warp & 1;
      const int r0 = 32 * blk + 16, c0 = 32 * blk;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      tile_mm3b<2>(d, LT + r0 * LDL + r0, LDL, XS + 16 * blk * LDX + 8 * nt, LDX, lane);
      tile_store(LT + r0 * LDL + c0 + 8 * nt, LDL, d, -1.f, lane);
    }
    __syncthreads();
    if (warp < 8) {
      const int mt = warp >> 2, nt = warp & 3;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      tile_mm3b<4>(d, LT + (32 + 16 * mt) * LDL, LDL, LT + 8 * nt, LDL, lane);
      tile_store(XS + 16 * mt * LDX + 8 * nt, LDX, d, 1.f, lane);
    }
    __syncthreads();
    if (warp < 8) {
      const int mt = warp >> 2, nt = warp & 3;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      if (mt == 0)
        tile_mm3b<2>(d, LT + 32 * LDL + 32, LDL, XS + 8 * nt, LDX, lane);
      else
        tile_mm3b<4>(d, LT + 48 * LDL + 32, LDL, XS + 8 * nt, LDX, lane);
      tile_store(LT + (32 + 16 * mt) * LDL + 8 * nt, LDL, d, -1.f, lane);
    }
    __syncthreads();

    // ---- 9. T as bf16 hi/lo: the record and the W' MMA's B operand [T_hi ; T_lo]
    if (tid < 256) {
      const int i = tid >> 2, c0 = (tid & 3) * 16;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = c0 + 8 * m + e;
          x[e] = (j <= i) ? LT[i * LDL + j] : 0.f;
        }
        uint4 hi, lo;
        split8(x, hi, lo);
        const uint32_t off = sw128_offset(i, c0 + 8 * m);
        *reinterpret_cast<uint4*>(sm + sTi + off) = hi;
        *reinterpret_cast<uint4*>(sm + sTi + 8192 + off) = lo;
        st_global16(rec + rbT + off, hi);
        st_global16(rec + rbT + 8192 + off, lo);
      }
    }
    fence_proxy_async();
    __syncthreads();

    // ---- 10. W'^T = (Gamma.K)^T T^T: [Gamma.K_hi] x [T_hi ; T_lo] (N = 128) plus
    //          [Gamma.K_lo] x T_hi (N = 64) into the first half
    if (tid == 0) {
      tc_fence_after();
      const uint32_t tb = smem_u32(sm + sTi), gk = smem_u32(sm + sGK);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + tW, desc_sw128(gk + ks * 2048, 8192, 1024), desc_sw128(tb + ks * 32, 16, 1024),
                 I_WT, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + tW, desc_sw128(gk + 16384 + ks * 2048, 8192, 1024),
                 desc_sw128(tb + ks * 32, 16, 1024), I_WT64, true);
      mma_commit(&bars[B_WP]);
      ++c_wp;
    }
    if (!cta_wait(B_WP, k & 1)) {
      abort = true;
      break;
    }
    tc_fence_after();
    {   // row = channel c (TMEM lane), 16 tokens per thread
      const int c = (warp & 3) * 32 + lane, pch = warp >> 2;
      float w[16];
      {
        float t16[16], u16[16];
        tmem_ld16(tmem + lane_off + tW + 16 * pch, t16);
        tmem_ld16(tmem + lane_off + tW + 64 + 16 * pch, u16);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = t16[e] + u16[e];
      }
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = w[8 * m + e];
        uint4 hi, lo;
        split8(x, hi, lo);
        const uint32_t off = sw128_offset(c, 16 * pch + 8 * m);
        st_global16(rec + rbWp + off, hi);
        st_global16(rec + rbWp + 16384 + off, lo);
      }
    }
    tc_fence_before();
    __syncthreads();
    it = nxt;
  }

  if (abort && tid == 0) {   // drain what this CTA may still have in flight, then report
    set_status(DR_ERR_TIMEOUT);
    if (c_kq) mbar_wait(&bars[B_KQ], (c_kq - 1) & 1, kWait / 4);
    if (c_la) mbar_wait(&bars[B_LA], (c_la - 1) & 1, kWait / 4);
    if (c_om) mbar_wait(&bars[B_OM], (c_om - 1) & 1, kWait / 4);
    if (c_gram) mbar_wait(&bars[B_GRAM], (c_gram - 1) & 1, kWait / 4);
    if (c_wp) mbar_wait(&bars[B_WP], (c_wp - 1) & 1, kWait / 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmem);
}

}  // namespace

bool pc_prep_supported(int variant, int dtype, int dk, int dv, int chunk) {
  return (variant == DR_KDN || variant == DR_KDA || variant == DR_PKDA || variant == DR_IKDN) &&
         dtype == DR_BF16 && dk == 128 && dv == 128 && chunk == 64;
}

// Launches the prep over every (b, h, chunk) task: one CTA per SM (at most one per
// task); chain = the hand-over flags (then the ticket and abort words), zeroed by
// the caller, or null when the gain state is already in the records (or absent).
cudaError_t launch_pc_prep(const FwdArgs& a, void* workspace, uint32_t* chain, int nsm, cudaStream_t st) {
  CUtensorMap mq, mk, mla, mom;
  if (!make_map(&mq, a.q, a.B, a.T, a.H, 128) || !make_map(&mk, a.k, a.B, a.T, a.H, 128) ||
      !make_map_f32(&mla, a.log_alpha, a.B, a.T, a.H))
    return cudaErrorInvalidValue;
  if (a.variant == DR_KDN) {
    if (!make_map_f32(&mom, a.omega, a.B, a.T, a.H)) return cudaErrorInvalidValue;
  } else {
    mom = mla;   // unused
  }
  const long ntask = (long)a.B * a.H * ((a.T + 63) / 64);
  const int grid = (int)(ntask < nsm ? ntask : nsm);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaErrorInvalidValue;
#define DR_PC(V_)                                                                           \
  if (a.variant == V_) {                                                                    \
    e = cudaFuncSetAttribute(pc_prep_kernel<V_>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             (int)kSmem);                                                   \
    if (e != cudaSuccess) return e;                                                         \
    pc_prep_kernel<V_><<<grid, kThreads, kSmem, st>>>(mq, mk, mla, mom, a, ws, chain);      \
    return cudaGetLastError();                                                              \
  }
  DR_PC(DR_KDN) DR_PC(DR_KDA) DR_PC(DR_PKDA) DR_PC(DR_IKDN)
#undef DR_PC
  return e;
}

}  // namespace dr
