// chunk_tc.cu — chunkwise forward on the 5th-generation tensor cores (tcgen05),
// bf16 operands, fp32 accumulators in tensor memory, TMA-fed.
//
// Scope: scalar decay (GDN, KLA, PGDN), bf16 q/k/v/out, dk = dv = 128, chunk 64.
// One CTA of 256 threads owns (b, h, one 64-column half of dv) and walks the
// chunks in order; its fp32 state slice S (128 x 64) lives in registers
// (thread = row, two warpgroups split the columns).
//
// Per chunk of C = 64 tokens with state S (KLA notes section 2.5, Eqs. (7)-(9),
// with a general write matrix W as in the PDN notes section 2.6):
//
//   gates   g = cumsum(log alpha), row norms, write coefficients
//   MMA 1   G = [K; Q] W^T                        (M=128, N=64, K=dk)
//   SIMT    L = strict_lower(G_K . e^{g_i-g_j}),  P = lower(G_Q . e^{g_i-g_j})
//           T = (I + L)^-1 in place (16x16 block forward substitution, fp32)
//   MMA 2   W' = (T diag(e^g c)) K,  U' = T V    (M=64)
//   MMA 3   E = U' - W' S   (accumulated onto U' with A negated),  QS = Q S
//   MMA 4   PE = P E,  dS = W^T (u . E)          (u_j = e^{g_C-g_j} x write coefficient)
//   SIMT    S <- gamma_C S + dS ;  o = e^{g} qn . QS + PE -> global
//
// Decay ratios come from log differences (KDN notes section 6, numerics).
// Precision: the raw bf16 K, Q, V tiles are used as MMA operands unchanged
// (they are exact), and every per-token scale is folded into an operand that
// is computed on chip anyway.  Those computed operands -- T, T diag(e^g c), W',
// P, E, u.E and S -- are fed as two bf16 terms (x = hi + lo, error ~2^-16; the
// lo x lo product is dropped).  W' needs its lo term for raw (unnormalised)
// keys, where E = U' - W' S cancels heavily.  All bounded waits give up with
// DR_ERR_TIMEOUT.
#include <cuda.h>

#include "dr_common.cuh"
#include "tc_common.cuh"

namespace dr {

namespace {

using namespace umma;
using namespace tc;

constexpr int kTcThreads = 256;
constexpr uint64_t kWaitLimit = 2000000000ull;   // 2 s per bounded wait

// shared-memory map (bytes from a 1024-aligned base).  The raw bf16 input tiles
// are never modified: every per-token scale is folded into an operand computed
// on chip, so no input is rounded twice.
constexpr uint32_t oKQ = 0;                     // 2 stages x [K rows 0-63 | Q rows 64-127] x 2 kblocks
constexpr uint32_t kKQBytes = 32768;
constexpr uint32_t oV = 2 * kKQBytes;           // V tile [64 tokens][64 cols]      8 KB
constexpr uint32_t oT = oV + 8192;              // T hi | T lo | Ts hi | Ts lo    32 KB
constexpr uint32_t oWp = oT + 32768;            // W' hi bf16 [64][128] (lo: E tiles) 16 KB
constexpr uint32_t oS = oWp + 16384;            // S hi | S lo  [128][64]          32 KB
constexpr uint32_t oP = oS + 32768;             // P hi | P lo  [64][64]           16 KB
constexpr uint32_t oE = oP + 16384;             // E hi | E lo | uE hi | uE lo     32 KB
constexpr uint32_t oW = oE + 32768;             // PGDN write keys [64][128]       16 KB
constexpr uint32_t oVec = oW + 16384;           // per-token vectors + scratch      8 KB
constexpr uint32_t kSmemBytes = oVec + 8192 + 1024;   // + alignment slack
constexpr int LDL = 68;                         // fp32 L/T row stride (aliases oE)
constexpr int LDX = 36;                         // fp32 scratch row stride (after L/T in oE)

// tensor-memory columns
constexpr uint32_t cGram = 0;    // M=128 x 64
constexpr uint32_t cWp = 64;     // M=64 x 128
constexpr uint32_t cE = 192;     // M=64 x 64   (U', then E)
constexpr uint32_t cQS = 256;    // M=64 x 64
constexpr uint32_t cPE = 320;    // M=64 x 64
constexpr uint32_t cDS = 384;    // M=128 x 64
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t ID_GRAM = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_WP = idesc_bf16(64, 128, 0, 1);
constexpr uint32_t ID_N64 = idesc_bf16(64, 64, 0, 1);
constexpr uint32_t ID_ENEG = idesc_bf16(64, 64, 0, 1, 1);
constexpr uint32_t ID_DS = idesc_bf16(128, 64, 1, 1);

template <int VARIANT>
__global__ void __launch_bounds__(kTcThreads, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar_kq[2];
  __shared__ uint64_t bar_v;
  __shared__ uint64_t bar_mma;
  __shared__ uint32_t tmem_base_s;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;          // TMEM lane quadrant of this warp
  const int chalf = warp >> 2;        // column half handled by this warpgroup
  const int half = blockIdx.x & 1;    // 64-column half of dv
  const int bh = blockIdx.x >> 1;
  const int b = bh / a.H, h = bh % a.H;
  const int NC = (a.T + 63) / 64;
  constexpr bool kPgdn = (VARIANT == DR_PGDN);

  float* vg = reinterpret_cast<float*>(sm + oVec);   // cumulative log-decay g_i
  float* va = vg + 64;      // coefficient of the raw key row in w (GDN/KLA); 1 for PGDN
  float* vcr = va + 64;     // key normalisation 1/||k|| (or 1)
  float* vqn = vcr + 64;    // query normalisation (or 1)
  float* vks = vqn + 64;    // e^{g_j} c_j: column scale of T giving W' = Ts K
  float* vqs = vks + 64;    // e^{g_i} qn_i: row scale of Q S
  float* vu = vqs + 64;     // e^{g_C - g_j} a_j: row scale of E giving dS = K^T (u.E)
  float* vla = vu + 64;
  float* veta = vla + 64;
  float* vaP = veta + 64;
  float* vbP = vaP + 64;
  float* vkk = vbP + 64;
  float* vqq = vkk + 64;
  float* vmisc = vqq + 64;  // [0] = gamma_C
  float* vC = vmisc + 128;  // [4 I][64 j] c_j e^{g_m(I) - g_j}: readout column factors
  float* LT = reinterpret_cast<float*>(sm + oE);     // L, inverted in place into T (fp32)
  float* XS = LT + 64 * LDL;                         // 32 x LDX fp32 scratch for the inverse

  if (tid == 0) {
    mbar_init(&bar_kq[0], 1);
    mbar_init(&bar_kq[1], 1);
    mbar_init(&bar_v, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    s_abort = 0;
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;

  // ---- state slice: row r = 32 quad + lane, columns 32 chalf + [0, 32)
  const int srow = quad * 32 + lane;
  float S[32];
  auto store_state_tiles = [&]() {
    uint8_t* sS = sm + oS;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = S[8 * m + e];
      uint4 hi, lo;
      split8(x, hi, lo);
      *reinterpret_cast<uint4*>(sS + sw128_offset(srow, chalf * 32 + 8 * m)) = hi;
      *reinterpret_cast<uint4*>(sS + 16384 + sw128_offset(srow, chalf * 32 + 8 * m)) = lo;
    }
  };
  {
    const long base = ((long)bh * 128 + srow) * a.dv + half * 64 + chalf * 32;
#pragma unroll
    for (int j = 0; j < 32; ++j) S[j] = a.S0 ? a.S0[base + j] : 0.f;
    store_state_tiles();
  }
  float carryA = 0.f;  // PGDN statistic for channel tid (tid < 128)
  if (kPgdn && tid < 128) carryA = a.aux0 ? a.aux0[(long)bh * 128 + tid] : 0.f;
  const float mu_h = kPgdn ? a.mu[h] : 0.f;

  auto issue_kq = [&](int c, int st) {
    uint8_t* base = sm + oKQ + st * kKQBytes;
    mbar_expect_tx(&bar_kq[st], kKQBytes);
    const int t0 = c * 64;
    tma_load_4d(base, &tmK, &bar_kq[st], 0, h, t0, b);
    tma_load_4d(base + 16384, &tmK, &bar_kq[st], 64, h, t0, b);
    tma_load_4d(base + 8192, &tmQ, &bar_kq[st], 0, h, t0, b);
    tma_load_4d(base + 16384 + 8192, &tmQ, &bar_kq[st], 64, h, t0, b);
  };
  auto issue_v = [&](int c) {
    mbar_expect_tx(&bar_v, 8192);
    tma_load_4d(sm + oV, &tmV, &bar_v, half * 64, h, c * 64, b);
  };
  if (tid == 0) {
    issue_kq(0, 0);
    issue_v(0);
  }
  fence_proxy_async();
  __syncthreads();

  // gates of the next chunk, prefetched into registers one chunk ahead (thread i < 64 = token i)
  float nla = 0.f, neta = 0.f, naP = 1.f, nbP = 0.f;
  auto prefetch_gates = [&](int c) {
    const int i = tid, t = c * 64 + i;
    if (i < 64 && t < a.T) {
      const long ti = ((long)b * a.T + t) * a.H + h;
      nla = a.log_alpha[ti];
      neta = a.eta[ti];
      if (kPgdn) {
        naP = a.alphaP[ti];
        nbP = a.betaP[ti];
      }
    } else {
      nla = 0.f; neta = 0.f; naP = 1.f; nbP = 0.f;
    }
  };
  prefetch_gates(0);

  uint32_t mma_phase = 0;
  bool bad = false;
  volatile int* abort_flag = &s_abort;
  auto wait_mma = [&]() {
    if (!*abort_flag && !mbar_wait(&bar_mma, mma_phase, kWaitLimit)) *abort_flag = 1;
    mma_phase ^= 1;
    tc_fence_after();
  };

  for (int c = 0; c < NC; ++c) {
    const int st = c & 1;
    uint8_t* KQ = sm + oKQ + st * kKQBytes;
    const int t0 = c * 64;
    const int Cc = min(64, a.T - t0);

    if (!mbar_wait(&bar_kq[st], (c >> 1) & 1, kWaitLimit)) s_abort = 1;
    __syncthreads();
    if (s_abort) break;
    if (tid == 0 && c + 1 < NC) issue_kq(c + 1, st ^ 1);

    // ---------------- 1. gates, norms, write coefficients
    if (tid < 64) {
      const int i = tid;
      vla[i] = nla;
      veta[i] = neta;
      if (kPgdn) {
        vaP[i] = naP;
        vbP[i] = nbP;
      }
    }
    if (c + 1 < NC) prefetch_gates(c + 1);
    {  // squared norms of k and q rows: 4 threads per row, 32 elements each
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
        vkk[i] = kk;
        vqq[i] = qq;
      }
    }
    __syncthreads();
    if (warp == 0) {  // inclusive scan of log-alpha, two tokens per lane
      const float x0 = vla[2 * lane], x1 = vla[2 * lane + 1];
      float s = x0 + x1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      vg[2 * lane] = s - x1;
      vg[2 * lane + 1] = s;
    }
    __syncthreads();
    if (tid < 64) {
      const int i = tid;
      const float gi = vg[i], gC = vg[63];
      const float kk = vkk[i], qq = vqq[i];
      const float cr = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
      const float qn = a.q_l2norm ? 1.f / fmaxf(sqrtf(qq), 1e-30f) : 1.f;
      float beta = veta[i];
      if (VARIANT == DR_KLA) beta = beta / (kk * cr * cr + a.eps);
      const float coef = kPgdn ? 1.f : beta * cr;
      va[i] = coef;
      vcr[i] = cr;
      vqn[i] = qn;
      const float eg = __expf(gi);
      vks[i] = eg * cr;
      vqs[i] = eg * qn;
      vu[i] = __expf(gC - gi) * coef;
      if (i == 0) vmisc[0] = __expf(gC);
    }
    __syncthreads();
    {
      const int I = tid >> 6, j = tid & 63;
      vC[tid] = va[j] * __expf(vg[16 * I + 7] - vg[j]);
    }
    __syncthreads();
    if (kPgdn) {  // statistic scan per channel -> write keys (K-major [64 tokens][128], 2 x 8 KB)
      uint8_t* Wt = sm + oW;
      if (tid < 128) {
        const int ch = tid, kb = ch >> 6, col = ch & 63;
        float A = carryA;
        for (int i0 = 0; i0 < 64; i0 += 8) {
          float kv[8], Av[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            kv[e] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                        KQ + kb * 16384 + sw128_offset(i0 + e, col))) * vcr[i0 + e];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            A = vaP[i0 + e] * A + vbP[i0 + e] * kv[e] * kv[e];
            Av[e] = A;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float rr = __logf(fmaxf(Av[e], a.log_floor)) - mu_h;
            const float sq = __fdividef(rr, 1.f + fabsf(rr));
            const float w = veta[i0 + e] * __expf(-a.ln_x * sq) * kv[e];
            *reinterpret_cast<__nv_bfloat16*>(Wt + kb * 8192 + sw128_offset(i0 + e, col)) =
                __float2bfloat16_rn(w);
          }
        }
        carryA = A;
      }
      fence_proxy_async();
      __syncthreads();
    }

    // ---------------- 2. MMA 1: Gram [K; Q] W^T  (W = raw K for GDN/KLA; write keys for PGDN)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t kq = smem_u32(KQ);
      const uint32_t wb = kPgdn ? smem_u32(sm + oW) : kq;
      const uint32_t wstride = kPgdn ? 8192 : 16384;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t da = desc_sw128(kq + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
        const uint64_t db = desc_sw128(wb + (ks >> 2) * wstride + (ks & 3) * 32, 16, 1024);
        mma_bf16(tmem + cGram, da, db, ID_GRAM, ks > 0);
      }
      mma_commit(&bar_mma);
    }
    wait_mma();

    // ---------------- 3. Gram readout: L (fp32, in the E area) and P (bf16 hi/lo)
    // warp (quad, chalf) reads rows 32 quad.. and columns 32 chalf..
    {
      const int row = quad * 32 + lane;          // lane of the M=128 accumulator
      const int i = row & 63, I = i >> 4;
      float gv[32];
      ld32cols(tmem + lane_off + cGram + chalf * 32, gv);
      tmem_ld_wait();
      // one reference token per 16-row block: G_ij [rs_i e^{g_i - g_m(I)}] [c_j e^{g_m(I) - g_j}]
      const float rf = ((row < 64) ? vcr[i] : vqn[i]) * __expf(vg[i] - vg[16 * I + 7]);
      const float* C = vC + I * 64 + chalf * 32;
      float x[32];
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 c4 = *reinterpret_cast<const float4*>(C + e);
        const int j = chalf * 32 + e;
        x[e] = (j <= i) ? gv[e] * rf * c4.x : 0.f;
        x[e + 1] = (j + 1 <= i) ? gv[e + 1] * rf * c4.y : 0.f;
        x[e + 2] = (j + 2 <= i) ? gv[e + 2] * rf * c4.z : 0.f;
        x[e + 3] = (j + 3 <= i) ? gv[e + 3] * rf * c4.w : 0.f;
      }
      if (row < 64) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int j = chalf * 32 + e;
          LT[i * LDL + j] = (j < i) ? x[e] : 0.f;
        }
      } else {
        uint8_t* Pt = sm + oP;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = x[8 * m + e];
          uint4 hi, lo;
          split8(y, hi, lo);
          *reinterpret_cast<uint4*>(Pt + sw128_offset(i, chalf * 32 + 8 * m)) = hi;
          *reinterpret_cast<uint4*>(Pt + 8192 + sw128_offset(i, chalf * 32 + 8 * m)) = lo;
        }
      }
    }
    __syncthreads();

    // ---------------- 4. T = (I + L)^-1 in place (fp32), 16x16 blocks
    {  // diagonal blocks: threads 0-63 each own one column, kept in registers
      const int j = tid & 15, I = (tid >> 4) & 3, r0 = 16 * I;
      float t[16];
#pragma unroll
      for (int l = 0; l < 16; ++l) t[l] = (l == j) ? 1.f : 0.f;
      if (tid < 64) {
#pragma unroll
        for (int i = 1; i < 16; ++i) {
          float s = 0.f;
#pragma unroll
          for (int l = 0; l < i; ++l) s += LT[(r0 + i) * LDL + r0 + l] * t[l];
          if (i > j) t[i] = -s;
        }
      }
      __syncthreads();
      if (tid < 64) {
#pragma unroll
        for (int i = 0; i < 16; ++i) LT[(r0 + i) * LDL + r0 + j] = t[i];
      }
    }
    __syncthreads();
    // level 1: T_10 = -T_11 (L_10 T_00) and T_32 = -T_33 (L_32 T_22); warp w < 4 owns
    // (block w >> 1, 8-column tile w & 1).  Level 2: rows 32-63 x cols 0-31,
    // T_C = -T_B (L_C T_A), one 16 x 8 output tile per warp.  (TF32 x3 products.)
    if (warp < 4) {
      const int blk = warp >> 1, nt = warp & 1;
      const int r0 = 32 * blk + 16, c0 = 32 * blk;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      tile_mm3<2>(d, LT + r0 * LDL + c0, LDL, LT + c0 * LDL + c0 + 8 * nt, LDL, lane);
      tile_store(XS + 16 * blk * LDX + 8 * nt, LDX, d, 1.f, lane);
    }
    __syncthreads();
    if (warp < 4) {
      const int blk = warp >> 1, nt = warp & 1;
      const int r0 = 32 * blk + 16, c0 = 32 * blk;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      tile_mm3<2>(d, LT + r0 * LDL + r0, LDL, XS + 16 * blk * LDX + 8 * nt, LDX, lane);
      tile_store(LT + r0 * LDL + c0 + 8 * nt, LDL, d, -1.f, lane);
    }
    __syncthreads();
    {
      const int mt = warp >> 2, nt = warp & 3;       // 2 x 4 tiles of 16 x 8
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      tile_mm3<4>(d, LT + (32 + 16 * mt) * LDL, LDL, LT + 8 * nt, LDL, lane);   // X = L_C T_A
      tile_store(XS + 16 * mt * LDX + 8 * nt, LDX, d, 1.f, lane);
    }
    __syncthreads();
    {
      const int mt = warp >> 2, nt = warp & 3;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      if (mt == 0)   // T_B is lower triangular: rows 32-47 only need columns 32-47
        tile_mm3<2>(d, LT + 32 * LDL + 32, LDL, XS + 8 * nt, LDX, lane);
      else
        tile_mm3<4>(d, LT + 48 * LDL + 32, LDL, XS + 8 * nt, LDX, lane);
      __syncthreads();   // every read of L_C (in X) is done; overwrite it with T_C
      tile_store(LT + (32 + 16 * mt) * LDL + 8 * nt, LDL, d, -1.f, lane);
    }
    __syncthreads();
    {  // T and Ts = T diag(ks) -> bf16 hi/lo, K-major [64 rows][64]
      const int i = tid >> 2, c0 = (tid & 3) * 16;
      uint8_t* Tt = sm + oT;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        float x[8], y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = c0 + 8 * m + e;
          const float tv = (j <= i) ? LT[i * LDL + j] : 0.f;
          x[e] = tv;
          y[e] = tv * vks[j];
        }
        uint4 hi, lo;
        split8(x, hi, lo);
        *reinterpret_cast<uint4*>(Tt + sw128_offset(i, c0 + 8 * m)) = hi;
        *reinterpret_cast<uint4*>(Tt + 8192 + sw128_offset(i, c0 + 8 * m)) = lo;
        split8(y, hi, lo);
        *reinterpret_cast<uint4*>(Tt + 16384 + sw128_offset(i, c0 + 8 * m)) = hi;
        *reinterpret_cast<uint4*>(Tt + 24576 + sw128_offset(i, c0 + 8 * m)) = lo;
      }
    }
    fence_proxy_async();
    __syncthreads();

    // ---------------- 5. MMA 2: W' = Ts K (N = 128),  U' = T V (N = 64); hi + lo along K
    if (!*abort_flag && !mbar_wait(&bar_v, c & 1, kWaitLimit)) *abort_flag = 1;
    if (tid == 0) {
      tc_fence_after();
      const uint32_t tb = smem_u32(sm + oT), kq = smem_u32(KQ), vt = smem_u32(sm + oV);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t dt = desc_sw128(tb + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
        const uint64_t dts = desc_sw128(tb + 16384 + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
        const uint64_t dk = desc_sw128(kq + (ks & 3) * 2048, 16384, 1024);
        const uint64_t dv = desc_sw128(vt + (ks & 3) * 2048, 8192, 1024);
        mma_bf16(tmem + cWp, dts, dk, ID_WP, ks > 0);
        mma_bf16(tmem + cE, dt, dv, ID_N64, ks > 0);
      }
      mma_commit(&bar_mma);
    }
    wait_mma();
    __syncthreads();
    if (tid == 0 && c + 1 < NC) issue_v(c + 1);   // V tile is free again

    // ---------------- 6. W' (M=64 layout: row 16 quad + lane, lanes < 16) -> bf16 hi/lo tiles
    {
      float w[64];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float t16[16];
        tmem_ld16(tmem + lane_off + cWp + chalf * 64 + 16 * m, t16);
#pragma unroll
        for (int e = 0; e < 16; ++e) w[16 * m + e] = t16[e];
      }
      tmem_ld_wait();
      if (lane < 16) {
        const int i = quad * 16 + lane;
        uint8_t* Wp = sm + oWp + chalf * 8192;
        uint8_t* Wl = sm + oE + chalf * 8192;   // lo term borrows the (free) E tiles
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = w[8 * m + e];
          uint4 hi, lo;
          split8(x, hi, lo);
          *reinterpret_cast<uint4*>(Wp + sw128_offset(i, 8 * m)) = hi;
          *reinterpret_cast<uint4*>(Wl + sw128_offset(i, 8 * m)) = lo;
        }
      }
    }
    fence_proxy_async();
    __syncthreads();

    // ---------------- 7. MMA 3: E = U' - (W'_hi S_hi + W'_hi S_lo + W'_lo S_hi),  QS = Q (S_hi + S_lo)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t kq = smem_u32(KQ), sb = smem_u32(sm + oS), wp = smem_u32(sm + oWp);
      const uint32_t wl = smem_u32(sm + oE);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t dsh = desc_sw128(sb + ks * 2048, 16384, 1024);
        const uint64_t dsl = desc_sw128(sb + 16384 + ks * 2048, 16384, 1024);
        const uint64_t dw = desc_sw128(wp + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
        const uint64_t dq = desc_sw128(kq + (ks >> 2) * 16384 + 8192 + (ks & 3) * 32, 16, 1024);
        const uint64_t dwl = desc_sw128(wl + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
        mma_bf16(tmem + cE, dw, dsh, ID_ENEG, true);
        mma_bf16(tmem + cE, dw, dsl, ID_ENEG, true);
        mma_bf16(tmem + cE, dwl, dsh, ID_ENEG, true);
        mma_bf16(tmem + cQS, dq, dsh, ID_N64, ks > 0);
        mma_bf16(tmem + cQS, dq, dsl, ID_N64, true);
      }
      mma_commit(&bar_mma);
    }
    wait_mma();

    // ---------------- 8. E and u.E -> bf16 hi/lo tiles (MN-major [64 tokens][64 columns])
    {
      float ev[32];
      ld32cols(tmem + lane_off + cE + chalf * 32, ev);
      tmem_ld_wait();
      if (lane < 16) {
        const int i = quad * 16 + lane;
        const float u = vu[i];
        uint8_t* Et = sm + oE;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float x[8], y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            x[e] = ev[8 * m + e];
            y[e] = u * x[e];
          }
          const uint32_t off = sw128_offset(i, chalf * 32 + 8 * m);
          uint4 hi, lo;
          split8(x, hi, lo);
          *reinterpret_cast<uint4*>(Et + off) = hi;
          *reinterpret_cast<uint4*>(Et + 8192 + off) = lo;
          split8(y, hi, lo);
          *reinterpret_cast<uint4*>(Et + 16384 + off) = hi;
          *reinterpret_cast<uint4*>(Et + 24576 + off) = lo;
        }
      }
    }
    fence_proxy_async();
    __syncthreads();

    // ---------------- 9. MMA 4: PE = P_hi E_hi + P_lo E_hi + P_hi E_lo ;  dS = W^T (uE_hi + uE_lo)
    if (tid == 0) {
      tc_fence_after();
      const uint32_t pb = smem_u32(sm + oP), eb = smem_u32(sm + oE);
      const uint32_t wb = kPgdn ? smem_u32(sm + oW) : smem_u32(KQ);
      const uint32_t wl = kPgdn ? 8192 : 16384;   // stride between the two 64-channel blocks
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t ph = desc_sw128(pb + ks * 32, 16, 1024);
        const uint64_t pl = desc_sw128(pb + 8192 + ks * 32, 16, 1024);
        const uint64_t eh = desc_sw128(eb + ks * 2048, 8192, 1024);
        const uint64_t el = desc_sw128(eb + 8192 + ks * 2048, 8192, 1024);
        const uint64_t uh = desc_sw128(eb + 16384 + ks * 2048, 8192, 1024);
        const uint64_t ul = desc_sw128(eb + 24576 + ks * 2048, 8192, 1024);
        const uint64_t dw = desc_sw128(wb + ks * 2048, wl, 1024);
        mma_bf16(tmem + cPE, ph, eh, ID_N64, ks > 0);
        mma_bf16(tmem + cPE, pl, eh, ID_N64, true);
        mma_bf16(tmem + cPE, ph, el, ID_N64, true);
        mma_bf16(tmem + cDS, dw, uh, ID_DS, ks > 0);
        mma_bf16(tmem + cDS, dw, ul, ID_DS, true);
      }
      mma_commit(&bar_mma);
    }
    wait_mma();

    // ---------------- 10. S <- gamma_C S + dS (M=128: row = lane) ; o = qs QS + PE -> global
    {
      const float gC = vmisc[0];
      float ds[32], qsv[32], pe[32];
      ld32cols(tmem + lane_off + cDS + chalf * 32, ds);
      ld32cols(tmem + lane_off + cQS + chalf * 32, qsv);
      ld32cols(tmem + lane_off + cPE + chalf * 32, pe);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) S[e] = gC * S[e] + ds[e];
      store_state_tiles();
      if (lane < 16) {
        const int i = quad * 16 + lane;
        if (i < Cc) {
          const float qs = vqs[i];
          __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out) +
                              (((long)b * a.T + t0 + i) * a.H + h) * a.dv + half * 64 + chalf * 32;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              x[e] = qs * qsv[8 * m + e] + pe[8 * m + e];
              if (a.check_finite) bad |= !finite_f(x[e]);
            }
            *reinterpret_cast<uint4*>(op + 8 * m) = pack8(x);
          }
        }
      }
    }
    fence_proxy_async();
    __syncthreads();
  }

  // ---- final state and aux
  if (!s_abort) {
    if (a.S) {
      const long base = ((long)bh * 128 + srow) * a.dv + half * 64 + chalf * 32;
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        *reinterpret_cast<float4*>(a.S + base + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        if (a.check_finite) bad |= !(finite_f(S[j]) && finite_f(S[j + 1]) && finite_f(S[j + 2]) && finite_f(S[j + 3]));
      }
    }
    if (kPgdn && a.aux && half == 0 && tid < 128) a.aux[(long)bh * 128 + tid] = carryA;
  } else {
    set_status(DR_ERR_TIMEOUT);
    // let any TMA still in flight land before the CTA exits
    if (tid == 0) {
      mbar_wait(&bar_kq[0], 0, kWaitLimit / 4);
      mbar_wait(&bar_v, 0, kWaitLimit / 4);
    }
  }
  if (bad) set_status(DR_ERR_NONFINITE);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

namespace {

// ------------------------------------------------------------------ host side

}  // namespace

bool chunk_tc_supported(int variant, int dtype, int dk, int dv, int chunk) {
  return (variant == DR_GDN || variant == DR_KLA || variant == DR_PGDN) && dtype == DR_BF16 &&
         dk == 128 && dv == 128 && chunk == 64;
}

cudaError_t launch_chunk_tc(const FwdArgs& a, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.B, a.T, a.H, 128) || !make_map(&mk, a.k, a.B, a.T, a.H, 128) ||
      !make_map(&mv, a.v, a.B, a.T, a.H, 128))
    return cudaErrorInvalidValue;
  const int grid = a.B * a.H * 2;
#define DR_TC(V_)                                                                          \
  if (a.variant == V_) {                                                                   \
    cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel<V_>,                              \
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,      \
                                         (int)kSmemBytes);                                 \
    if (e != cudaSuccess) return e;                                                        \
    chunk_tc_kernel<V_><<<grid, kTcThreads, kSmemBytes, st>>>(mq, mk, mv, a);              \
    return cudaGetLastError();                                                             \
  }
  DR_TC(DR_GDN) DR_TC(DR_KLA) DR_TC(DR_PGDN)
#undef DR_TC
  return cudaErrorInvalidValue;
}

}  // namespace dr
