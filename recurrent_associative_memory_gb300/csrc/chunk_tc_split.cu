// chunk_tc_split.cu — two-phase tcgen05 chunkwise forward: GDN and KLA (scalar
// decay, w = coefficient x raw key) and PGDN (explicit write keys), bf16
// q/k/v/out, dk = dv = 128, chunk 64; the carry also runs over Diagonal KDN
// records written by the CUDA-core prep of chunk_simt.cu.
//
// The chunk algebra is that of chunk_tc_ws.cu (KLA notes section 2.5, Eqs. (7)-(9),
// with the write matrix of the PDN notes section 2.6).  Everything in it that
// does not involve the state is independent across chunks (the chunkwise form
// exists for exactly that reason), so it is split off into a first kernel that
// runs on every SM at once, and the sequential carry over chunks becomes a
// second kernel whose critical path holds only the state-dependent products:
//
//   chunk_prep   one task per (b, h, chunk), 2 CTAs per SM, persistent.
//                Gram [K; Q] W^T on tcgen05; gates, norms and write coefficients;
//                L and P = lower((Q W^T) . e^{g_i - g_j}); T = (I + L)^-1 by
//                16x16 forward substitution and recursive doubling on bf16 hi/lo warp products;
//                W' = T diag(e^g c) K on tcgen05.  Writes one record per chunk
//                to the workspace: T, W' and P as bf16 hi/lo pairs, and the row
//                vectors e^g qn, e^{g_C - g} c, gamma_C (PGDN adds its write keys
//                and the statistic's chunk map).  (W' needs its lo term: with raw
//                GDN keys E = U' - W' S cancels heavily, and a single bf16 W'
//                costs ~1e-2 of the state.)
//   chunk_carry  one CTA per (b, h, 64-column half of dv): 8 state warps, an
//                issue lane, a PE lane and 4 output warps.  Per chunk:
//                U' = T V,  E = U' - W' S,  dS = K^T (u . E),
//                S <- gamma_C S + dS,  o = e^g qn . Q S + P E, with the bf16
//                hi/lo splits folded into few wide MMAs (see the carry section).
//                The record and the K, Q, V tiles arrive by bulk / tensor copies
//                issued as soon as the previous chunk's MMAs free each buffer.
//
// The records are intermediates of the method, not algorithmic traffic; the
// workspace is caller-owned (dr_chunk_fwd_workspace_bytes).  Every wait is
// bounded in wall-clock time; a timeout sets DR_ERR_TIMEOUT and the CTA drains
// its copies in flight before it frees TMEM and exits.
#include "dr_common.cuh"
#include "tc_common.cuh"

namespace dr {

namespace {

using namespace umma;
using namespace tc;

constexpr uint64_t kWait = 2000000000ull;   // 2 s per bounded wait
constexpr int LDL = 68;                     // fp32 L/T row stride
constexpr int LDX = 36;                     // fp32 scratch row stride

// ---- per-chunk record in the workspace (bytes); 128B-swizzled tile images
constexpr uint32_t rT = 0;          // T hi | T lo       (64 x 64 bf16 each)
constexpr uint32_t rWp = 16384;     // W'^T hi [128 dk][64 tok], then W'^T lo
constexpr uint32_t rP = 49152;      // P hi | P lo
constexpr uint32_t rVec = 65536;    // fp32 [0,64) e^g qn ; [64,128) e^{g_C-g} c ; [128] gamma_C ;
                                    //      [192,256) e^g cr (GDN/KLA)
constexpr uint32_t kRec = 66560;
// PGDN records add the explicit write keys and the statistic's chunk map
constexpr uint32_t rW = 66560;      // W hi [64 tok][128] (2 k-blocks), then W lo      32 KB
constexpr uint32_t rAux = 99328;    // fp32 [0] prod alphaP, [1,129) chunk offset of A,
                                    //      [256,384) A at the chunk start
constexpr uint32_t kRecP = 101376;

template <int VARIANT>
__host__ __device__ constexpr uint32_t rec_bytes() { return VARIANT == DR_PGDN ? kRecP : kRec; }

// ================================================================= chunk_prep
constexpr int kPrepThreads = 9 * 32;        // warps 0-7 prep, warp 8 issue
constexpr uint32_t pKQ = 0;                 // 2 stages x [K kb0 | Q kb0 | K kb1 | Q kb1], 32 KB each
constexpr uint32_t pT = 65536;              // T hi | T lo | Ts hi | Ts lo (L/T fp32 aliases it)
constexpr uint32_t pVec = pT + 32768;       // vectors, 4 KB
constexpr uint32_t kPrepSmem = pVec + 4096 + 1024;
constexpr uint32_t tG0 = 0;                 // 2 Gram slots, M=128 x 64
constexpr uint32_t tPWt = 128;              // W'^T = K^T [Ts_hi ; Ts_lo]^T, M=128 x 128 (halves added)
constexpr uint32_t kPrepTmem = 256;

constexpr uint32_t I_GRAM = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t I_WT = idesc_bf16(128, 128, 1, 0);    // A = K (MN-major), B = [Ts_hi ; Ts_lo] (K-major)
constexpr uint32_t I_N64 = idesc_bf16(64, 64, 0, 1);
constexpr uint32_t I_DS = idesc_bf16(128, 64, 1, 1);
// N = 128 over a [hi | lo] pair of B tiles one 64-column group apart: one MMA
// reads A once for both halves of the split operand (the two products land in
// columns [0, 64) and [64, 128) and are added on readout)
constexpr uint32_t I_DS2 = idesc_bf16(128, 128, 1, 1);

enum { P_KQ0, P_KQ1, P_G0, P_G1, P_W, P_GFREE0, P_GFREE1, P_TREADY, P_WFREE, P_WREADY, P_PREAD, P_COUNT };

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int VARIANT>
__global__ void __launch_bounds__(kPrepThreads, 2)
    chunk_prep_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      FwdArgs a, uint8_t* __restrict__ ws) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bars[P_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int s_abort;
  __shared__ volatile int s_ok;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NC = (a.T + 63) / 64;
  const int ntask = a.B * a.H * NC;
  // tasks of this CTA: blockIdx.x + k gridDim.x
  auto task_of = [&](int k) { return blockIdx.x + k * gridDim.x; };
  const int nmine = (blockIdx.x < ntask) ? (ntask - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  float* vC = reinterpret_cast<float*>(sm + pVec);   // [4 I][64 j] c_j e^{g_m(I) - g_j}
  float* vg = vC + 256;     // cumulative log-decay
  float* va = vg + 64;      // coefficient of the raw key row in w
  float* vcr = va + 64;     // key normalisation
  float* vqn = vcr + 64;    // query normalisation
  float* vks = vqn + 64;    // e^{g_j} c_j
  float* vkk = vks + 64;
  float* vqq = vkk + 64;
  float* vla = vqq + 64;
  float* veta = vla + 64;
  float* vaP = veta + 64;   // PGDN statistic decay / gain per token
  float* vbP = vaP + 64;
  constexpr bool kPgdn = (VARIANT == DR_PGDN);
  constexpr uint32_t kRecV = rec_bytes<VARIANT>();
  const float mu_h_unused = 0.f;
  (void)mu_h_unused;
  float* LT = reinterpret_cast<float*>(sm + pT);
  float* XS = LT + 64 * LDL;

  if (tid == 0) {
    for (int i = 0; i < P_COUNT; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    s_abort = 0;
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, kPrepTmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp < 8) {
    // ===================================================================== prep warps
    const int ptid = tid, pwarp = warp;
    const int quad = warp & 3, pchalf = pwarp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const bool leader = (ptid == 0);
    auto group_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (leader) {
        bool ok = !s_abort && mbar_wait(bar, parity, kWait);
        if (!ok) s_abort = 1;
        s_ok = ok ? 1 : 0;
      }
      named_bar(1, 256);
      const bool ok = s_ok != 0;
      named_bar(1, 256);
      return ok;
    };

    float nla = 0.f, neta = 0.f, naP = 1.f, nbP = 0.f;   // gates of the next task (ptid < 64 = token)
    auto prefetch_gates = [&](int k) {
      const int t = task_of(k), bh = t / NC, c = t % NC;
      const int i = ptid, tok = c * 64 + i;
      if (i < 64 && tok < a.T) {
        const long ti = ((long)(bh / a.H) * a.T + tok) * a.H + (bh % a.H);
        nla = a.log_alpha[ti];
        neta = a.eta[ti];
        if (kPgdn) {
          naP = a.alphaP[ti];
          nbP = a.betaP[ti];
        }
      } else {
        nla = 0.f;
        neta = 0.f;
        naP = 1.f;
        nbP = 0.f;
      }
    };
    if (nmine > 0) prefetch_gates(0);

    for (int k = 0; k < nmine; ++k) {
      const int t = task_of(k);
      uint8_t* rec = ws + (size_t)t * kRecV;   // tasks are numbered (b h) major, chunk minor
      const int st = k & 1;
      uint8_t* KQ = sm + pKQ + st * 32768;

      // ---- gates: decay, norms, write coefficients, the carry's row vectors
      if (!group_wait(&bars[P_KQ0 + st], (k >> 1) & 1)) break;
      if (ptid < 64) {
        vla[ptid] = nla;
        veta[ptid] = neta;
        if (kPgdn) {
          vaP[ptid] = naP;
          vbP[ptid] = nbP;
        }
      }
      if (k + 1 < nmine) prefetch_gates(k + 1);
      {
        const int i = ptid >> 2, part = ptid & 3, kb = part >> 1, c0 = (part & 1) * 32;
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
      named_bar(1, 256);
      if (pwarp == 0) {
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
      named_bar(1, 256);
      if (ptid < 64) {
        const int i = ptid;
        const float gi = vg[i], gC = vg[63];
        const float kk = vkk[i], qq = vqq[i];
        const float cr = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
        const float qn = a.q_l2norm ? 1.f / fmaxf(sqrtf(qq), 1e-30f) : 1.f;
        float beta = veta[i];
        if (VARIANT == DR_KLA) beta = beta / (kk * cr * cr + a.eps);
        const float coef = kPgdn ? 1.f : beta * cr;   // PGDN: w is explicit (below)
        va[i] = coef;
        vcr[i] = cr;
        vqn[i] = qn;
        const float eg = __expf(gi);
        vks[i] = eg * cr;
        float* rv = reinterpret_cast<float*>(rec + rVec);
        rv[i] = eg * qn;
        rv[64 + i] = __expf(gC - gi) * coef;
        rv[192 + i] = eg * cr;   // e^g cr: the backward's (Gamma.K^) rows
        if (i == 0) rv[128] = __expf(gC);
      }
      if (kPgdn && leader) bulk_wait_read<0>();   // the previous W'^T copy has left the T region
      named_bar(1, 256);
      if (kPgdn) {
        // statistic scan from the chunk-start value (prefix of the chunk maps), the
        // bounded map B(A) and the write keys w = eta B(A) . k^ (PDN notes Eq. (9)),
        // as bf16 hi/lo [64 tokens][128] tiles in the T region: the Gram's B operand
        // and the carry's dS operand (one bulk copy into the record)
        {   // two threads per channel: tokens 0-31 and 32-63 (the second runs the
            // statistic's recurrence over the first half to its own start)
          const int ch = ptid & 127, hf = ptid >> 7, kb = ch >> 6, col = ch & 63;
          const float mu_h = a.mu[(t / NC) % a.H];
          float A = reinterpret_cast<const float*>(rec + rAux)[256 + ch];
          uint8_t* Wt = sm + pT;
          if (hf) {
#pragma unroll 8
            for (int i = 0; i < 32; ++i) {
              const float kx = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                                   KQ + kb * 16384 + sw128_offset(i, col))) * vcr[i];
              A = vaP[i] * A + vbP[i] * kx * kx;
            }
          }
          for (int i0 = 32 * hf; i0 < 32 * hf + 32; i0 += 8) {
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
              const __nv_bfloat16 wh = __float2bfloat16_rn(w);
              const __nv_bfloat16 wl = __float2bfloat16_rn(w - __bfloat162float(wh));
              const uint32_t off = kb * 8192 + sw128_offset(i0 + e, col);
              *reinterpret_cast<__nv_bfloat16*>(Wt + off) = wh;
              *reinterpret_cast<__nv_bfloat16*>(Wt + 16384 + off) = wl;
            }
          }
        }
        fence_proxy_async();
        named_bar(1, 256);
        if (leader) {
          bulk_store(rec + rW, sm + pT, 32768);
          bulk_commit();
          mbar_arrive(&bars[P_WREADY]);
        }
      }

      // ---- Gram readout -> L (fp32, smem) and P (bf16 hi/lo, staged in the Q half of
      //      the K/Q stage, which the Gram was the last to read, then one bulk copy).
      //      Each 16-row block I takes its sub-chunk's middle token m(I) as the
      //      reference: L_ij = G_ij [rs_i e^{g_i - g_m(I)}] [c_j e^{g_m(I) - g_j}] for
      //      j <= i, where the column factor is <= 1 below block I and bounded by the
      //      decay over 8 tokens inside it; above the diagonal the select drops it.
      {
        const int I = ptid >> 6, j = ptid & 63;
        vC[ptid] = va[j] * __expf(vg[16 * I + 7] - vg[j]);
      }
      if (leader) bulk_wait_read<0>();   // the previous task's W' copy has left the T region
      if (!group_wait(&bars[P_G0 + st], (k >> 1) & 1)) break;
      tc_fence_after();
      {
        const int row = quad * 32 + lane;
        const int i = row & 63, I = i >> 4;
        float gv[32];
        ld32cols(tmem + lane_off + tG0 + st * 64 + pchalf * 32, gv);
        tmem_ld_wait();
        const float rf = ((row < 64) ? vcr[i] : vqn[i]) * __expf(vg[i] - vg[16 * I + 7]);
        const float* C = vC + I * 64 + pchalf * 32;
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 c4 = *reinterpret_cast<const float4*>(C + e);
          const int j = pchalf * 32 + e;
          x[e] = (j <= i) ? gv[e] * rf * c4.x : 0.f;
          x[e + 1] = (j + 1 <= i) ? gv[e + 1] * rf * c4.y : 0.f;
          x[e + 2] = (j + 2 <= i) ? gv[e + 2] * rf * c4.z : 0.f;
          x[e + 3] = (j + 3 <= i) ? gv[e + 3] * rf * c4.w : 0.f;
        }
        if (row < 64) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const int j = pchalf * 32 + e;
            *reinterpret_cast<float4*>(LT + i * LDL + j) =
                make_float4(j < i ? x[e] : 0.f, j + 1 < i ? x[e + 1] : 0.f,
                            j + 2 < i ? x[e + 2] : 0.f, j + 3 < i ? x[e + 3] : 0.f);
          }
        } else {
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = x[8 * m + e];
            uint4 hi, lo;
            split8(y, hi, lo);
            *reinterpret_cast<uint4*>(KQ + 8192 + sw128_offset(i, pchalf * 32 + 8 * m)) = hi;
            *reinterpret_cast<uint4*>(KQ + 24576 + sw128_offset(i, pchalf * 32 + 8 * m)) = lo;
          }
        }
      }
      tc_fence_before();
      fence_proxy_async();
      named_bar(1, 256);
      if (leader) {
        mbar_arrive(&bars[P_GFREE0 + st]);
        bulk_store(rec + rP, KQ + 8192, 8192);
        bulk_store(rec + rP + 8192, KQ + 24576, 8192);
        bulk_commit();
      }
      // ---- T = (I + L)^-1 in place: diagonal 16x16 blocks (threads 0-63, one column each)
      {
        const int j = ptid & 15, I = (ptid >> 4) & 3, r0 = 16 * I;
        float tt[16];
#pragma unroll
        for (int l = 0; l < 16; ++l) tt[l] = (l == j) ? 1.f : 0.f;
        if (ptid < 64) {
#pragma unroll
          for (int i = 1; i < 16; ++i) {
            float s = 0.f;
#pragma unroll
            for (int l = 0; l < i; ++l) s += LT[(r0 + i) * LDL + r0 + l] * tt[l];
            if (i > j) tt[i] = -s;
          }
        }
        named_bar(1, 256);
        if (ptid < 64) {
#pragma unroll
          for (int i = 0; i < 16; ++i) LT[(r0 + i) * LDL + r0 + j] = tt[i];
        }
      }
      named_bar(1, 256);
      // level 1: T_10, T_32 ; level 2: the 32 x 32 lower-left block (bf16 hi/lo mma.sync)
      if (pwarp < 4) {
        const int blk = pwarp >> 1, nt = pwarp & 1;
        const int r0 = 32 * blk + 16, c0 = 32 * blk;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mm3b<2>(d, LT + r0 * LDL + c0, LDL, LT + c0 * LDL + c0 + 8 * nt, LDL, lane);
        tile_store(XS + 16 * blk * LDX + 8 * nt, LDX, d, 1.f, lane);
      }
      named_bar(1, 256);
      if (pwarp < 4) {
        const int blk = pwarp >> 1, nt = pwarp & 1;
        const int r0 = 32 * blk + 16, c0 = 32 * blk;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mm3b<2>(d, LT + r0 * LDL + r0, LDL, XS + 16 * blk * LDX + 8 * nt, LDX, lane);
        tile_store(LT + r0 * LDL + c0 + 8 * nt, LDL, d, -1.f, lane);
      }
      named_bar(1, 256);
      {
        const int mt = pwarp >> 2, nt = pwarp & 3;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mm3b<4>(d, LT + (32 + 16 * mt) * LDL, LDL, LT + 8 * nt, LDL, lane);
        tile_store(XS + 16 * mt * LDX + 8 * nt, LDX, d, 1.f, lane);
      }
      named_bar(1, 256);
      {
        const int mt = pwarp >> 2, nt = pwarp & 3;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        if (mt == 0)
          tile_mm3b<2>(d, LT + 32 * LDL + 32, LDL, XS + 8 * nt, LDX, lane);
        else
          tile_mm3b<4>(d, LT + 48 * LDL + 32, LDL, XS + 8 * nt, LDX, lane);
        tile_store(LT + (32 + 16 * mt) * LDL + 8 * nt, LDL, d, -1.f, lane);
      }
      named_bar(1, 256);
      // ---- T (record) and Ts = T diag(ks) (smem, for W'); the tiles alias L/T, so read first
      {
        const int i = ptid >> 2, c0 = (ptid & 3) * 16;
        float tv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = c0 + e;
          tv[e] = (j <= i) ? LT[i * LDL + j] : 0.f;
        }
        named_bar(1, 256);
        uint8_t* Tt = sm + pT;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          float x[8], y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            x[e] = tv[8 * m + e];
            y[e] = x[e] * vks[c0 + 8 * m + e];
          }
          const uint32_t off = sw128_offset(i, c0 + 8 * m);
          uint4 hi, lo;
          split8(x, hi, lo);
          *reinterpret_cast<uint4*>(Tt + off) = hi;
          *reinterpret_cast<uint4*>(Tt + 8192 + off) = lo;
          split8(y, hi, lo);
          *reinterpret_cast<uint4*>(Tt + 16384 + off) = hi;
          *reinterpret_cast<uint4*>(Tt + 24576 + off) = lo;
        }
      }
      fence_proxy_async();
      named_bar(1, 256);
      if (leader) {
        bulk_store(rec + rT, sm + pT, 16384);
        bulk_commit();
        mbar_arrive(&bars[P_TREADY]);
      }
      // ---- W'^T readout (row = dk index = TMEM lane, 32 tokens per thread), staged
      //      over T / Ts (both read by now), then one bulk copy into the record.  The
      //      P copy has left the K/Q stage too, so the stage may be reloaded (PREAD).
      if (leader) bulk_wait_read<0>();
      if (!group_wait(&bars[P_W], k & 1)) break;
      if (leader) mbar_arrive(&bars[P_PREAD]);
      tc_fence_after();
      {
        const int r = quad * 32 + lane;
        uint8_t* Wg = sm + pT;
        float w[32];
        {
          float t16[16], u16[16];
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            tmem_ld16(tmem + lane_off + tPWt + pchalf * 32 + 16 * part, t16);
            tmem_ld16(tmem + lane_off + tPWt + 64 + pchalf * 32 + 16 * part, u16);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) w[16 * part + e] = t16[e] + u16[e];
          }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = w[8 * m + e];
          uint4 hi, lo;
          split8(x, hi, lo);
          *reinterpret_cast<uint4*>(Wg + sw128_offset(r, pchalf * 32 + 8 * m)) = hi;
          *reinterpret_cast<uint4*>(Wg + 16384 + sw128_offset(r, pchalf * 32 + 8 * m)) = lo;
        }
      }
      tc_fence_before();
      fence_proxy_async();
      named_bar(1, 256);
      if (leader) {
        mbar_arrive(&bars[P_WFREE]);
        bulk_store(rec + rWp, sm + pT, 32768);
        bulk_commit();
      }
    }
    if (leader) bulk_wait_all();   // every record byte is in global memory before exit
  } else if (lane == 0) {
    // ===================================================================== issue lane
    auto wait = [&](int id, uint32_t parity) -> bool {
      if (s_abort) return false;
      if (!mbar_wait(&bars[id], parity, kWait)) {
        s_abort = 1;
        return false;
      }
      return true;
    };
    int kq_issued = 0;   // KQ loads issued so far (task k uses stage k & 1)
    auto issue_kq = [&](int k) {
      const int t = task_of(k), bh = t / NC, c = t % NC;
      const int b = bh / a.H, h = bh % a.H, st = k & 1;
      uint8_t* base = sm + pKQ + st * 32768;
      mbar_expect_tx(&bars[P_KQ0 + st], 32768);
      tma_load_4d(base, &tmK, &bars[P_KQ0 + st], 0, h, c * 64, b);
      tma_load_4d(base + 16384, &tmK, &bars[P_KQ0 + st], 64, h, c * 64, b);
      tma_load_4d(base + 8192, &tmQ, &bars[P_KQ0 + st], 0, h, c * 64, b);
      tma_load_4d(base + 16384 + 8192, &tmQ, &bars[P_KQ0 + st], 64, h, c * 64, b);
      kq_issued = k + 1;
    };
    // Gram [K; Q] W^T into slot k & 1: W = K itself (GDN/KLA, A and B share one
    // descriptor), or the PGDN write keys (bf16 hi/lo) the prep warps left in the T region
    auto gram = [&](int k) {
      const uint32_t kq = smem_u32(sm + pKQ + (k & 1) * 32768);
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t d = desc_sw128(kq + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
        if (kPgdn) {
          const uint32_t wb = smem_u32(sm + pT) + (ks >> 2) * 8192 + (ks & 3) * 32;
          mma_bf16(tmem + tG0 + (k & 1) * 64, d, desc_sw128(wb, 16, 1024), I_GRAM, ks > 0);
          mma_bf16(tmem + tG0 + (k & 1) * 64, d, desc_sw128(wb + 16384, 16, 1024), I_GRAM, true);
        } else {
          mma_bf16(tmem + tG0 + (k & 1) * 64, d, d, I_GRAM, ks > 0);
        }
      }
      mma_commit(&bars[P_G0 + (k & 1)]);
    };
    bool ok = true;
    if (nmine > 0) issue_kq(0);
    if (nmine > 1) issue_kq(1);
    if (!kPgdn && nmine > 0 && (ok = wait(P_KQ0, 0))) gram(0);
    int w_done = 0;   // W' MMAs committed
    for (int k = 0; ok && k < nmine; ++k) {
      const int st = k & 1;
      if (kPgdn) {
        // PGDN: the Gram needs this task's write keys, so it follows WREADY(k)
        // (the slot's previous readout, task k-2, finished before WREADY(k-1))
        if (!(ok = wait(P_WREADY, k & 1) && wait(P_KQ0 + st, (k >> 1) & 1))) break;
        gram(k);
      } else if (k + 1 < nmine) {
        // Gram of the next task into the other slot once its readout (task k-1) is done
        if (!(ok = wait(P_KQ0 + (st ^ 1), ((k + 1) >> 1) & 1))) break;
        if (k >= 1 && !(ok = wait(P_GFREE0 + (st ^ 1), ((k - 1) >> 1) & 1))) break;
        gram(k + 1);
      }
      // W'(k) = Ts K once the tiles are ready and W'(k-1) has been read out
      if (!(ok = wait(P_TREADY, k & 1))) break;
      if (k >= 1 && !(ok = wait(P_WFREE, (k - 1) & 1))) break;
      tc_fence_after();
      {
        const uint32_t tb = smem_u32(sm + pT), kq = smem_u32(sm + pKQ + st * 32768);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {   // B = [Ts_hi ; Ts_lo] stacked along N
          const uint64_t dts = desc_sw128(tb + 16384 + ks * 32, 16, 1024);
          const uint64_t dk = desc_sw128(kq + ks * 2048, 16384, 1024);
          mma_bf16(tmem + tPWt, dk, dts, I_WT, ks > 0);
        }
        mma_commit(&bars[P_W]);
        w_done = k + 1;
      }
      // stage st is free once W'(k) (its last MMA reader) is done and the P copy
      // out of its Q half has been read (PREAD(k), arrived after the prep warps
      // have seen W'(k) complete, so it cannot run a phase ahead of this wait)
      if (k + 2 < nmine) {
        if (!(ok = wait(P_W, k & 1) && wait(P_PREAD, k & 1))) break;
        issue_kq(k + 2);
      }
    }
    if (!ok) set_status(DR_ERR_TIMEOUT);
    // drain: the last W' MMA and every KQ load issued
    if (w_done > 0) mbar_wait(&bars[P_W], (w_done - 1) & 1, kWait / 4);
    for (int k = (kq_issued > 2 ? kq_issued - 2 : 0); k < kq_issued; ++k)
      mbar_wait(&bars[P_KQ0 + (k & 1)], (k >> 1) & 1, kWait / 4);
  }

  if (warp == 8) __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (s_abort && tid == 0) set_status(DR_ERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tmem, kPrepTmem);
}

// ================================================================= pgdn_stat
// The PGDN key statistic A_t = alphaP_t A_{t-1} + betaP_t (k^_t . k^_t) (PDN notes
// Eq. (9), first line) is linear in A, so over one chunk it is the affine map
// A -> a_c A + b_c with a_c = prod alphaP and b_c the chunk's own accumulation
// from 0 (the chunked form of the PDN notes section 2.6).
//   pgdn_map_kernel   two warps per (b, h, chunk), four chunks per block: the
//                     chunk's key tile arrives by TMA (two 64-channel boxes, 16 KB,
//                     zero past the end), then a thread per token forms the key
//                     norm and a thread per channel pair runs the affine map over
//                     the chunk's 64 tokens out of shared memory.
//   pgdn_scan_kernel  one thread per (b, h, channel) composes the maps in chunk
//                     order and leaves A at every chunk start in the chunk's
//                     record (and the final A).
constexpr int kMapTasks = 4;                            // chunk tasks per block
constexpr uint32_t kMapSmem = kMapTasks * 16384 + 1024; // key tiles (+ 1 KB alignment)

__global__ void __launch_bounds__(kMapTasks * 64) pgdn_map_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                   FwdArgs a, uint8_t* __restrict__ ws) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bars[kMapTasks];
  __shared__ float s_cr[kMapTasks][64], s_aP[kMapTasks][64], s_bP[kMapTasks][64];
  const int tid = threadIdx.x, slot = tid >> 6, sub = tid & 63;
  const int NC = (a.T + 63) / 64;
  const long ntask = (long)a.B * a.H * NC;
  const long task = (long)blockIdx.x * kMapTasks + slot;
  const bool live = task < ntask;
  const int bh = live ? (int)(task / NC) : 0, c = live ? (int)(task % NC) : 0;
  const int b = bh / a.H, h = bh % a.H;
  uint8_t* tile = sm + slot * 16384;   // [64 tok][64 ch] bf16, channels 0-63 | 64-127
  if (tid == 0) {
    for (int q = 0; q < kMapTasks; ++q) mbar_init(&bars[q], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (live && sub == 0) {
    mbar_expect_tx(&bars[slot], 16384);
    tma_load_4d(tile, &tmK, &bars[slot], 0, h, c * 64, b);
    tma_load_4d(tile + 8192, &tmK, &bars[slot], 64, h, c * 64, b);
  }
  {   // the statistic's gates of token sub, under the copy (identity past the end)
    const int tok = c * 64 + sub;
    const bool real = live && tok < a.T;
    const long ti = ((long)b * a.T + tok) * a.H + h;
    s_aP[slot][sub] = real ? a.alphaP[ti] : 1.f;
    s_bP[slot][sub] = real ? a.betaP[ti] : 0.f;
  }
  bool ok = true;
  if (live) {
    ok = mbar_wait(&bars[slot], 0, kWait);
    if (!ok) {   // report, and let the copy land before the block's memory is released
      set_status(DR_ERR_TIMEOUT);
      mbar_wait(&bars[slot], 0, kWait / 4);
    }
  }
  if (live && ok) {   // key norm of token sub
    float kk = 0.f;
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        float f[8];
        unpack8(*reinterpret_cast<const uint4*>(tile + kb * 8192 + sw128_offset(sub, 8 * m)), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) kk += f[e] * f[e];
      }
    s_cr[slot][sub] = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
  }
  __syncthreads();
  if (!live || !ok) return;
  // channels 2 sub, 2 sub + 1: A -> prod(alphaP) A + acc over the chunk (acc from 0)
  const int kb = sub >> 5, col = 2 * (sub & 31);
  float acc0 = 0.f, acc1 = 0.f, prod = 1.f;
#pragma unroll 8
  for (int i = 0; i < 64; ++i) {
    const __nv_bfloat162 k2 = *reinterpret_cast<const __nv_bfloat162*>(tile + kb * 8192 + sw128_offset(i, col));
    const float cr = s_cr[slot][i], aP = s_aP[slot][i], bP = s_bP[slot][i];
    const float k0 = __low2float(k2) * cr, k1 = __high2float(k2) * cr;
    acc0 = aP * acc0 + bP * k0 * k0;
    acc1 = aP * acc1 + bP * k1 * k1;
    prod *= aP;
  }
  float* aux = reinterpret_cast<float*>(ws + (size_t)task * kRecP + rAux);
  if (sub == 0) aux[0] = prod;
  aux[1 + 64 * kb + col] = acc0;
  aux[2 + 64 * kb + col] = acc1;
}

__global__ void __launch_bounds__(128) pgdn_scan_kernel(FwdArgs a, uint8_t* __restrict__ ws) {
  const int bh = blockIdx.x, ch = threadIdx.x;
  const int NC = (a.T + 63) / 64;
  uint8_t* recs = ws + (size_t)bh * NC * kRecP;
  float A = a.aux0 ? a.aux0[(long)bh * 128 + ch] : 0.f;
  constexpr int D = 8;   // maps loaded ahead of their use
  float am[D], bm[D];
#pragma unroll
  for (int d = 0; d < D; ++d) {
    const float* m = reinterpret_cast<const float*>(recs + (size_t)min(d, NC - 1) * kRecP + rAux);
    am[d] = m[0];
    bm[d] = m[1 + ch];
  }
  for (int c0 = 0; c0 < NC; c0 += D) {
    float an[D], bn[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {   // next block of maps, in flight during this block
      const float* m = reinterpret_cast<const float*>(recs + (size_t)min(c0 + D + d, NC - 1) * kRecP + rAux);
      an[d] = m[0];
      bn[d] = m[1 + ch];
    }
#pragma unroll
    for (int d = 0; d < D; ++d) {
      if (c0 + d < NC) {
        reinterpret_cast<float*>(recs + (size_t)(c0 + d) * kRecP + rAux)[256 + ch] = A;
        A = am[d] * A + bm[d];
      }
    }
#pragma unroll
    for (int d = 0; d < D; ++d) {
      am[d] = an[d];
      bm[d] = bn[d];
    }
  }
  if (a.aux) a.aux[(long)bh * 128 + ch] = A;
}

// ================================================================= chunk_carry
// Roles (14 warps):
//   state  warps 0-7   thread = one TMEM lane x 32 of the CTA's 64 columns:
//                      E readout -> E, u.E tiles; S <- gamma_C S + dS.  Its
//                      leader issues the two MMAs of the carry's critical path
//                      itself (E(c), dS(c)), so no hand-off sits on that path.
//   issue  warp 8      copies (T, V, W', Q) and the off-path MMAs QS = Q S and
//                      U'(c+1) = T V.
//   PE     warp 13     the off-path MMA PE = P E (a second issuing thread: one
//                      thread issues about one MMA per 60-70 cycles, so U' and
//                      PE, both due while the state is updated, come from two),
//                      and the P copies, which wait on PE (the state leader
//                      refills K the moment dS has read it).
//   output warps 9-12  o = e^g qn . QS + PE for every row of the chunk.
// MMA shapes.  One issuing thread sustains about one tcgen05.mma per 55-65
// cycles, and the tensor pipe takes an M=128 x N=128 step in about 1.7x the
// time of an M=64 x N=64 one, so the bf16 hi/lo splits are folded into few,
// wide MMAs instead of one MMA per pair of parts:
//   U', E   A = [T_hi ; T_lo], [W'_hi ; W'_lo] stacked along M (TMEM lanes
//           64-127 hold the lo-part rows), B = [S_hi | S_lo] along N; the E
//           readout adds the four quadrants (lanes i and 64 + i, columns j and
//           64 + j), the lo x lo product included.
//   dS      B = [uE_hi | uE_lo] (N = 128), the two column halves added.
//   QS, PE  (M = 64) B = [S_hi | S_lo] and [E_hi | E_lo] (N = 128).
// MODE 0 (GDN, KLA): dS = K^T (u.E) with K by TMA.  MODE 1 (PGDN): dS from the
// record's write keys.  MODE 2 (Diagonal KDN): Q S and dS take the record's
// (Gamma.Q) and (exp(g_C - g_j).w_j) as bf16 hi/lo operands (per-channel decay
// is folded into them), u = 1, and gamma_C is per state row.
// The row vectors (e^g qn, u, gamma_C) are read from the record in global
// memory, one chunk ahead, so no shared buffer of them needs recycling.
constexpr int kCarryThreads = 14 * 32;
constexpr uint32_t cT = 0;                  // T hi | T lo              16 KB
constexpr uint32_t cV = 16384;              // V [64 tok][64 col]       8 KB
constexpr uint32_t cW = 24576;              // 2 slots x W' [hi kb0|kb1, lo kb0|kb1]   64 KB
constexpr uint32_t cQ = 90112;              // Q kb0 | kb1 (16 KB); KDN: Q~ hi | lo (32 KB)
// then the dS operand + P: GDN/KLA [K kb0 | K kb1 | P hi | P lo] 32 KB; PGDN / KDN
// [W hi | W lo | P hi | P lo] 48 KB; S hi | S lo [128][64] (32 KB); E hi | E lo |
// uE hi | uE lo (32 KB; KDN, where u = 1: E hi | E lo, 16 KB).  The E readout
// exchanges its lo-part rows through the W' slot that E has just consumed.
// KDN record (bf16 images; rT, rWp, rP, rVec as above, gamma_C per channel at
// float 128 of rVec, ones elsewhere): (Gamma.Q) and Wbar as [64 tok][128] hi | lo
constexpr uint32_t rQk = 66560;
constexpr uint32_t rWk = 99328;
constexpr uint32_t kRecKdn = 135168;        // also holds the variance chunk map and p0
constexpr int kXs = 68;                     // fp32 row stride of the E exchange buffer
template <int MODE>
struct CarryMap {
  static constexpr uint32_t kQ = MODE == 2 ? 32768 : 16384;
  static constexpr uint32_t KP = cQ + kQ;
  static constexpr uint32_t kKP = MODE == 0 ? 32768 : 49152;
  static constexpr uint32_t P = MODE == 0 ? 16384 : 32768;     // P inside the K/P buffer
  static constexpr uint32_t S = KP + kKP;
  static constexpr uint32_t E = S + 32768;
  static constexpr uint32_t bytes = E + (MODE == 2 ? 16384 : 32768) + 1024;
  static constexpr uint32_t rec = MODE == 0 ? kRec : (MODE == 1 ? kRecP : kRecKdn);
  static constexpr uint32_t rW_ = MODE == 1 ? rW : rWk;        // record dS operand
};
constexpr uint32_t tE = 0;                  // 2 slots M=128 x 128: U' then E, in four quadrants
constexpr uint32_t tO = 256;                // M=64 x 128: Q S_hi | Q S_lo, then (once read)
                                            //   (P_hi + P_lo) E_hi | P_hi E_lo
constexpr uint32_t tDS = 384;               // M=128 x 128: K^T uE_hi (+ W_lo^T uE_hi) | K^T uE_lo
constexpr uint32_t kCarryTmem = 512;
constexpr uint32_t I_U2 = idesc_bf16(128, 64, 0, 1);         // [T_hi ; T_lo] V
constexpr uint32_t I_E1 = idesc_bf16(128, 64, 1, 1, 1);      // -[W'_hi ; W'_lo] S_hi (or S_lo)
constexpr uint32_t I_E2 = idesc_bf16(128, 128, 1, 1, 1);     // -[W'_hi ; W'_lo] [S_hi | S_lo]
constexpr uint32_t I_Q2 = idesc_bf16(64, 128, 0, 1);         // Q [S_hi | S_lo], P_hi [E_hi | E_lo]

enum {
  C_TV, C_W0, C_W1, C_Q, C_K, C_P,          // copies landed
  C_M2, C_E, C_QS, C_DS, C_PE,              // MMAs complete
  C_SREADY, C_EREADY, C_QSFREE, C_OUTDONE,  // group hand-offs to the issuing lanes
  C_COUNT
};

// SAVE: the backward's rerun, which also stores every chunk-start state and E (a
// separate instantiation, so the forward's code carries none of it)
template <int MODE, bool SAVE>
__global__ void __launch_bounds__(kCarryThreads, 1)
    chunk_carry_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, FwdArgs a,
                       const uint8_t* __restrict__ ws) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bars[C_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NCt = (a.T + 63) / 64;
  // This CTA's work: a row (b, h), a 64-column half of the state, and a run of
  // chunks c0 .. c0 + NC - 1 (the whole row unless the carry is segmented).  The
  // loops below count chunks locally (barrier phases, buffer slots); records,
  // tokens and saved states are addressed by the absolute chunk c0 + c.
  int half, bh, c0 = 0, NC = NCt;
  int s0mode = 0;                  // 0: init_state (or zero), 1: zero, 2: identity, 3: seg start
  bool out_on = a.out != nullptr, vzero = false, fin_out = true;
  float* sfin = nullptr;           // this row's final state [dk][dv], or null
  const float* s0p = nullptr;      // this row's start state [dk][dv] (s0mode 0 / 3)
  auto segmat = [&](int row, int g, int which) -> float* {   // 0: end, 1: map, 2: start
    return a.seg_buf + (((size_t)row * a.seg_G + g) * 3 + which) * 128 * 128;
  };
  if (a.seg_pass == 0) {
    half = blockIdx.x & 1;
    bh = blockIdx.x >> 1;
    s0p = a.S0 ? a.S0 + (size_t)bh * 128 * a.dv : nullptr;
    sfin = a.S ? a.S + (size_t)bh * 128 * a.dv : nullptr;
  } else if (a.seg_pass == 1) {
    const int per = 2 + 4 * (a.seg_G - 2);
    bh = blockIdx.x / per;
    const int j = blockIdx.x % per;
    if (j < 2) {   // segment 0 from the true initial state, with its outputs
      half = j;
      NC = a.seg_len;
      s0p = a.S0 ? a.S0 + (size_t)bh * 128 * a.dv : nullptr;
      sfin = segmat(bh, 0, 0);
      fin_out = false;
    } else {       // a middle segment: the end state from zero, or the transition map
      const int g = 1 + (j - 2) / 4, r = (j - 2) % 4;
      half = r & 1;
      c0 = g * a.seg_len;
      NC = a.seg_len;
      out_on = false;
      s0mode = r < 2 ? 1 : 2;
      vzero = r >= 2;
      sfin = segmat(bh, g, r < 2 ? 0 : 1);
      fin_out = false;
    }
  } else {         // replay of segment g >= 1 from its start state
    const int per = 2 * (a.seg_G - 1);
    bh = blockIdx.x / per;
    const int g = 1 + (blockIdx.x % per) / 2;
    half = blockIdx.x & 1;
    c0 = g * a.seg_len;
    NC = min(a.seg_len, NCt - c0);
    s0mode = 3;
    s0p = segmat(bh, g, 2);
    sfin = (g == a.seg_G - 1 && a.S) ? a.S + (size_t)bh * 128 * a.dv : nullptr;
  }
  const int b = bh / a.H, h = bh % a.H;
  using CM = CarryMap<MODE>;
  constexpr uint32_t cS = CM::S, cE = CM::E, kRecV = CM::rec, cKP = CM::KP;
  constexpr bool kKdn = (MODE == 2), kExplicitW = (MODE != 0);
  const uint8_t* recs = ws + ((size_t)bh * NCt + c0) * kRecV;

  if (tid == 0) {
    for (int i = 0; i < C_COUNT; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    s_abort = 0;
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (vzero) {   // the map's carry reads V = 0 (U' = 0); no V copy ever lands here
    for (int e = tid; e < 8192 / 16; e += kCarryThreads)
      reinterpret_cast<uint4*>(sm + cV)[e] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, kCarryTmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  // Every thread of a group waits itself (bounded), then one named barrier makes
  // the outcome uniform: a timeout anywhere sets s_abort, which all read after it.
  auto group_wait2 = [&](int bar_id, int nthreads, uint64_t* b1, uint32_t p1, uint64_t* b2,
                         uint32_t p2) -> bool {
    if (!s_abort) {
      bool ok = mbar_wait(b1, p1, kWait);
      if (ok && b2) ok = mbar_wait(b2, p2, kWait);
      if (!ok) s_abort = 1;
    }
    named_bar(bar_id, nthreads);
    return !s_abort;
  };

  if (warp < 8) {
    // ===================================================================== state warps
    const int quad = warp & 3, hc = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const bool leader = (tid == 0);
    const int srow = quad * 32 + lane;          // state row (dk index) = TMEM lane
    // E readout: lanes 0-63 hold the hi-part rows of E, lanes 64-127 the lo-part
    // rows; partners (same row, same 32 columns) split the columns between them
    const int erow = 32 * (quad & 1) + lane;
    const int keep = quad >> 1, send = 1 - keep;
    float S[32];
    uint64_t* last_bar = nullptr;               // leader: its last MMA commit
    uint32_t last_par = 0;
    int n_k = 0;                                // leader: K copies issued
    auto load_k = [&](int c) {    // the dS operand: K, or the record's write keys
      mbar_expect_tx(&bars[C_K], kExplicitW ? 32768 : 16384);
      if (kExplicitW) {
        bulk_load(sm + cKP, recs + (size_t)c * kRecV + CM::rW_, 32768, &bars[C_K]);
      } else {
        tma_load_4d(sm + cKP, &tmK, &bars[C_K], 0, h, (c0 + c) * 64, b);
        tma_load_4d(sm + cKP + 8192, &tmK, &bars[C_K], 64, h, (c0 + c) * 64, b);
      }
      n_k = c + 1;
    };
    if (leader) load_k(0);
    auto store_state_tiles = [&]() {
      uint8_t* sS = sm + cS;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = S[8 * m + e];
        uint4 hi, lo;
        split8(x, hi, lo);
        *reinterpret_cast<uint4*>(sS + sw128_offset(srow, 32 * hc + 8 * m)) = hi;
        *reinterpret_cast<uint4*>(sS + 16384 + sw128_offset(srow, 32 * hc + 8 * m)) = lo;
      }
    };
    // E(c) = U' - [W'_hi ; W'_lo] [S_hi | S_lo].  Descriptors advance by the
    // k-step's 2048 bytes in their start-address field (address >> 4; every
    // operand lies inside shared memory, so the field cannot carry over).  The
    // first k-step starts the S_lo columns (64-127) instead of accumulating.
    auto issue_e = [&](int c) {
      tc_fence_after();
      const uint64_t dsh0 = desc_sw128(smem_u32(sm + cS), 16384, 1024);
      const uint64_t dw0 = desc_sw128(smem_u32(sm + cW + (c & 1) * 32768), 16384, 1024);
      const uint32_t acc = tmem + tE + (c & 1) * 128;
      mma_bf16(acc, dw0, dsh0, I_E1, true);
      mma_bf16(acc + 64, dw0, dsh0 + (16384 >> 4), I_E1, false);
#pragma unroll 1
      for (int ks = 1; ks < 8; ++ks)
        mma_bf16(acc, dw0 + ks * (2048 >> 4), dsh0 + ks * (2048 >> 4), I_E2, true);
      mma_commit(&bars[C_E]);
      last_bar = &bars[C_E];
      last_par = c & 1;
    };
    {
      const long base = (long)srow * a.dv + half * 64 + 32 * hc;
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 v = (s0mode == 0 || s0mode == 3) && s0p
                             ? *reinterpret_cast<const float4*>(s0p + base + j)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        S[j] = v.x; S[j + 1] = v.y; S[j + 2] = v.z; S[j + 3] = v.w;
      }
      if (s0mode == 2) {   // the identity's columns: the transition map of the segment
#pragma unroll
        for (int j = 0; j < 32; ++j) S[j] = (srow == half * 64 + 32 * hc + j) ? 1.f : 0.f;
      }
      store_state_tiles();
    }
    tc_fence_before();
    fence_proxy_async();
    named_bar(1, 256);
    bool ok = true;
    if (leader) {
      if (!s_abort && mbar_wait(&bars[C_M2], 0, kWait) && mbar_wait(&bars[C_W0], 0, kWait)) {
        issue_e(0);
        mbar_arrive(&bars[C_SREADY]);   // S tiles of chunk 0 (for QS(0))
      } else {
        s_abort = 1;
      }
    }
    // row vectors of chunk 0: u (this thread's E row) and gamma_C
    float u_cur = reinterpret_cast<const float*>(recs + rVec)[64 + erow];
    float g_cur = reinterpret_cast<const float*>(recs + rVec)[kKdn ? 128 + srow : 128];
    bool bad = false;

    for (int c = 0; c < NC; ++c) {
      const int slot = c & 1;
      if (SAVE) {   // backward: the state at this chunk's start, as [32 column
                        // quads][128 rows][4] (a warp's rows side by side: 512-byte stores)
        float* dst = a.save_S + ((size_t)bh * NCt + c0 + c) * 16384 + 4 * srow;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(dst + (size_t)((half * 64 + 32 * hc + j) >> 2) * 512) =
              make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
      }
      float u_nxt = 0.f, g_nxt = 0.f;
      if (c + 1 < NC) {   // one chunk ahead; consumed next iteration
        const float* rv = reinterpret_cast<const float*>(recs + (size_t)(c + 1) * kRecV + rVec);
        u_nxt = rv[64 + erow];
        g_nxt = rv[kKdn ? 128 + srow : 128];
      }
      // ---- E -> E and u.E hi/lo tiles, once E(c) is done and PE(c-1) has read
      // the previous E tiles
      if (!(ok = group_wait2(1, 256, &bars[C_E], c & 1, c >= 1 ? &bars[C_PE] : nullptr, (c - 1) & 1)))
        break;
      tc_fence_after();
      {
        float* X = reinterpret_cast<float*>(sm + cW + slot * 32768);   // W'(c) is consumed
        const uint32_t e0 = tmem + lane_off + tE + slot * 128 + 32 * hc;
        float kv[16], t16[16];
        {   // all four loads in flight, one wait; the partner's 16 columns (column
            // halves added) are handed over in X
          float s16[16], u16[16];
          tmem_ld16(e0 + 16 * send, s16);
          tmem_ld16(e0 + 64 + 16 * send, u16);
          tmem_ld16(e0 + 16 * keep, kv);
          tmem_ld16(e0 + 64 + 16 * keep, t16);
          tmem_ld_wait();
          float* xr = X + erow * kXs + 32 * hc + 16 * send;
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(xr + e) =
                make_float4(s16[e] + u16[e], s16[e + 1] + u16[e + 1], s16[e + 2] + u16[e + 2],
                            s16[e + 3] + u16[e + 3]);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) kv[e] += t16[e];
        named_bar(1, 256);
        {
          const float* xk = X + erow * kXs + 32 * hc + 16 * keep;
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const float4 p = *reinterpret_cast<const float4*>(xk + e);
            kv[e] += p.x; kv[e + 1] += p.y; kv[e + 2] += p.z; kv[e + 3] += p.w;
          }
        }
        if (SAVE) {   // backward: E(c), this thread's row and 16 columns, as
                          // [32 column quads][64 rows][4]
          float* dst = a.save_E + ((size_t)bh * NCt + c0 + c) * 8192 + 4 * erow;
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(dst + (size_t)((half * 64 + 32 * hc + 16 * keep + e) >> 2) * 256) =
                make_float4(kv[e], kv[e + 1], kv[e + 2], kv[e + 3]);
        }
        uint8_t* Et = sm + cE;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          float p[8], q8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            p[e] = kv[8 * m + e];
            q8[e] = u_cur * p[e];
          }
          const uint32_t off = sw128_offset(erow, 32 * hc + 16 * keep + 8 * m);
          uint4 hi, lo;
          split8(p, hi, lo);
          *reinterpret_cast<uint4*>(Et + off) = hi;
          *reinterpret_cast<uint4*>(Et + 8192 + off) = lo;
          if (!kKdn) {
            split8(q8, hi, lo);
            *reinterpret_cast<uint4*>(Et + 16384 + off) = hi;
            *reinterpret_cast<uint4*>(Et + 24576 + off) = lo;
          }
        }
      }
      // the leader takes the waits for dS(c)'s and E(c+1)'s other operands off the
      // chain: K(c) before the E-tile barrier, U'(c+1) and W'(c+1) during dS(c)
      bool k_ok = true;
      if (leader) k_ok = !s_abort && mbar_wait(&bars[C_K], c & 1, kWait);
      tc_fence_before();
      fence_proxy_async();
      named_bar(1, 256);
      // ---- leader: dS(c) = K^T [uE_hi | uE_lo]
      bool e_ok = true;
      if (leader) {
        if (k_ok && !s_abort) {
          tc_fence_after();
          const uint32_t kb = smem_u32(sm + cKP), eb = smem_u32(sm + cE);
          const uint32_t ub = kKdn ? eb : eb + 16384;   // u.E (KDN: u = 1, the E tiles)
          const uint64_t du0 = desc_sw128(ub, 8192, 1024), dk0 = desc_sw128(kb, 8192, 1024);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            mma_bf16(tmem + tDS, dk0 + ks * (2048 >> 4), du0 + ks * (2048 >> 4), I_DS2, ks > 0);
            if (kExplicitW)   // PGDN / KDN: dS = (W_hi + W_lo)^T (u.E)
              mma_bf16(tmem + tDS, dk0 + ((16384 + ks * 2048) >> 4), du0 + ks * (2048 >> 4), I_DS, true);
          }
          mma_commit(&bars[C_DS]);
          last_bar = &bars[C_DS];
          last_par = c & 1;
          mbar_arrive(&bars[C_EREADY]);
          if (c + 1 < NC)
            e_ok = mbar_wait(&bars[C_M2], (c + 1) & 1, kWait) &&
                   mbar_wait(&bars[C_W0 + ((c + 1) & 1)], ((c + 1) >> 1) & 1, kWait);
        } else {
          s_abort = 1;
        }
      }
      // ---- S <- gamma_C S + dS (QS(c) must be done reading the old S tiles); the
      // leader refills K for dS(c+1) the moment dS(c) has read it
      if (!(ok = group_wait2(1, 256, &bars[C_DS], c & 1, &bars[C_QS], c & 1))) break;
      if (leader && c + 1 < NC) load_k(c + 1);
      tc_fence_after();
      {
        float t16[16], l16[16], t16b[16], l16b[16];
        const uint32_t dcol0 = tmem + lane_off + tDS + 32 * hc;
        tmem_ld16(dcol0, t16);   // all four loads in flight, one wait
        tmem_ld16(dcol0 + 64, l16);
        tmem_ld16(dcol0 + 16, t16b);
        tmem_ld16(dcol0 + 80, l16b);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          S[e] = g_cur * S[e] + (t16[e] + l16[e]);
          S[16 + e] = g_cur * S[16 + e] + (t16b[e] + l16b[e]);
        }
        store_state_tiles();
      }
      tc_fence_before();
      fence_proxy_async();
      named_bar(1, 256);
      // ---- leader: E(c+1) once S(c+1), U'(c+1) and W'(c+1) are in place
      if (leader) {
        if (c + 1 < NC) {
          if (!s_abort && e_ok)
            issue_e(c + 1);
          else
            s_abort = 1;
        }
        mbar_arrive(&bars[C_SREADY]);
      }
      u_cur = u_nxt;
      g_cur = g_nxt;
    }
    // the leader's MMAs complete before TMEM is freed (its commits track all of them),
    // and its K copies land before the CTA exits
    if (leader && last_bar) mbar_wait(last_bar, last_par, kWait / 4);
    if (leader && n_k > 0) mbar_wait(&bars[C_K], (n_k - 1) & 1, kWait / 4);
    if (!s_abort && sfin) {
      const long base = (long)srow * a.dv + half * 64 + 32 * hc;
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        *reinterpret_cast<float4*>(sfin + base + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        if (a.check_finite && fin_out)
          bad |= !(finite_f(S[j]) && finite_f(S[j + 1]) && finite_f(S[j + 2]) && finite_f(S[j + 3]));
      }
    }
    if (bad) set_status(DR_ERR_NONFINITE);
  } else if (warp >= 9 && warp <= 12) {
    // ===================================================================== output warps
    const int quad = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const bool oleader = (warp == 9 && lane == 0);
    const int i = quad * 16 + (lane & 15);       // token row (M=64 layout: lanes 0-15)
    bool bad = false;
    float qs_cur = reinterpret_cast<const float*>(recs + rVec)[i];
    for (int c = 0; c < NC; ++c) {
      float qs_nxt = 0.f;
      if (c + 1 < NC) qs_nxt = reinterpret_cast<const float*>(recs + (size_t)(c + 1) * kRecV + rVec)[i];
      const int t0 = (c0 + c) * 64, Cc = min(64, a.T - t0);
      // e^g qn . Q S first; the accumulator is released as soon as it is read,
      // and PE(c) lands in it next
      float qv[2][16];
      if (!group_wait2(2, 128, &bars[C_QS], c & 1, nullptr, 0)) break;
      tc_fence_after();
#pragma unroll
      for (int hcol = 0; hcol < 2; ++hcol) {
        const uint32_t q0 = tmem + lane_off + tO + 32 * hcol;
        float qa[16], qb[16];
        tmem_ld16(q0 + 16, qa);   // columns 16-31 of the 32: lanes 16-31 take them from lanes 0-15
        tmem_ld16(q0 + 80, qb);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) qv[hcol][e] = __shfl_sync(0xffffffffu, qs_cur * (qa[e] + qb[e]), lane & 15);
        tmem_ld16(q0, qa);        // columns 0-15
        tmem_ld16(q0 + 64, qb);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) qv[hcol][e] = (lane < 16) ? qs_cur * (qa[e] + qb[e]) : qv[hcol][e];
      }
      tc_fence_before();
      named_bar(2, 128);
      if (oleader) mbar_arrive(&bars[C_QSFREE]);
      if (!group_wait2(2, 128, &bars[C_PE], c & 1, nullptr, 0)) break;
      tc_fence_after();
      __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out) +
                          (((long)b * a.T + t0 + i) * a.H + h) * a.dv + half * 64;
#pragma unroll
      for (int hcol = 0; hcol < 2; ++hcol) {
        const uint32_t p0 = tmem + lane_off + tO + 32 * hcol;
        float x[16], pa[16], pb[16];
        tmem_ld16(p0 + 16, pa);
        tmem_ld16(p0 + 80, pb);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = __shfl_sync(0xffffffffu, pa[e] + pb[e], lane & 15);
        tmem_ld16(p0, pa);
        tmem_ld16(p0 + 64, pb);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = qv[hcol][e] + ((lane < 16) ? pa[e] + pb[e] : x[e]);
        if (out_on && i < Cc) {
          const int col = 32 * hcol + ((lane < 16) ? 0 : 16);
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            float y8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              y8[e] = x[8 * m + e];
              if (a.check_finite) bad |= !finite_f(y8[e]);
            }
            *reinterpret_cast<uint4*>(op + col + 8 * m) = pack8(y8);
          }
        }
      }
      tc_fence_before();
      named_bar(2, 128);
      if (oleader) mbar_arrive(&bars[C_OUTDONE]);
      qs_cur = qs_nxt;
    }
    if (bad) set_status(DR_ERR_NONFINITE);
  } else if (warp == 8 && lane == 0) {
    // ===================================================================== issue lane
    auto wait = [&](int id, uint32_t parity) -> bool {
      if (s_abort) return false;
      if (!mbar_wait(&bars[id], parity, kWait)) {
        s_abort = 1;
        return false;
      }
      return true;
    };
    int n_tv = 0, n_w = 0, n_q = 0;             // copies issued per buffer group
    uint64_t* last_bar = nullptr;               // this thread's last MMA commit
    uint32_t last_par = 0;
    auto load_tv = [&](int c) {
      const uint8_t* rec = recs + (size_t)c * kRecV;
      mbar_expect_tx(&bars[C_TV], vzero ? 16384 : 16384 + 8192);
      bulk_load(sm + cT, rec + rT, 16384, &bars[C_TV]);
      if (!vzero) tma_load_4d(sm + cV, &tmV, &bars[C_TV], half * 64, h, (c0 + c) * 64, b);
      n_tv = c + 1;
    };
    auto load_w = [&](int c) {   // slot c & 1
      uint64_t* bar = &bars[C_W0 + (c & 1)];
      mbar_expect_tx(bar, 32768);
      bulk_load(sm + cW + (c & 1) * 32768, recs + (size_t)c * kRecV + rWp, 32768, bar);
      n_w = c + 1;
    };
    auto load_q = [&](int c) {   // KDN: the record's (Gamma.Q) hi | lo
      mbar_expect_tx(&bars[C_Q], CM::kQ);
      if (kKdn) {
        bulk_load(sm + cQ, recs + (size_t)c * kRecV + rQk, 32768, &bars[C_Q]);
      } else {
        tma_load_4d(sm + cQ, &tmQ, &bars[C_Q], 0, h, (c0 + c) * 64, b);
        tma_load_4d(sm + cQ + 8192, &tmQ, &bars[C_Q], 64, h, (c0 + c) * 64, b);
      }
      n_q = c + 1;
    };
    // U'(c) = [T_hi ; T_lo] V into E slot c & 1 (columns 0-63)
    auto issue_u = [&](int c) {
      tc_fence_after();
      const uint64_t dt0 = desc_sw128(smem_u32(sm + cT), 16, 1024);
      const uint64_t dv0 = desc_sw128(smem_u32(sm + cV), 8192, 1024);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + tE + (c & 1) * 128, dt0 + ks * (32 >> 4), dv0 + ks * (2048 >> 4), I_U2, ks > 0);
      mma_commit(&bars[C_M2]);
      last_bar = &bars[C_M2];
      last_par = c & 1;
    };
    load_tv(0);
    load_w(0);
    if (NC > 1) load_w(1);
    load_q(0);
    bool ok = wait(C_TV, 0);
    if (ok) issue_u(0);
    // T/V of chunk 1 once U'(0) has read chunk 0's
    if (ok && NC > 1 && (ok = wait(C_M2, 0))) load_tv(1);
    // Pipe order per chunk: E(c) [state leader], QS(c) and U'(c+1) [here, while
    // E(c) is read out], dS(c) [state leader], PE(c) [PE lane] while the state is
    // updated, E(c+1).  Each refill follows the last read of its buffer
    // and precedes, in this thread's order, the MMA whose completion could start
    // the buffer's next phase, so no waiter can fall two phases behind.
    for (int c = 0; ok && c < NC; ++c) {
      // QS(c) = Q [S_hi | S_lo]: S(c) tiles ready, PE(c-1) read out of tO
      if (!(ok = wait(C_SREADY, c & 1))) break;
      if (c >= 1 && !(ok = wait(C_OUTDONE, (c - 1) & 1))) break;
      if (!(ok = wait(C_Q, c & 1))) break;
      tc_fence_after();
      {
        const uint64_t ds0 = desc_sw128(smem_u32(sm + cS), 16384, 1024);
        const uint64_t dq0 = desc_sw128(smem_u32(sm + cQ), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t dq = dq0 + (((ks >> 2) * 8192 + (ks & 3) * 32) >> 4);
          const uint64_t ds = ds0 + ks * (2048 >> 4);
          mma_bf16(tmem + tO, dq, ds, I_Q2, ks > 0);
          if (kKdn)   // (Gamma.Q) is a computed operand: its lo term against S_hi
            mma_bf16(tmem + tO, dq + (16384 >> 4), ds, I_N64, true);
        }
        mma_commit(&bars[C_QS]);
        last_bar = &bars[C_QS];
        last_par = c & 1;
      }
      // U'(c+1) into the other E slot (E(c-1) was read out of it before
      // EREADY(c-1)), in the pipe behind QS(c) while E(c) is read out
      if (c + 1 < NC) {
        if (!(ok = wait(C_TV, (c + 1) & 1))) break;
        issue_u(c + 1);
      }
      // W' slot c & 1 for chunk c+2: E(c) and the exchange through the slot
      // finished before EREADY(c)
      if (!(ok = wait(C_EREADY, c & 1))) break;
      if (c + 2 < NC) load_w(c + 2);
      // Q of chunk c+1 once QS(c) has read it
      if (!(ok = wait(C_QS, c & 1))) break;
      if (c + 1 < NC) load_q(c + 1);
      // T/V of chunk c+2 once U'(c+1) has read them
      if (c + 2 < NC) {
        if (!(ok = wait(C_M2, (c + 1) & 1))) break;
        load_tv(c + 2);
      }
    }
    if (!ok) set_status(DR_ERR_TIMEOUT);
    // drain: this thread's last MMAs and every copy issued, so nothing lands after exit
    if (last_bar) mbar_wait(last_bar, last_par, kWait / 4);
    if (n_tv > 0) mbar_wait(&bars[C_TV], (n_tv - 1) & 1, kWait / 4);
    if (n_q > 0) mbar_wait(&bars[C_Q], (n_q - 1) & 1, kWait / 4);
    for (int k = (n_w > 2 ? n_w - 2 : 0); k < n_w; ++k)
      mbar_wait(&bars[C_W0 + (k & 1)], (k >> 1) & 1, kWait / 4);
  } else if (warp == 13 && lane == 0) {
    // ===================================================================== PE lane
    // also refills the P buffer, so the issue lane never waits on PE
    int n_pe = 0, n_p = 0;
    bool ok = true;
    auto load_p = [&](int c) {
      mbar_expect_tx(&bars[C_P], 16384);
      bulk_load(sm + cKP + CM::P, recs + (size_t)c * kRecV + rP, 16384, &bars[C_P]);
      n_p = c + 1;
    };
    load_p(0);
    for (int c = 0; c < NC; ++c) {
      // PE(c) = P_hi [E_hi | E_lo] + P_lo E_hi once the E tiles are written and
      // the output warps have read QS(c) out of tO
      if (s_abort || !mbar_wait(&bars[C_EREADY], c & 1, kWait) || !mbar_wait(&bars[C_P], c & 1, kWait) ||
          !mbar_wait(&bars[C_QSFREE], c & 1, kWait)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t dp0 = desc_sw128(smem_u32(sm + cKP) + CM::P, 16, 1024);
      const uint64_t de0 = desc_sw128(smem_u32(sm + cE), 8192, 1024);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t dp = dp0 + ks * (32 >> 4), de = de0 + ks * (2048 >> 4);
        mma_bf16(tmem + tO, dp, de, I_Q2, ks > 0);
        mma_bf16(tmem + tO, dp + (8192 >> 4), de, I_N64, true);
      }
      mma_commit(&bars[C_PE]);
      n_pe = c + 1;
      if (c + 1 < NC) {
        // P of chunk c+1 once PE(c) has read it
        if (s_abort || !mbar_wait(&bars[C_PE], c & 1, kWait)) {
          ok = false;
          break;
        }
        load_p(c + 1);
      }
    }
    if (!ok && !s_abort) {
      s_abort = 1;
      set_status(DR_ERR_TIMEOUT);
    }
    if (n_pe > 0) mbar_wait(&bars[C_PE], (n_pe - 1) & 1, kWait / 4);
    if (n_p > 0) mbar_wait(&bars[C_P], (n_p - 1) & 1, kWait / 4);
  }

  if (warp == 8 || warp == 13) __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (s_abort && tid == 0) set_status(DR_ERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tmem, kCarryTmem);
}

// ================================================================= segment composition
// Start state of every replayed segment: S_1 = the end state of segment 0, and
// S_{g+1} = M_g S_g + N_g (the middle segment's transition map applied to its
// start, plus its end state from zero).  One CTA per (row, 32 state columns).
__global__ void __launch_bounds__(256) seg_compose_kernel(FwdArgs a) {
  __shared__ float sM[128][129];
  __shared__ float sX[128][33];
  const int tid = threadIdx.x, bh = blockIdx.x >> 2, cb = blockIdx.x & 3;
  const int r = tid >> 1, c16 = 16 * (tid & 1);
  auto mat = [&](int g, int which) {
    return a.seg_buf + (((size_t)bh * a.seg_G + g) * 3 + which) * 128 * 128;
  };
  for (int e = tid; e < 128 * 32; e += 256) {
    const int i = e >> 5, j = e & 31;
    const float x = mat(0, 0)[i * 128 + 32 * cb + j];
    sX[i][j] = x;
    mat(1, 2)[i * 128 + 32 * cb + j] = x;
  }
  for (int g = 1; g + 1 < a.seg_G; ++g) {
    __syncthreads();
    for (int e = tid; e < 128 * 128; e += 256) sM[e >> 7][e & 127] = mat(g, 1)[e];
    __syncthreads();
    float acc[16];
    const float* N = mat(g, 0) + r * 128 + 32 * cb + c16;
#pragma unroll
    for (int q = 0; q < 16; ++q) acc[q] = N[q];
    for (int k = 0; k < 128; ++k) {
      const float m = sM[r][k];
#pragma unroll
      for (int q = 0; q < 16; ++q) acc[q] = fmaf(m, sX[k][c16 + q], acc[q]);
    }
    __syncthreads();
    float* dst = mat(g + 1, 2) + r * 128 + 32 * cb + c16;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      sX[r][c16 + q] = acc[q];
      dst[q] = acc[q];
    }
  }
}

int sm_count() {
  static int count[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!count[dev]) cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev);
  return count[dev];
}

}  // namespace

bool chunk_tc_split_supported(int variant, int dtype, int dk, int dv, int chunk) {
  return (variant == DR_GDN || variant == DR_KLA || variant == DR_PGDN) && dtype == DR_BF16 &&
         dk == 128 && dv == 128 && chunk == 64;
}

// Segments for the carry: with few rows the carry runs on few SMs, so each row
// is cut into G segments.  A first pass runs segment 0 and, for every middle
// segment, its end state from a zero start and its transition map (the same
// carry over V = 0 from the identity); a small kernel composes the start states;
// a second pass replays segments 1 .. G-1 from them.  Two passes over Ls chunks
// instead of one over NC: worth it from G = 3.  The first pass has
// rows (2 + 4 (G - 2)) CTAs, at most one wave of the SM count.
bool seg_plan(int nsm, long rows, int NC, int* G_out, int* Ls_out) {
  *G_out = 0;
  *Ls_out = 0;
  if (nsm <= 0 || rows * 6 > nsm) return false;
  int G = (int)((nsm / rows - 2) / 4) + 2;
  if (G > 64) G = 64;
  for (; G >= 3; --G) {
    const int Ls = (NC + G - 1) / G;
    if (Ls >= 2 && (long)(G - 1) * Ls < NC) {
      *G_out = G;
      *Ls_out = Ls;
      return true;
    }
  }
  return false;
}

size_t chunk_tc_split_workspace_bytes(int variant, int B, int T, int H) {
  const int NC = (T + 63) / 64;
  size_t bytes = (size_t)B * H * NC * (variant == DR_PGDN ? kRecP : kRec);
  int G, Ls;
  if (seg_plan(sm_count(), (long)B * H, NC, &G, &Ls))
    bytes += (size_t)B * H * G * 3 * 128 * 128 * sizeof(float);
  return bytes;
}

cudaError_t launch_chunk_tc_split(const FwdArgs& a, void* workspace, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.B, a.T, a.H, 128) || !make_map(&mk, a.k, a.B, a.T, a.H, 128) ||
      !make_map(&mv, a.v, a.B, a.T, a.H, 128))
    return cudaErrorInvalidValue;
  const int nsm = sm_count();
  if (nsm <= 0) return cudaErrorInvalidValue;
  const long ntask = (long)a.B * a.H * ((a.T + 63) / 64);
  const int pgrid = (int)(ntask < 2L * nsm ? ntask : 2L * nsm);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e;
  if (a.variant == DR_PGDN) {   // chunk-start values of the key statistic first
    e = cudaFuncSetAttribute(pgdn_map_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMapSmem);
    if (e != cudaSuccess) return e;
    pgdn_map_kernel<<<(int)((ntask + kMapTasks - 1) / kMapTasks), kMapTasks * 64, kMapSmem, st>>>(mk, a, ws);
    pgdn_scan_kernel<<<a.B * a.H, 128, 0, st>>>(a, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
#define DR_PREP(V_)                                                                        \
  if (a.variant == V_) {                                                                   \
    e = cudaFuncSetAttribute(chunk_prep_kernel<V_>,                                        \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem); \
    if (e != cudaSuccess) return e;                                                        \
    chunk_prep_kernel<V_><<<pgrid, kPrepThreads, kPrepSmem, st>>>(mq, mk, a, ws);          \
  }
  DR_PREP(DR_GDN) else DR_PREP(DR_KLA) else DR_PREP(DR_PGDN) else return cudaErrorInvalidValue;
#undef DR_PREP
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
#define DR_CARRY1(M_, S_)                                                                  \
  {                                                                                        \
    e = cudaFuncSetAttribute(chunk_carry_kernel<M_, S_>,                                   \
                             cudaFuncAttributeMaxDynamicSharedMemorySize,                  \
                             (int)CarryMap<M_>::bytes);                                    \
    if (e != cudaSuccess) return e;                                                        \
    chunk_carry_kernel<M_, S_><<<a.B * a.H * 2, kCarryThreads, CarryMap<M_>::bytes, st>>>( \
        mq, mk, mv, a, ws);                                                                \
  }
#define DR_CARRY(M_)                   \
  if (a.save_S && a.save_E)            \
    DR_CARRY1(M_, true)                \
  else if (!a.save_S && !a.save_E)     \
    DR_CARRY1(M_, false)               \
  else                                 \
    return cudaErrorInvalidValue;
  const int NC = (a.T + 63) / 64;
  int G, Ls;
  if (!a.save_S && seg_plan(nsm, (long)a.B * a.H, NC, &G, &Ls)) {
    FwdArgs s1 = a;
    s1.seg_pass = 1;
    s1.seg_G = G;
    s1.seg_len = Ls;
    s1.seg_buf = reinterpret_cast<float*>(ws + (size_t)a.B * a.H * NC *
                                               (a.variant == DR_PGDN ? kRecP : kRec));
    FwdArgs s3 = s1;
    s3.seg_pass = 2;
#define DR_CARRY_SEG(M_)                                                                   \
  {                                                                                        \
    e = cudaFuncSetAttribute(chunk_carry_kernel<M_, false>,                                \
                             cudaFuncAttributeMaxDynamicSharedMemorySize,                  \
                             (int)CarryMap<M_>::bytes);                                    \
    if (e != cudaSuccess) return e;                                                        \
    chunk_carry_kernel<M_, false><<<a.B * a.H * (2 + 4 * (G - 2)), kCarryThreads,          \
                                    CarryMap<M_>::bytes, st>>>(mq, mk, mv, s1, ws);        \
    seg_compose_kernel<<<a.B * a.H * 4, 256, 0, st>>>(s1);                                 \
    chunk_carry_kernel<M_, false><<<a.B * a.H * 2 * (G - 1), kCarryThreads,                \
                                    CarryMap<M_>::bytes, st>>>(mq, mk, mv, s3, ws);        \
  }
    if (a.variant == DR_PGDN) DR_CARRY_SEG(1) else DR_CARRY_SEG(0)
#undef DR_CARRY_SEG
    return cudaGetLastError();
  }
  if (a.variant == DR_PGDN) DR_CARRY(1) else DR_CARRY(0)
  return cudaGetLastError();
}

// The tensor-core carry over Diagonal KDN records (bf16 inputs; records written by
// the CUDA-core prep of chunk_simt.cu in the bf16 tile format above).
cudaError_t launch_carry_kdn_tc(const FwdArgs& a, void* workspace, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.B, a.T, a.H, 128) || !make_map(&mk, a.k, a.B, a.T, a.H, 128) ||
      !make_map(&mv, a.v, a.B, a.T, a.H, 128))
    return cudaErrorInvalidValue;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e;
  DR_CARRY(2)
#undef DR_CARRY
  return cudaGetLastError();
}

}  // namespace dr
