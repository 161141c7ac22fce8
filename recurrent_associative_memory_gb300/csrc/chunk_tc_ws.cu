// chunk_tc_ws.cu — warp-specialised tcgen05 chunkwise forward for GDN and KLA
// (scalar decay, w = coefficient x raw key), bf16 q/k/v/out, dk = dv = 128, chunk 64.
//
// Same chunk algebra as chunk_tc.cu (KLA notes section 2.5, Eqs. (7)-(9), with a
// general write matrix as in the PDN notes section 2.6), reorganised so that
// the chunk-local preparation of chunk c+1 runs concurrently with the state
// carry of chunk c.  One CTA per (b, h, 64-column half of dv); 13 warps:
//
//   chain  (warps 0-3)   state carry of chunk c: E = U' - W' S readout as bf16
//                        hi/lo tiles, then S <- gamma_C S + dS and the output
//                        o = e^g qn . QS + PE.  The fp32 state slice (128 x 64)
//                        lives in these warps' registers.
//   prep   (warps 4-11)  chunk c+1: gates, norms and write coefficients; the
//                        Gram readout into L (fp32) and P (bf16 hi/lo); the
//                        block inverse T = (I + L)^-1; T and T diag(e^g c) as
//                        bf16 hi/lo tiles; W' readout.
//   issue  (warp 12)     one lane issues every TMA load and tcgen05 MMA in the
//                        order M2(c), G(c+1), M3(c), M4(c):
//                          G   Gram [K; Q] K^T                      (M=128)
//                          M2  W' = (T diag(e^g c)) K,  U' = T V    (M=64)
//                          M3  QS = Q S,  E = U' - W' S             (M=64)
//                          M4  PE = P E,  dS = K^T (u . E)          (M=64 / M=128)
//
// Hand-offs are count-1 mbarriers armed by one elected thread of a group after
// the group's named barrier (and fence.proxy.async for shared-memory operands
// the tensor cores read).  Per-slot barriers are used wherever a waiter could
// otherwise fall two phases behind.  Every wait is bounded in wall-clock time;
// a timeout sets DR_ERR_TIMEOUT and every group leaves its loop.
#include "dr_common.cuh"
#include "tc_common.cuh"

namespace dr {

namespace {

using namespace umma;
using namespace tc;

constexpr int kWsThreads = 13 * 32;
constexpr uint64_t kWsWait = 2000000000ull;   // 2 s per bounded wait

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t wKQ = 0;                 // 2 stages x 32 KB: [K rows 0-63 | Q rows 64-127] x 2 kblocks
constexpr uint32_t wV = 65536;              // V tile [64][64]                          8 KB
constexpr uint32_t wT = wV + 8192;          // T hi | T lo | Ts hi | Ts lo             32 KB
                                            //   (L/T fp32 and scratch alias it during the inverse)
constexpr uint32_t wWp = wT + 32768;        // W' hi [64][128] bf16 (lo: E tiles)      16 KB
constexpr uint32_t wS = wWp + 16384;        // S hi | S lo [128][64]                   32 KB
constexpr uint32_t wP = wS + 32768;         // 2 slots x (P hi | P lo)                 32 KB
constexpr uint32_t wE = wP + 32768;         // E hi | E lo | uE hi | uE lo             32 KB
constexpr uint32_t wVec = wE + 32768;       // vectors                                   4 KB
constexpr uint32_t kWsSmem = wVec + 5120 + 1024;   // vectors + readout column factors
constexpr int LDL = 68;                     // fp32 L/T row stride
constexpr int LDX = 36;                     // fp32 scratch row stride

// tensor-memory columns
constexpr uint32_t tGram = 0;               // M=128 x 64
constexpr uint32_t tWp = 64;                // M=64 x 128
constexpr uint32_t tE0 = 192;               // 2 slots of M=64 x 64 (U', then E)
constexpr uint32_t tQS = 320;               // M=64 x 64
constexpr uint32_t tPE = 384;               // M=64 x 64
constexpr uint32_t tDS = 448;               // M=128 x 64
constexpr uint32_t kWsTmem = 512;

constexpr uint32_t I_GRAM = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t I_WP = idesc_bf16(64, 128, 0, 1);
constexpr uint32_t I_N64 = idesc_bf16(64, 64, 0, 1);
constexpr uint32_t I_NEG = idesc_bf16(64, 64, 0, 1, 1);
constexpr uint32_t I_DS = idesc_bf16(128, 64, 1, 1);

// mbarrier indices
enum {
  B_KQ0, B_KQ1, B_V, B_G, B_M2, B_M3, B_M4, B_PF0, B_PF1,   // TMA landed / MMA complete
  B_TREADY, B_PREP, B_SREADY, B_EREADY, B_VF0, B_VF1,       // group hand-offs
  B_COUNT
};

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int VARIANT>
__global__ void __launch_bounds__(kWsThreads, 1)
    chunk_tc_ws_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bars[B_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int s_abort;
  __shared__ volatile int s_ok[3];          // per-group result of the elected wait

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = blockIdx.x & 1;
  const int bh = blockIdx.x >> 1;
  const int b = bh / a.H, h = bh % a.H;
  const int NC = (a.T + 63) / 64;

  // vectors: prep-private, and two slots shared with the chain group
  float* vg = reinterpret_cast<float*>(sm + wVec);   // cumulative log-decay
  float* va = vg + 64;      // coefficient of the raw key row in w
  float* vcr = va + 64;     // key normalisation
  float* vqn = vcr + 64;    // query normalisation
  float* vks = vqn + 64;    // e^{g_j} c_j
  float* vkk = vks + 64;
  float* vqq = vkk + 64;
  float* vla = vqq + 64;
  float* veta = vla + 64;
  float* vslot = veta + 64;   // 2 slots x [vqs 64 | vu 64 | gamma_C 1 (+pad)] = 2 x 192 floats
  float* vC = vslot + 384;    // [4 I][64 j] c_j e^{g_m(I) - g_j}: readout column factors
  float* LT = reinterpret_cast<float*>(sm + wT);
  float* XS = LT + 64 * LDL;

  if (tid == 0) {
    for (int i = 0; i < B_COUNT; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    s_abort = 0;
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, kWsTmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  // elected bounded wait for a whole group; the result is uniform across the group
  auto group_wait = [&](int grp, int bar_id, int nthreads, uint64_t* bar, uint32_t parity,
                        bool leader) -> bool {
    if (leader) {
      bool ok = !s_abort && mbar_wait(bar, parity, kWsWait);
      if (!ok) s_abort = 1;
      s_ok[grp] = ok ? 1 : 0;
    }
    named_bar(bar_id, nthreads);
    const bool ok = s_ok[grp] != 0;
    named_bar(bar_id, nthreads);   // everyone has read s_ok before it is reused
    return ok;
  };

  if (warp < 4) {
    // =====================================================================================
    // chain group: warps 0-3.  Thread = row r of the state slice (TMEM lane r), all 64 columns.
    const int quad = warp;
    const int srow = tid;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const bool leader = (tid == 0);
    float S[64];
    auto store_state_tiles = [&]() {
      uint8_t* sS = sm + wS;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = S[8 * m + e];
        uint4 hi, lo;
        split8(x, hi, lo);
        *reinterpret_cast<uint4*>(sS + sw128_offset(srow, 8 * m)) = hi;
        *reinterpret_cast<uint4*>(sS + 16384 + sw128_offset(srow, 8 * m)) = lo;
      }
    };
    {
      const long base = ((long)bh * 128 + srow) * a.dv + half * 64;
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        const float4 v = a.S0 ? *reinterpret_cast<const float4*>(a.S0 + base + j)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        S[j] = v.x; S[j + 1] = v.y; S[j + 2] = v.z; S[j + 3] = v.w;
      }
      store_state_tiles();
    }
    fence_proxy_async();
    named_bar(1, 128);
    if (leader) mbar_arrive(&bars[B_SREADY]);   // S tiles of chunk 0
    bool bad = false;

    for (int c = 0; c < NC; ++c) {
      const int slot = c & 1;
      const float* vqs = vslot + slot * 192;
      const float* vu = vqs + 64;
      const int t0 = c * 64, Cc = min(64, a.T - t0);
      if (!group_wait(0, 1, 128, &bars[B_M3], c & 1, leader)) break;
      tc_fence_after();
      // E (M=64 layout: rows on lanes 0-15 of each quadrant) -> E and u.E hi/lo tiles
      {
        const int i = quad * 16 + lane;
        const float u = vu[i & 63];
        uint8_t* Et = sm + wE;
#pragma unroll
        for (int hf = 0; hf < 4; ++hf) {
          float ev[16];
          tmem_ld16(tmem + lane_off + tE0 + slot * 64 + 16 * hf, ev);
          tmem_ld_wait();
          if (lane < 16) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              float x[8], y[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                x[e] = ev[8 * m + e];
                y[e] = u * x[e];
              }
              const uint32_t off = sw128_offset(i, 16 * hf + 8 * m);
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
      }
      tc_fence_before();
      fence_proxy_async();
      named_bar(1, 128);
      if (leader) mbar_arrive(&bars[B_EREADY]);
      if (!group_wait(0, 1, 128, &bars[B_M4], c & 1, leader)) break;
      tc_fence_after();
      // epilogue: S <- gamma_C S + dS ; o = qs QS + PE
      {
        const float gC = vqs[128];
#pragma unroll
        for (int hf = 0; hf < 4; ++hf) {
          float ds[16];
          tmem_ld16(tmem + lane_off + tDS + 16 * hf, ds);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) S[16 * hf + e] = gC * S[16 * hf + e] + ds[e];
        }
        store_state_tiles();
        const int i = quad * 16 + lane;
        const float qs = vqs[i & 63];
        __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out) +
                            (((long)b * a.T + t0 + (i & 63)) * a.H + h) * a.dv + half * 64;
#pragma unroll
        for (int hf = 0; hf < 4; ++hf) {
          float qv[16], pe[16];
          tmem_ld16(tmem + lane_off + tQS + 16 * hf, qv);
          tmem_ld16(tmem + lane_off + tPE + 16 * hf, pe);
          tmem_ld_wait();
          if (lane < 16 && i < Cc) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              float x[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                x[e] = qs * qv[8 * m + e] + pe[8 * m + e];
                if (a.check_finite) bad |= !finite_f(x[e]);
              }
              *reinterpret_cast<uint4*>(op + 16 * hf + 8 * m) = pack8(x);
            }
          }
        }
      }
      tc_fence_before();
      fence_proxy_async();
      named_bar(1, 128);
      if (leader) {
        mbar_arrive(&bars[B_SREADY]);            // S tiles of chunk c+1
        mbar_arrive(&bars[B_VF0 + slot]);        // vector slot free again
      }
    }
    if (!s_abort && a.S) {
      const long base = ((long)bh * 128 + srow) * a.dv + half * 64;
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        *reinterpret_cast<float4*>(a.S + base + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        if (a.check_finite)
          bad |= !(finite_f(S[j]) && finite_f(S[j + 1]) && finite_f(S[j + 2]) && finite_f(S[j + 3]));
      }
    }
    if (bad) set_status(DR_ERR_NONFINITE);
  } else if (warp < 12) {
    // =====================================================================================
    // prep group: warps 4-11
    const int ptid = tid - 128, pwarp = warp - 4;
    const int quad = warp & 3, pchalf = pwarp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const bool leader = (ptid == 0);

    float nla = 0.f, neta = 0.f;   // next chunk's gates (thread ptid < 64 = token)
    auto prefetch_gates = [&](int c) {
      const int i = ptid, t = c * 64 + i;
      if (i < 64 && t < a.T) {
        const long ti = ((long)b * a.T + t) * a.H + h;
        nla = a.log_alpha[ti];
        neta = a.eta[ti];
      } else {
        nla = 0.f;
        neta = 0.f;
      }
    };
    // gates of chunk c: decay, norms, write coefficients; vector slot c & 1
    auto gates = [&](int c) -> bool {
      const int st = c & 1;
      const uint8_t* KQ = sm + wKQ + st * 32768;
      if (!group_wait(1, 2, 256, &bars[B_KQ0 + st], (c >> 1) & 1, leader)) return false;
      if (c >= 2 && !group_wait(1, 2, 256, &bars[B_VF0 + st], ((c - 2) >> 1) & 1, leader))
        return false;
      if (ptid < 64) {
        vla[ptid] = nla;
        veta[ptid] = neta;
      }
      if (c + 1 < NC) prefetch_gates(c + 1);
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
      named_bar(2, 256);
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
      named_bar(2, 256);
      if (ptid < 64) {
        const int i = ptid;
        float* vqs = vslot + st * 192;
        float* vu = vqs + 64;
        const float gi = vg[i], gC = vg[63];
        const float kk = vkk[i], qq = vqq[i];
        const float cr = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
        const float qn = a.q_l2norm ? 1.f / fmaxf(sqrtf(qq), 1e-30f) : 1.f;
        float beta = veta[i];
        if (VARIANT == DR_KLA) beta = beta / (kk * cr * cr + a.eps);
        const float coef = beta * cr;
        va[i] = coef;
        vcr[i] = cr;
        vqn[i] = qn;
        const float eg = __expf(gi);
        vks[i] = eg * cr;
        vqs[i] = eg * qn;
        vu[i] = __expf(gC - gi) * coef;
        if (i == 0) vqs[128] = __expf(gC);
      }
      named_bar(2, 256);
      {   // column factors of the readout (read after the next group wait)
        const int I = ptid >> 6, j = ptid & 63;
        vC[ptid] = va[j] * __expf(vg[16 * I + 7] - vg[j]);
      }
      return true;
    };

    prefetch_gates(0);
    bool ok = gates(0);
    for (int c = 0; ok && c < NC; ++c) {
      const int slot = c & 1;
      // ---- Gram readout -> L (fp32) and P (bf16 hi/lo, slot c & 1)
      if (!group_wait(1, 2, 256, &bars[B_G], c & 1, leader)) break;
      if (c >= 2 && !group_wait(1, 2, 256, &bars[B_PF0 + slot], ((c - 2) >> 1) & 1, leader)) break;
      tc_fence_after();
      {
        const int row = quad * 32 + lane;
        const int i = row & 63, I = i >> 4;
        float gv[32];
        ld32cols(tmem + lane_off + tGram + pchalf * 32, gv);
        tmem_ld_wait();
        // one reference token per 16-row block: L_ij = G_ij [rs_i e^{g_i - g_m(I)}] [c_j e^{g_m(I) - g_j}]
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
          uint8_t* Pt = sm + wP + slot * 16384;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = x[8 * m + e];
            uint4 hi, lo;
            split8(y, hi, lo);
            *reinterpret_cast<uint4*>(Pt + sw128_offset(i, pchalf * 32 + 8 * m)) = hi;
            *reinterpret_cast<uint4*>(Pt + 8192 + sw128_offset(i, pchalf * 32 + 8 * m)) = lo;
          }
        }
      }
      tc_fence_before();
      named_bar(2, 256);
      // ---- T = (I + L)^-1 in place: diagonal 16x16 blocks (threads 0-63, one column each)
      {
        const int j = ptid & 15, I = (ptid >> 4) & 3, r0 = 16 * I;
        float t[16];
#pragma unroll
        for (int l = 0; l < 16; ++l) t[l] = (l == j) ? 1.f : 0.f;
        if (ptid < 64) {
#pragma unroll
          for (int i = 1; i < 16; ++i) {
            float s = 0.f;
#pragma unroll
            for (int l = 0; l < i; ++l) s += LT[(r0 + i) * LDL + r0 + l] * t[l];
            if (i > j) t[i] = -s;
          }
        }
        named_bar(2, 256);
        if (ptid < 64) {
#pragma unroll
          for (int i = 0; i < 16; ++i) LT[(r0 + i) * LDL + r0 + j] = t[i];
        }
      }
      named_bar(2, 256);
      // level 1: T_10, T_32 ; level 2: the 32 x 32 lower-left block (TF32x3 mma.sync)
      if (pwarp < 4) {
        const int blk = pwarp >> 1, nt = pwarp & 1;
        const int r0 = 32 * blk + 16, c0 = 32 * blk;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mm3<2>(d, LT + r0 * LDL + c0, LDL, LT + c0 * LDL + c0 + 8 * nt, LDL, lane);
        tile_store(XS + 16 * blk * LDX + 8 * nt, LDX, d, 1.f, lane);
      }
      named_bar(2, 256);
      if (pwarp < 4) {
        const int blk = pwarp >> 1, nt = pwarp & 1;
        const int r0 = 32 * blk + 16, c0 = 32 * blk;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mm3<2>(d, LT + r0 * LDL + r0, LDL, XS + 16 * blk * LDX + 8 * nt, LDX, lane);
        tile_store(LT + r0 * LDL + c0 + 8 * nt, LDL, d, -1.f, lane);
      }
      named_bar(2, 256);
      {
        const int mt = pwarp >> 2, nt = pwarp & 3;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        tile_mm3<4>(d, LT + (32 + 16 * mt) * LDL, LDL, LT + 8 * nt, LDL, lane);
        tile_store(XS + 16 * mt * LDX + 8 * nt, LDX, d, 1.f, lane);
      }
      named_bar(2, 256);
      {
        const int mt = pwarp >> 2, nt = pwarp & 3;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        if (mt == 0)
          tile_mm3<2>(d, LT + 32 * LDL + 32, LDL, XS + 8 * nt, LDX, lane);
        else
          tile_mm3<4>(d, LT + 48 * LDL + 32, LDL, XS + 8 * nt, LDX, lane);
        named_bar(2, 256);
        tile_store(LT + (32 + 16 * mt) * LDL + 8 * nt, LDL, d, -1.f, lane);
      }
      named_bar(2, 256);
      // ---- T and Ts = T diag(ks) -> bf16 hi/lo tiles; they alias L/T, so read first
      {
        const int i = ptid >> 2, c0 = (ptid & 3) * 16;
        float tv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = c0 + e;
          tv[e] = (j <= i) ? LT[i * LDL + j] : 0.f;
        }
        named_bar(2, 256);
        uint8_t* Tt = sm + wT;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          float x[8], y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            x[e] = tv[8 * m + e];
            y[e] = x[e] * vks[c0 + 8 * m + e];
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
      named_bar(2, 256);
      if (leader) mbar_arrive(&bars[B_TREADY]);
      // ---- gates of the next chunk while M2(c) runs
      if (c + 1 < NC && !gates(c + 1)) break;
      // ---- W' readout as a bf16 hi/lo pair (after M2(c)).  The hi tile is free once
      //      M3(c-1) is done; the lo tile borrows the E tiles, free once M4(c-1) is done
      //      (the carry rewrites them only after M3(c), the lo tile's one reader).
      if (!group_wait(1, 2, 256, &bars[B_M2], c & 1, leader)) break;
      if (c >= 1 && !group_wait(1, 2, 256, &bars[B_M3], (c - 1) & 1, leader)) break;
      if (c >= 1 && !group_wait(1, 2, 256, &bars[B_M4], (c - 1) & 1, leader)) break;
      tc_fence_after();
      {
        const int i = quad * 16 + lane;
        uint8_t* Wp = sm + wWp + pchalf * 8192;
        uint8_t* Wl = sm + wE + pchalf * 8192;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float w[16];
          tmem_ld16(tmem + lane_off + tWp + pchalf * 64 + 16 * m, w);
          tmem_ld_wait();
          if (lane < 16) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              float x[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) x[e] = w[8 * hh + e];
              uint4 hi, lo;
              split8(x, hi, lo);
              *reinterpret_cast<uint4*>(Wp + sw128_offset(i, 16 * m + 8 * hh)) = hi;
              *reinterpret_cast<uint4*>(Wl + sw128_offset(i, 16 * m + 8 * hh)) = lo;
            }
          }
        }
      }
      tc_fence_before();
      fence_proxy_async();
      named_bar(2, 256);
      if (leader) mbar_arrive(&bars[B_PREP]);
    }
  } else if (lane == 0) {
    // =====================================================================================
    // issue lane (warp 12): TMA and tcgen05 MMAs
    auto wait = [&](int id, uint32_t parity) -> bool {
      if (s_abort) return false;
      if (!mbar_wait(&bars[id], parity, kWsWait)) {
        s_abort = 1;
        return false;
      }
      return true;
    };
    auto issue_kq = [&](int c) {
      const int st = c & 1;
      uint8_t* base = sm + wKQ + st * 32768;
      mbar_expect_tx(&bars[B_KQ0 + st], 32768);
      const int t0 = c * 64;
      tma_load_4d(base, &tmK, &bars[B_KQ0 + st], 0, h, t0, b);
      tma_load_4d(base + 16384, &tmK, &bars[B_KQ0 + st], 64, h, t0, b);
      tma_load_4d(base + 8192, &tmQ, &bars[B_KQ0 + st], 0, h, t0, b);
      tma_load_4d(base + 16384 + 8192, &tmQ, &bars[B_KQ0 + st], 64, h, t0, b);
    };
    auto issue_v = [&](int c) {
      mbar_expect_tx(&bars[B_V], 8192);
      tma_load_4d(sm + wV, &tmV, &bars[B_V], half * 64, h, c * 64, b);
    };
    auto gram = [&](int c) {
      const uint32_t kq = smem_u32(sm + wKQ + (c & 1) * 32768);
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t d = desc_sw128(kq + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
        mma_bf16(tmem + tGram, d, d, I_GRAM, ks > 0);
      }
      mma_commit(&bars[B_G]);
    };
    issue_kq(0);
    if (NC > 1) issue_kq(1);
    issue_v(0);
    bool ok = wait(B_KQ0, 0);
    if (ok) gram(0);
    for (int c = 0; ok && c < NC; ++c) {
      const int slot = c & 1;
      const uint32_t kq = smem_u32(sm + wKQ + slot * 32768);
      // M2(c): W' = Ts K, U' = T V (T = hi + lo along K)
      if (!(ok = wait(B_TREADY, c & 1) && wait(B_V, c & 1))) break;
      tc_fence_after();
      {
        const uint32_t tb = smem_u32(sm + wT), vt = smem_u32(sm + wV);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t dt = desc_sw128(tb + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
          const uint64_t dts = desc_sw128(tb + 16384 + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
          const uint64_t dk = desc_sw128(kq + (ks & 3) * 2048, 16384, 1024);
          const uint64_t dv = desc_sw128(vt + (ks & 3) * 2048, 8192, 1024);
          mma_bf16(tmem + tWp, dts, dk, I_WP, ks > 0);
          mma_bf16(tmem + tE0 + slot * 64, dt, dv, I_N64, ks > 0);
        }
        mma_commit(&bars[B_M2]);
      }
      // G(c+1) as soon as its inputs landed (the prep group finished reading G(c))
      if (c + 1 < NC) {
        if (!(ok = wait(B_KQ0 + (slot ^ 1), ((c + 1) >> 1) & 1))) break;
        gram(c + 1);
        if (!(ok = wait(B_M2, c & 1))) break;      // V tile free again
        issue_v(c + 1);
      }
      // M3(c): QS = Q (S_hi + S_lo),  E = U' - (W'_hi S_hi + W'_hi S_lo + W'_lo S_hi)
      if (!(ok = wait(B_PREP, c & 1) && wait(B_SREADY, c & 1))) break;
      tc_fence_after();
      {
        const uint32_t sb = smem_u32(sm + wS), wp = smem_u32(sm + wWp), wl = smem_u32(sm + wE);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t dsh = desc_sw128(sb + ks * 2048, 16384, 1024);
          const uint64_t dsl = desc_sw128(sb + 16384 + ks * 2048, 16384, 1024);
          const uint64_t dq = desc_sw128(kq + (ks >> 2) * 16384 + 8192 + (ks & 3) * 32, 16, 1024);
          const uint64_t dw = desc_sw128(wp + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
          const uint64_t dwl = desc_sw128(wl + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
          mma_bf16(tmem + tQS, dq, dsh, I_N64, ks > 0);
          mma_bf16(tmem + tQS, dq, dsl, I_N64, true);
          mma_bf16(tmem + tE0 + slot * 64, dw, dsh, I_NEG, true);
          mma_bf16(tmem + tE0 + slot * 64, dw, dsl, I_NEG, true);
          mma_bf16(tmem + tE0 + slot * 64, dwl, dsh, I_NEG, true);
        }
        mma_commit(&bars[B_M3]);
      }
      // M4(c): PE = P_hi E_hi + P_lo E_hi + P_hi E_lo ;  dS = K^T (uE_hi + uE_lo)
      if (!(ok = wait(B_EREADY, c & 1))) break;
      tc_fence_after();
      {
        const uint32_t pb = smem_u32(sm + wP + slot * 16384), eb = smem_u32(sm + wE);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ph = desc_sw128(pb + ks * 32, 16, 1024);
          const uint64_t pl = desc_sw128(pb + 8192 + ks * 32, 16, 1024);
          const uint64_t eh = desc_sw128(eb + ks * 2048, 8192, 1024);
          const uint64_t el = desc_sw128(eb + 8192 + ks * 2048, 8192, 1024);
          const uint64_t uh = desc_sw128(eb + 16384 + ks * 2048, 8192, 1024);
          const uint64_t ul = desc_sw128(eb + 24576 + ks * 2048, 8192, 1024);
          const uint64_t dk = desc_sw128(kq + ks * 2048, 16384, 1024);
          mma_bf16(tmem + tPE, ph, eh, I_N64, ks > 0);
          mma_bf16(tmem + tPE, pl, eh, I_N64, true);
          mma_bf16(tmem + tPE, ph, el, I_N64, true);
          mma_bf16(tmem + tDS, dk, uh, I_DS, ks > 0);
          mma_bf16(tmem + tDS, dk, ul, I_DS, true);
        }
        mma_commit(&bars[B_M4]);
        mma_commit(&bars[B_PF0 + slot]);
      }
      if (c + 2 < NC) {   // the K/Q stage of chunk c is free once M4(c) is done
        if (!(ok = wait(B_M4, c & 1))) break;
        issue_kq(c + 2);
      }
    }
    if (!ok) set_status(DR_ERR_TIMEOUT);
    // let TMA and MMAs still in flight finish before the CTA frees its resources
    mbar_wait(&bars[B_M4], (NC - 1) & 1, kWsWait / 4);
  }

  if (warp == 12) __syncwarp();   // lanes 1-31 of the issue warp wait for lane 0
  tc_fence_before();
  __syncthreads();
  if (s_abort && tid == 0) set_status(DR_ERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tmem, kWsTmem);
}

}  // namespace

bool chunk_tc_ws_supported(int variant, int dtype, int dk, int dv, int chunk) {
  return (variant == DR_GDN || variant == DR_KLA) && dtype == DR_BF16 && dk == 128 &&
         dv == 128 && chunk == 64;
}

cudaError_t launch_chunk_tc_ws(const FwdArgs& a, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.B, a.T, a.H, 128) || !make_map(&mk, a.k, a.B, a.T, a.H, 128) ||
      !make_map(&mv, a.v, a.B, a.T, a.H, 128))
    return cudaErrorInvalidValue;
  const int grid = a.B * a.H * 2;
#define DR_WS(V_)                                                                          \
  if (a.variant == V_) {                                                                   \
    cudaError_t e = cudaFuncSetAttribute(chunk_tc_ws_kernel<V_>,                           \
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,      \
                                         (int)kWsSmem);                                    \
    if (e != cudaSuccess) return e;                                                        \
    chunk_tc_ws_kernel<V_><<<grid, kWsThreads, kWsSmem, st>>>(mq, mk, mv, a);              \
    return cudaGetLastError();                                                             \
  }
  DR_WS(DR_GDN) DR_WS(DR_KLA)
#undef DR_WS
  return cudaErrorInvalidValue;
}

}  // namespace dr
