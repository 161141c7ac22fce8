// kalman.cu — exact Kalman memory with a dense key covariance, token by token.
//
// KDN notes section 2.2, Eqs. (12)-(17), per (batch, head) and token:
//   S^ = D S,  P^ = D P D^T + diag(omega),  D = diag(alpha)
//   kappa = P^ k / (r + k^T P^ k)
//   S = S^ + kappa (v - S^^T k)^T,  P = (I - kappa k^T) P^,  o = S^T q (after the write)
// With y = P^ k and z = k^T y, k^T P^ = y^T (P^ is symmetric when P_0 is, as a
// covariance is, and each update keeps it so), so the covariance
// update is the symmetric rank-1 downdate P = P^ - y y^T / (r + z), and
// o = S^^T q + (y^T q / (r + z)) e with e = v - S^^T k.  The covariance follows a
// Riccati recursion with no chunked form (the notes' comparison table), so each
// CTA walks the tokens of one (b, h) in order.
//
// CTA = 512 threads = 16 warps, one CTA per (b, h), P and S in registers: warp w
// holds DK/16 rows of P (lane l the columns l + 32 c) and DV/16 columns of S
// (lane l the rows l + 32 c), so every reduction of a token stays inside a warp
// except the two scalars z and y^T q.  The inputs arrive 16 tokens at a time
// by cp.async into a double-buffered shared area, one block ahead; once a block
// has landed, the normalised q and k and the decays of its 16 tokens are formed
// in one pass, so the token loop reads shared memory only.  Two barriers per
// token.  The decode step is the same kernel with T = 1.
#include "dr_common.cuh"

namespace dr {

namespace {

constexpr int kKfWarps = 16;
constexpr int kKfThreads = kKfWarps * 32;
constexpr int kKfTB = 16;   // tokens per staged block

__device__ __forceinline__ void kf_cp16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void kf_cp4(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}

// Full sums over the 32 lanes of x[0 .. N-1] (N a power of two <= 32) by
// halving exchanges: lane l ends up with the sum of x[(l >> (5 - log2 N)) & (N-1)]
// (N - 1 + 5 - log2 N shuffles instead of 5 N).
template <int N>
__device__ __forceinline__ float reduce_scatter(const float* x, int lane, int mask) {
  if constexpr (N == 1) {
    float s = x[0];
#pragma unroll
    for (int m = mask; m >= 1; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    return s;
  } else {
    const bool up = (lane & mask) != 0;   // this lane keeps the upper half
    float w[N / 2];
#pragma unroll
    for (int r = 0; r < N / 2; ++r) {
      const float send = up ? x[r] : x[r + N / 2];
      const float keep = up ? x[r + N / 2] : x[r];
      w[r] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
    }
    return reduce_scatter<N / 2>(w, lane, mask >> 1);
  }
}
template <int N> constexpr int kf_log2() { return N <= 1 ? 0 : 1 + kf_log2<N / 2>(); }

// Dynamic shared memory of one CTA: two raw input blocks, then the processed
// block (fp32 normalised k, q and the decays).
template <int DK, int DV, typename Tin>
struct KfSmem {
  static constexpr int kRaw = kKfTB * (2 * DK * (int)sizeof(Tin) + DV * (int)sizeof(Tin) +
                                       2 * DK * 4) + kKfTB * 4;   // k, q, v, log alpha, omega, r
  static constexpr int kProc = 3 * kKfTB * DK * 4;                  // k^, q^, alpha
  static constexpr int bytes = 2 * kRaw + kProc;
};

// One CTA per (b, h).  Covariance: warp w rows RW w .. RW w + RW - 1, lane l the
// columns l + 32 c.  State: warp w the columns CPW w .. CPW w + CPW - 1, lane l
// the rows l + 32 c -- so S^T k and S^T q reduce within a warp.
template <int DK, int DV, typename Tin>
__global__ void __launch_bounds__(kKfThreads, 1) kalman_kernel(FwdArgs a) {
  constexpr int RW = DK / kKfWarps;   // covariance rows per warp
  constexpr int CPL = DK / 32;        // covariance columns per lane = state rows per lane
  constexpr int CPW = DV / kKfWarps;  // state columns per warp
  constexpr int kOwnRW = 5 - kf_log2<RW>(), kOwnCW = 5 - kf_log2<CPW>();
  static_assert(RW >= 1 && RW <= 32 && CPW >= 1 && CPW <= 32 && CPL >= 1, "tiling");
  const int bh = blockIdx.x;
  const int b = bh / a.H, h = bh % a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = warp * RW, v0 = warp * CPW;

  extern __shared__ __align__(16) uint8_t kf_smem[];
  using SM = KfSmem<DK, DV, Tin>;
  __shared__ float s_y[DK];
  __shared__ float s_zp[kKfWarps], s_yqp[kKfWarps];
  __shared__ float s_e[DV], s_sq[DV];

  float P[RW][CPL], S[CPL][CPW];
#pragma unroll
  for (int i = 0; i < RW; ++i)
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int j = lane + 32 * c;
      P[i][c] = a.aux0 ? a.aux0[((long)bh * DK + r0 + i) * DK + j] : (r0 + i == j ? 1.f : 0.f);
    }
#pragma unroll
  for (int c = 0; c < CPL; ++c)
#pragma unroll
    for (int u = 0; u < CPW; ++u)
      S[c][u] = a.S0 ? a.S0[((long)bh * DK + lane + 32 * c) * DV + v0 + u] : 0.f;

  auto tok = [&](int t) { return ((long)b * a.T + t) * a.H + h; };
  // raw block layout (bytes): k [TB][DK], q [TB][DK], v [TB][DV] (Tin), log alpha
  // [TB][DK], omega [TB][DK], r [TB] (fp32)
  constexpr int oK = 0, oQ = kKfTB * DK * (int)sizeof(Tin), oV = 2 * oQ;
  constexpr int oLA = oV + kKfTB * DV * (int)sizeof(Tin), oOM = oLA + kKfTB * DK * 4;
  constexpr int oR = oOM + kKfTB * DK * 4;
  float* pk = reinterpret_cast<float*>(kf_smem + 2 * SM::kRaw);   // k^ [TB][DK]
  float* pq = pk + kKfTB * DK;                                      // q^ [TB][DK]
  float* pal = pq + kKfTB * DK;                                     // alpha [TB][DK]
  auto fetch = [&](int blk) {   // the raw inputs of tokens 16 blk .. 16 blk + 15 (zero past T)
    uint8_t* raw = kf_smem + (blk & 1) * SM::kRaw;
    constexpr int pr = DK * (int)sizeof(Tin) / 16, pv = DV * (int)sizeof(Tin) / 16, pf = DK / 4;
    constexpr int per_tok = 2 * pr + pv + 2 * pf;
    for (int e = tid; e < kKfTB * per_tok; e += kKfThreads) {
      const int tt = e / per_tok, x = e % per_tok, t = blk * kKfTB + tt;
      const bool real = t < a.T;
      const long ti = tok(real ? t : 0);
      if (x < pr) {
        kf_cp16(raw + oK + tt * DK * sizeof(Tin) + x * 16,
                static_cast<const uint8_t*>(a.k) + ti * DK * sizeof(Tin) + x * 16, real ? 16 : 0);
      } else if (x < 2 * pr) {
        const int y = x - pr;
        kf_cp16(raw + oQ + tt * DK * sizeof(Tin) + y * 16,
                static_cast<const uint8_t*>(a.q) + ti * DK * sizeof(Tin) + y * 16, real ? 16 : 0);
      } else if (x < 2 * pr + pv) {
        const int y = x - 2 * pr;
        kf_cp16(raw + oV + tt * DV * sizeof(Tin) + y * 16,
                static_cast<const uint8_t*>(a.v) + ti * DV * sizeof(Tin) + y * 16, real ? 16 : 0);
      } else if (x < 2 * pr + pv + pf) {
        const int y = x - 2 * pr - pv;
        kf_cp16(raw + oLA + tt * DK * 4 + y * 16, a.log_alpha + ti * DK + y * 4, real ? 16 : 0);
      } else {
        const int y = x - 2 * pr - pv - pf;
        kf_cp16(raw + oOM + tt * DK * 4 + y * 16, a.omega + ti * DK + y * 4, real ? 16 : 0);
      }
    }
    if (tid < kKfTB) {
      const int t = blk * kKfTB + tid;
      kf_cp4(raw + oR + tid * 4, a.r + tok(t < a.T ? t : 0), t < a.T ? 4 : 0);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  auto process = [&](int blk) {   // k^, q^ (warp per token) and alpha of a landed block
    const uint8_t* raw = kf_smem + (blk & 1) * SM::kRaw;
    const Tin* kr = reinterpret_cast<const Tin*>(raw + oK);
    const Tin* qr = reinterpret_cast<const Tin*>(raw + oQ);
    const float* lar = reinterpret_cast<const float*>(raw + oLA);
    for (int tt = warp; tt < kKfTB; tt += kKfWarps) {
      float kx[CPL], qx[CPL], kk = 0.f, qq = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        kx[c] = to_f<Tin>(kr[tt * DK + lane + 32 * c]);
        qx[c] = to_f<Tin>(qr[tt * DK + lane + 32 * c]);
        kk += kx[c] * kx[c];
        qq += qx[c] * qx[c];
      }
      kk = warp_sum(kk);
      qq = warp_sum(qq);
      const float kn = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
      const float qn = a.q_l2norm ? 1.f / fmaxf(sqrtf(qq), 1e-30f) : 1.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        pk[tt * DK + lane + 32 * c] = kx[c] * kn;
        pq[tt * DK + lane + 32 * c] = qx[c] * qn;
        pal[tt * DK + lane + 32 * c] = expf(lar[tt * DK + lane + 32 * c]);
      }
    }
  };

  bool bad = false;
  const int nblk = (a.T + kKfTB - 1) / kKfTB;
  fetch(0);
  if (nblk > 1) fetch(1);
  for (int t = 0; t < a.T; ++t) {
    const int tt = t % kKfTB, blk = t / kKfTB;
    if (tt == 0) {   // a new block: wait for it, form k^, q^, alpha
      if (blk + 1 < nblk)
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      else
        asm volatile("cp.async.wait_group 0;" ::: "memory");
      __syncthreads();
      process(blk);
      __syncthreads();
    }
    const uint8_t* raw = kf_smem + (blk & 1) * SM::kRaw;
    const float* s_kt = pk + tt * DK;
    const float* s_qt = pq + tt * DK;
    const float* s_alt = pal + tt * DK;
    const float* s_omt = reinterpret_cast<const float*>(raw + oOM) + tt * DK;
    const Tin* s_vt = reinterpret_cast<const Tin*>(raw + oV) + tt * DV;
    const float s_rt = reinterpret_cast<const float*>(raw + oR)[tt];
    // this lane's columns j = lane + 32 c (covariance columns and state rows)
    float alj[CPL], kj[CPL], qj[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      alj[c] = s_alt[lane + 32 * c];
      kj[c] = s_kt[lane + 32 * c];
      qj[c] = s_qt[lane + 32 * c];
    }
    // ---- predict P^ = D P D + diag(omega); row partials of y = P^ k
    float acc[RW];
#pragma unroll
    for (int i = 0; i < RW; ++i) {
      const int ri = r0 + i;
      const float ai = s_alt[ri];
      acc[i] = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        float p = ai * alj[c] * P[i][c];
        if (lane + 32 * c == ri) p += s_omt[ri];
        P[i][c] = p;
        acc[i] += p * kj[c];
      }
    }
    {   // y for row rho of this warp on its owner lanes; z and y^T q partials
      const float yr = reduce_scatter<RW>(acc, lane, 16);
      const int rho = (lane >> kOwnRW) & (RW - 1);
      const bool own = (lane & ((1 << kOwnRW) - 1)) == 0;
      float zp = 0.f, yqp = 0.f;
      if (own) {
        s_y[r0 + rho] = yr;
        zp = s_kt[r0 + rho] * yr;
        yqp = s_qt[r0 + rho] * yr;
      }
      zp = warp_sum(zp);
      yqp = warp_sum(yqp);
      if (lane == 0) {
        s_zp[warp] = zp;
        s_yqp[warp] = yqp;
      }
    }
    {   // S^ = D S; this warp's columns of S^^T k and S^^T q -> e = v - S^^T k
      float dk_[CPW], dq_[CPW];
#pragma unroll
      for (int u = 0; u < CPW; ++u) {
        dk_[u] = 0.f;
        dq_[u] = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          S[c][u] *= alj[c];
          dk_[u] += S[c][u] * kj[c];
          dq_[u] += S[c][u] * qj[c];
        }
      }
      const float sk = reduce_scatter<CPW>(dk_, lane, 16);
      const float sq = reduce_scatter<CPW>(dq_, lane, 16);
      if ((lane & ((1 << kOwnCW) - 1)) == 0) {
        const int col = v0 + ((lane >> kOwnCW) & (CPW - 1));
        s_e[col] = to_f<Tin>(s_vt[col]) - sk;
        s_sq[col] = sq;
      }
    }
    __syncthreads();
    // ---- update: P = P^ - y y^T/(r + z); S = S^ + (y/(r + z)) e^T;
    //      o = S^^T q + (y^T q/(r + z)) e
    float z = 0.f, yq = 0.f;
#pragma unroll
    for (int w = 0; w < kKfWarps; ++w) {
      z += s_zp[w];
      yq += s_yqp[w];
    }
    const float inv = 1.f / (s_rt + z);
    float yj[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) yj[c] = s_y[lane + 32 * c] * inv;
#pragma unroll
    for (int i = 0; i < RW; ++i) {
      const float yi = s_y[r0 + i];
#pragma unroll
      for (int c = 0; c < CPL; ++c) P[i][c] -= yi * yj[c];
    }
#pragma unroll
    for (int u = 0; u < CPW; ++u) {
      const float e = s_e[v0 + u];
#pragma unroll
      for (int c = 0; c < CPL; ++c) S[c][u] += yj[c] * e;
    }
    if (lane < CPW) {
      const float o = s_sq[v0 + lane] + yq * inv * s_e[v0 + lane];
      static_cast<Tin*>(a.out)[tok(t) * DV + v0 + lane] = from_f<Tin>(o);
      if (a.check_finite) bad |= !finite_f(o);
    }
    __syncthreads();
    if (tt == kKfTB - 1 && blk + 2 < nblk) fetch(blk + 2);   // this block's buffer is free
  }

  if (a.S) {
#pragma unroll
    for (int c = 0; c < CPL; ++c)
#pragma unroll
      for (int u = 0; u < CPW; ++u) {
        a.S[((long)bh * DK + lane + 32 * c) * DV + v0 + u] = S[c][u];
        if (a.check_finite) bad |= !finite_f(S[c][u]);
      }
  }
  if (a.aux) {
#pragma unroll
    for (int i = 0; i < RW; ++i)
#pragma unroll
      for (int c = 0; c < CPL; ++c) a.aux[((long)bh * DK + r0 + i) * DK + lane + 32 * c] = P[i][c];
  }
  if (bad) set_status(DR_ERR_NONFINITE);
}

}  // namespace

// Forward or decode step (T = 1): one CTA per (b, h); state and covariance may
// be updated in place (each CTA reads its own head's before writing it).
cudaError_t launch_kalman(const FwdArgs& a, int dtype, cudaStream_t st) {
  const int grid = a.B * a.H;
#define DR_KF(DK_, DV_, T_)                                                           \
  if (a.dk == DK_ && a.dv == DV_) {                                                   \
    constexpr int smem = KfSmem<DK_, DV_, T_>::bytes;                                  \
    cudaError_t e = cudaFuncSetAttribute(kalman_kernel<DK_, DV_, T_>,                  \
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem); \
    if (e != cudaSuccess) return e;                                                   \
    kalman_kernel<DK_, DV_, T_><<<grid, kKfThreads, smem, st>>>(a);                   \
    return cudaGetLastError();                                                        \
  }
  if (dtype == DR_BF16) {
    DR_KF(64, 64, __nv_bfloat16) DR_KF(128, 64, __nv_bfloat16)
    DR_KF(64, 128, __nv_bfloat16) DR_KF(128, 128, __nv_bfloat16)
  } else {
    DR_KF(64, 64, float) DR_KF(128, 64, float) DR_KF(64, 128, float) DR_KF(128, 128, float)
  }
#undef DR_KF
  return cudaErrorInvalidValue;
}

}  // namespace dr
