// kalman.cu — exact Kalman memory with a dense key covariance, token by token.
//
// KDN notes section 2.2, Eqs. (12)-(17), per (batch, head) and token:
//   S^ = D S,  P^ = D P D^T + diag(omega),  D = diag(alpha)
//   kappa = P^ k / (r + k^T P^ k)
//   S = S^ + kappa (v - S^^T k)^T,  P = (I - kappa k^T) P^,  o = S^T q (after the write)
// With y = P^ k and z = k^T y, k^T P^ = y^T (P^ is symmetric), so the covariance
// update is the symmetric rank-1 downdate P = P^ - y y^T / (r + z), and
// o = S^^T q + (y^T q / (r + z)) e with e = v - S^^T k.  The covariance follows a
// Riccati recursion with no chunked form (the notes' comparison table), so each
// CTA walks the tokens of one (b, h) in order.
//
// CTA = 512 threads = 16 warps; warp w holds rows DK/16 w .. DK/16 (w + 1) - 1 of P
// and of the CTA's NVC-column slice of S in registers, lane l the P columns
// l + 32 c and the S columns l + 32 c.  The inputs arrive 16 tokens at a time
// by cp.async into a double-buffered shared area, one block ahead; once a block
// has landed, the normalised q and k and the decays of its 16 tokens are formed
// in one pass, so the token loop reads shared memory only.  Two barriers per
// token.  Forward: 32 state columns per CTA (the covariance is
// recomputed by every slice, only slice 0 writes it) while those 4 B H CTAs fit
// in one wave at one CTA per SM, else all columns in one CTA per head; the
// decode step always takes the latter, so state and covariance are updated in
// place.
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

// Dynamic shared memory of one CTA: two raw input blocks, then the processed
// block (fp32 normalised k, q and the decays).
template <int DK, int NVC, typename Tin>
struct KfSmem {
  static constexpr int kRaw = kKfTB * (2 * DK * (int)sizeof(Tin) + NVC * (int)sizeof(Tin) +
                                       2 * DK * 4) + kKfTB * 4;   // k, q, v, log alpha, omega, r
  static constexpr int kProc = 3 * kKfTB * DK * 4;                  // k^, q^, alpha
  static constexpr int bytes = 2 * kRaw + kProc;
};

template <int DK, int NVC, typename Tin>
__global__ void __launch_bounds__(kKfThreads, 1) kalman_kernel(FwdArgs a) {
  constexpr int RW = DK / kKfWarps;   // rows per warp
  constexpr int CPL = DK / 32;    // covariance columns per lane
  constexpr int SPL = NVC / 32;   // state columns per lane
  static_assert(RW <= 32 && CPL >= 1 && SPL >= 1, "tiling");
  const int nsl = a.dv / NVC;
  const int slice = blockIdx.x % nsl, bh = blockIdx.x / nsl;
  const int b = bh / a.H, h = bh % a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = warp * RW;

  extern __shared__ __align__(16) uint8_t kf_smem[];
  using SM = KfSmem<DK, NVC, Tin>;
  __shared__ float s_y[DK];
  __shared__ float s_zp[kKfWarps], s_yqp[kKfWarps];
  __shared__ float s_dp[kKfWarps][NVC], s_qp[kKfWarps][NVC];

  float P[RW][CPL], S[RW][SPL];
#pragma unroll
  for (int i = 0; i < RW; ++i) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int j = lane + 32 * c;
      P[i][c] = a.aux0 ? a.aux0[((long)bh * DK + r0 + i) * DK + j] : (r0 + i == j ? 1.f : 0.f);
    }
#pragma unroll
    for (int c = 0; c < SPL; ++c) {
      const int v = slice * NVC + lane + 32 * c;
      S[i][c] = a.S0 ? a.S0[((long)bh * DK + r0 + i) * a.dv + v] : 0.f;
    }
  }

  auto tok = [&](int t) { return ((long)b * a.T + t) * a.H + h; };
  // raw block layout (bytes): k [TB][DK], q [TB][DK], v [TB][NVC] (Tin), log alpha
  // [TB][DK], omega [TB][DK], r [TB] (fp32)
  constexpr int oK = 0, oQ = kKfTB * DK * (int)sizeof(Tin), oV = 2 * oQ;
  constexpr int oLA = oV + kKfTB * NVC * (int)sizeof(Tin), oOM = oLA + kKfTB * DK * 4;
  constexpr int oR = oOM + kKfTB * DK * 4;
  float* pk = reinterpret_cast<float*>(kf_smem + 2 * SM::kRaw);   // k^ [TB][DK]
  float* pq = pk + kKfTB * DK;                                      // q^ [TB][DK]
  float* pal = pq + kKfTB * DK;                                     // alpha [TB][DK]
  auto fetch = [&](int blk) {   // the raw inputs of tokens 16 blk .. 16 blk + 15 (zero past T)
    uint8_t* raw = kf_smem + (blk & 1) * SM::kRaw;
    constexpr int pr = DK * (int)sizeof(Tin) / 16, pv = NVC * (int)sizeof(Tin) / 16, pf = DK / 4;
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
        kf_cp16(raw + oV + tt * NVC * sizeof(Tin) + y * 16,
                static_cast<const uint8_t*>(a.v) + (ti * a.dv + slice * NVC) * sizeof(Tin) + y * 16,
                real ? 16 : 0);
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
    if (tt == 0) {   // a new block: wait for it, form k^, q^, alpha, refill the other buffer
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
    const Tin* s_vt = reinterpret_cast<const Tin*>(raw + oV) + tt * NVC;
    const float s_rt = reinterpret_cast<const float*>(raw + oR)[tt];
    // ---- predict; y = P^ k (row sums), z = k^T y and y^T q (warp partials); S^ = D S
    //      and the column partials of S^^T k, S^^T q
    float y[RW];
    float zp = 0.f, yqp = 0.f;
    float alj[CPL], kj[CPL];   // this lane's columns
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      alj[c] = s_alt[lane + 32 * c];
      kj[c] = s_kt[lane + 32 * c];
    }
#pragma unroll
    for (int i = 0; i < RW; ++i) {
      const int ri = r0 + i;
      const float ai = s_alt[ri];
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int j = lane + 32 * c;
        float p = ai * alj[c] * P[i][c];
        if (j == ri) p += s_omt[ri];
        P[i][c] = p;
        acc += p * kj[c];
      }
      acc = warp_sum(acc);
      y[i] = acc;
      zp += s_kt[ri] * acc;
      yqp += s_qt[ri] * acc;
      if (lane == i) s_y[ri] = acc;
    }
    if (lane == 0) {
      s_zp[warp] = zp;
      s_yqp[warp] = yqp;
    }
#pragma unroll
    for (int c = 0; c < SPL; ++c) {
      float dk_ = 0.f, dq_ = 0.f;
#pragma unroll
      for (int i = 0; i < RW; ++i) {
        S[i][c] *= s_alt[r0 + i];
        dk_ += S[i][c] * s_kt[r0 + i];
        dq_ += S[i][c] * s_qt[r0 + i];
      }
      s_dp[warp][lane + 32 * c] = dk_;
      s_qp[warp][lane + 32 * c] = dq_;
    }
    __syncthreads();
    // ---- update: P = P^ - y y^T/(r + z); e = v - S^^T k; S = S^ + (y/(r + z)) e^T;
    //      o = S^^T q + (y^T q/(r + z)) e
    float z = 0.f, yq = 0.f;
#pragma unroll
    for (int w = 0; w < kKfWarps; ++w) {
      z += s_zp[w];
      yq += s_yqp[w];
    }
    const float inv = 1.f / (s_rt + z);
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const float yj = s_y[lane + 32 * c] * inv;
#pragma unroll
      for (int i = 0; i < RW; ++i) P[i][c] -= y[i] * yj;
    }
#pragma unroll
    for (int c = 0; c < SPL; ++c) {
      const int vl = lane + 32 * c;
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int w = 0; w < kKfWarps; ++w) {
        sk += s_dp[w][vl];
        sq += s_qp[w][vl];
      }
      const float e = to_f<Tin>(s_vt[vl]) - sk;
#pragma unroll
      for (int i = 0; i < RW; ++i) S[i][c] += y[i] * inv * e;
      if (warp == 0) {
        const float o = sq + yq * inv * e;
        static_cast<Tin*>(a.out)[tok(t) * a.dv + slice * NVC + vl] = from_f<Tin>(o);
        if (a.check_finite) bad |= !finite_f(o);
      }
    }
    __syncthreads();
    if (tt == kKfTB - 1 && blk + 2 < nblk) fetch(blk + 2);   // this block's buffer is free
  }

  if (a.S) {
#pragma unroll
    for (int i = 0; i < RW; ++i)
#pragma unroll
      for (int c = 0; c < SPL; ++c) {
        a.S[((long)bh * DK + r0 + i) * a.dv + slice * NVC + lane + 32 * c] = S[i][c];
        if (a.check_finite) bad |= !finite_f(S[i][c]);
      }
  }
  if (a.aux && slice == 0) {
#pragma unroll
    for (int i = 0; i < RW; ++i)
#pragma unroll
      for (int c = 0; c < CPL; ++c) a.aux[((long)bh * DK + r0 + i) * DK + lane + 32 * c] = P[i][c];
  }
  if (bad) set_status(DR_ERR_NONFINITE);
}

}  // namespace

int kalman_sm_count() {
  static int count[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!count[dev]) cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev);
  return count[dev];
}

// Forward with 32 state columns per CTA, or with all of them in one CTA per
// head (few heads per SM left to use, and the decode step: T = 1, state and
// covariance in place).
cudaError_t launch_kalman(const FwdArgs& a, int dtype, cudaStream_t st, bool whole_columns) {
  const int nvc = whole_columns ? a.dv : 32;
  const int grid = a.B * a.H * (a.dv / nvc);
#define DR_KF(DK_, NVC_, T_)                                                          \
  if (a.dk == DK_ && nvc == NVC_) {                                                   \
    constexpr int smem = KfSmem<DK_, NVC_, T_>::bytes;                                 \
    cudaError_t e = cudaFuncSetAttribute(kalman_kernel<DK_, NVC_, T_>,                 \
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem); \
    if (e != cudaSuccess) return e;                                                   \
    kalman_kernel<DK_, NVC_, T_><<<grid, kKfThreads, smem, st>>>(a);                  \
    return cudaGetLastError();                                                        \
  }
  if (dtype == DR_BF16) {
    DR_KF(64, 32, __nv_bfloat16) DR_KF(128, 32, __nv_bfloat16) DR_KF(64, 64, __nv_bfloat16)
    DR_KF(128, 64, __nv_bfloat16) DR_KF(64, 128, __nv_bfloat16) DR_KF(128, 128, __nv_bfloat16)
  } else {
    DR_KF(64, 32, float) DR_KF(128, 32, float) DR_KF(64, 64, float)
    DR_KF(128, 64, float) DR_KF(64, 128, float) DR_KF(128, 128, float)
  }
#undef DR_KF
  return cudaErrorInvalidValue;
}

}  // namespace dr
