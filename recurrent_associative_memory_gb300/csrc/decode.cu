// decode.cu — one tokenwise step of the recurrence for every (batch, head).
//
// Bandwidth-bound: per (b, h) the fp32 state (dk x dv) is read once and written
// once, everything else is O(dk + dv).  One CTA of 256 threads owns a
// (b, h, column slice) and holds its slice of S in registers between the read
// and the write:
//
//   1. issue the 128-bit streaming loads of S (they fly while 2-3 run);
//   2. load q, k, v and the gates; L2-normalise; form the decay d and the write
//      vector w for the variant (KLA notes Algorithm 1; PDN notes section 2.5,
//      two states A and S; KDN notes section 2.2, predict -> gain -> update;
//      KDA / PKDA: the GDN / PGDN write under per-channel decay; isotropic KDN:
//      one variance per head, KDN notes section 7);
//   3. one pass over S gives both S~^T k and S~^T q (S~ = D S), reduced over
//      rows with registers + shared memory;
//   4. e = v - S~^T k;  o = S~^T q + (w^T q) e  (= S_t^T q, read after write);
//   5. S <- S~ + w e^T, streamed back with 128-bit stores.
#include "dr_common.cuh"

namespace dr {

namespace {

constexpr int kDecodeThreads = 256;

template <typename T>
__device__ __forceinline__ float ld_in(const void* p, long i) {
  return to_f<T>(static_cast<const T*>(p)[i]);
}

// The cluster barrier in two halves: every thread of every CTA in the cluster
// arrives, and a wait (acquire) returns once all have arrived.  The arrive is
// relaxed: a release would hold the thread until its streaming state loads,
// still in flight, had completed; the value it must order (the old gain state)
// has been consumed before the arrive, so the write after the partner's wait
// cannot reach it.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Block-wide sum of one value per thread (all threads must call).
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kDecodeThreads / 32; ++i) s += red[i];
  return s;
}

// Block-wide sums of N values per thread in one pass (two barriers in all);
// red holds N x (warps) floats.
template <int N>
__device__ __forceinline__ void block_sums(float (&v)[N], float* red) {
  constexpr int NW = kDecodeThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = warp_sum(v[i]);
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < N; ++i) red[i * NW + warp] = v[i];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) t += red[i * NW + w];
    v[i] = t;
  }
}

// DK rows x DVS columns of S per CTA.  Slices of up to 128 x 64 keep 32 state
// values per thread, so four CTAs share an SM (more state bytes in flight);
// full 128 x 128 slices keep 64 and run two per SM.
template <int DK, int DVS, typename Tin>
__global__ void __launch_bounds__(kDecodeThreads, (DK * DVS <= 8192) ? 4 : 2)
    decode_kernel(FwdArgs a) {
  constexpr int NCG = DVS / 4;            // float4 column groups
  constexpr int RPW = 32 / NCG;           // rows covered by one warp-wide access
  constexpr int NROWG = 8 * RPW;          // row groups across the CTA
  constexpr int NM = DK / NROWG;          // float4 per thread
  static_assert(NM * NROWG == DK, "tiling");

  __shared__ float s_k[DK], s_q[DK], s_w[DK], s_d[DK];
  __shared__ float s_v[DVS], s_e[DVS];
  __shared__ float s_red[5 * (kDecodeThreads / 32)];
  __shared__ float4 s_pk[NROWG][NCG], s_pq[NROWG][NCG];

  const int nslice = a.dv / DVS;
  const int slice = blockIdx.x % nslice;
  const int bh = blockIdx.x / nslice;
  const int h = bh % a.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cg = lane % NCG, rsub = lane / NCG;
  const int col0 = slice * DVS + 4 * cg;

  // 1. state slice into registers (streaming: read once)
  float4* S4 = reinterpret_cast<float4*>(a.S);
  const long srow0 = (long)bh * DK;
  float4 s[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    const int r = warp * RPW + rsub + NROWG * m;
    s[m] = __ldcs(S4 + (((srow0 + r) * a.dv + col0) >> 2));
  }

  // 2. token inputs and gates (every load issued before the first reduction)
  const long tok = (long)bh;                    // decode layout [B, H, d]
  const bool perchan_la = a.variant == DR_KDN || a.variant == DR_IKDN || a.variant == DR_KDA ||
                          a.variant == DR_PKDA;
  float kc = 0.f, qc = 0.f, g_la = 0.f, g_aux = 0.f, g_om = 0.f;
  if (tid < DK) {
    kc = ld_in<Tin>(a.k, tok * DK + tid);
    qc = ld_in<Tin>(a.q, tok * DK + tid);
    g_la = a.log_alpha[perchan_la ? tok * DK + tid : tok];
    if (a.variant == DR_KDN || a.variant == DR_PGDN || a.variant == DR_PKDA)
      g_aux = a.aux[tok * DK + tid];
    if (a.variant == DR_KDN) g_om = a.omega[tok * DK + tid];
  }
  const float g_r = (a.variant == DR_KDN || a.variant == DR_IKDN) ? a.r[tok] : 0.f;
  const float g_eta = (a.variant == DR_KDN || a.variant == DR_IKDN) ? 0.f : a.eta[tok];
  const float g_aP = (a.variant == DR_PGDN || a.variant == DR_PKDA) ? a.alphaP[tok] : 0.f;
  const float g_bP = (a.variant == DR_PGDN || a.variant == DR_PKDA) ? a.betaP[tok] : 0.f;
  const float g_mu = (a.variant == DR_PGDN || a.variant == DR_PKDA) ? a.mu[h] : 0.f;
  const float g_auxh = a.variant == DR_IKDN ? a.aux[tok] : 0.f;
  const float g_omh = a.variant == DR_IKDN ? a.omega[tok] : 0.f;
  if (tid < DVS) s_v[tid] = ld_in<Tin>(a.v, tok * a.dv + slice * DVS + tid);

  // One block reduction for every sum over channels that needs no normalised key
  // (the norms are applied to the sums): ||k||^2, ||q||^2, k.q, and for Diagonal
  // KDN sum p^ k^2 and sum p^ k q, for isotropic KDN sum alpha^2.
  const bool kdn = a.variant == DR_KDN, ikdn = a.variant == DR_IKDN;
  float alpha = 0.f, p_hat = 0.f;
  if (tid < DK) {
    alpha = expf(g_la);   // per row of S for the per-channel variants, per head otherwise
    if (kdn) p_hat = alpha * alpha * g_aux + g_om;
  }
  float sums[5] = {kc * kc, qc * qc, kc * qc, kdn ? p_hat * kc * kc : (ikdn ? alpha * alpha : 0.f),
                   kdn ? p_hat * kc * qc : 0.f};
  block_sums<5>(sums, s_red);
  const float kk = sums[0], qq = sums[1];
  const float cr = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
  const float qn = a.q_l2norm ? 1.f / fmaxf(sqrtf(qq), 1e-30f) : 1.f;
  kc *= cr;
  qc *= qn;
  const float kk_eff = kk * cr * cr;          // ||k^||^2
  const float kq = sums[2] * cr * qn;         // k^ . q^

  // The gain state (PGDN / PKDA statistic, KDN variance, isotropic KDN variance)
  // is updated in place.  Every slice of a head forms the same gains from it; the
  // slices of a head form one cluster, and the new value is written by slice 0
  // only after every slice has read the old one (cluster barrier below).
  float w = 0.f, d = alpha, aux_new = 0.f, wq = 0.f;
  if (kdn) {
    const float rr = g_r, den = rr + sums[3] * cr * cr;   // r + sum p^ k^2
    if (tid < DK) {
      w = p_hat * kc / den;
      const float u = (a.info_scale / rr) * kc * kc;
      aux_new = p_hat / (1.f + u * p_hat);
    }
    wq = sums[4] * cr * qn / den;
  } else if (ikdn) {   // one variance per head (aux [B, H])
    const float rr = g_r;
    const float b_hat = sums[3] / DK * g_auxh + g_omh;
    const float beta = b_hat / (rr + b_hat * kk_eff);
    if (tid < DK) w = beta * kc;
    wq = beta * kq;
    const float u = a.info_scale * kk_eff / (DK * rr);
    aux_new = b_hat / (1.f + u * b_hat);
  } else if (a.variant == DR_GDN || a.variant == DR_KDA) {
    if (tid < DK) w = g_eta * kc;
    wq = g_eta * kq;
  } else if (a.variant == DR_KLA) {
    const float beta = g_eta / (kk_eff + a.eps);
    if (tid < DK) w = beta * kc;
    wq = beta * kq;
  } else {   // DR_PGDN, DR_PKDA: the bound is per channel, so w . q needs its own sum
    if (tid < DK) {
      const float A = g_aP * g_aux + g_bP * kc * kc;
      // fast log / exp, as in the chunkwise preps (~1e-6 relative in the bound)
      const float rr = __logf(fmaxf(A, a.log_floor)) - g_mu;
      const float sq = __fdividef(rr, 1.f + fabsf(rr));
      w = g_eta * __expf(-a.ln_x * sq) * kc;
      aux_new = A;
    }
  }

  if (tid < DK) {
    s_k[tid] = kc;
    s_q[tid] = qc;
    s_w[tid] = w;
    s_d[tid] = d;
  }
  if (a.variant == DR_PGDN || a.variant == DR_PKDA)
    wq = block_sum(tid < DK ? w * qc : 0.f, s_red);   // includes a __syncthreads
  else
    __syncthreads();
  // every slice has read the old gain state by now (its gains are formed): arrive
  // at the cluster barrier here and wait only before the write at the end, so no
  // slice waits for its partner's whole state pass
  const bool has_aux = a.variant == DR_PGDN || a.variant == DR_PKDA || a.variant == DR_KDN ||
                       a.variant == DR_IKDN;
  if (has_aux && nslice > 1) cluster_arrive();

  // 3. S~^T k and S~^T q partials over this thread's rows
  float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    const int r = warp * RPW + rsub + NROWG * m;
    const float dk_ = s_d[r] * s_k[r], dq_ = s_d[r] * s_q[r];
    pk.x += s[m].x * dk_; pk.y += s[m].y * dk_; pk.z += s[m].z * dk_; pk.w += s[m].w * dk_;
    pq.x += s[m].x * dq_; pq.y += s[m].y * dq_; pq.z += s[m].z * dq_; pq.w += s[m].w * dq_;
  }
  s_pk[warp * RPW + rsub][cg] = pk;
  s_pq[warp * RPW + rsub][cg] = pq;
  __syncthreads();

  // 4. residual and output for this slice's columns
  if (tid < DVS) {
    const float* fk = reinterpret_cast<const float*>(&s_pk[0][0]);
    const float* fq = reinterpret_cast<const float*>(&s_pq[0][0]);
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int g = 0; g < NROWG; ++g) {
      sk += fk[g * DVS + tid];
      sq += fq[g * DVS + tid];
    }
    const float e = s_v[tid] - sk;
    const float o = sq + wq * e;
    s_e[tid] = e;
    static_cast<Tin*>(a.out)[tok * a.dv + slice * DVS + tid] = from_f<Tin>(o);
    if (a.check_finite && !finite_f(o)) set_status(DR_ERR_NONFINITE);
  }
  __syncthreads();

  // 5. S <- D S + w e^T
  const float4 e4 = make_float4(s_e[4 * cg], s_e[4 * cg + 1], s_e[4 * cg + 2], s_e[4 * cg + 3]);
  bool bad = false;
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    const int r = warp * RPW + rsub + NROWG * m;
    const float dr_ = s_d[r], wr = s_w[r];
    float4 n;
    n.x = dr_ * s[m].x + wr * e4.x;
    n.y = dr_ * s[m].y + wr * e4.y;
    n.z = dr_ * s[m].z + wr * e4.z;
    n.w = dr_ * s[m].w + wr * e4.w;
    if (a.check_finite) bad |= !(finite_f(n.x) && finite_f(n.y) && finite_f(n.z) && finite_f(n.w));
    __stcs(S4 + (((srow0 + r) * a.dv + col0) >> 2), n);
  }
  if (bad) set_status(DR_ERR_NONFINITE);
  // 6. the gain state, in place, once every slice of this head has read the old one
  if (has_aux) {
    if (nslice > 1) cluster_wait();
    if (slice == 0) {
      if (a.variant == DR_IKDN) {
        if (tid == 0) a.aux[tok] = aux_new;
      } else if (tid < DK) {
        a.aux[tok * DK + tid] = aux_new;
      }
    }
  }
}

}  // namespace

// Dispatch on (dtype, dk, slice width).  dv = 128 is split into two 64-column
// slices, one CTA each (four per SM): the two slices of a head are launched as a
// cluster of two, so the in-place update of a gain state can wait for both
// slices' reads of it.
cudaError_t launch_decode(const FwdArgs& a, int dtype, cudaStream_t st) {
  const bool split = (a.dv == 128);
  const int dvs = split ? 64 : a.dv;
  const int grid = a.B * a.H * (a.dv / dvs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.dv / dvs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
#define DR_DEC(DK_, DVS_, T_)                                                  \
  if (a.dk == DK_ && dvs == DVS_) {                                            \
    return cudaLaunchKernelEx(&cfg, decode_kernel<DK_, DVS_, T_>, a);          \
  }
  if (dtype == DR_BF16) {
    DR_DEC(64, 64, __nv_bfloat16) DR_DEC(128, 64, __nv_bfloat16)
    DR_DEC(64, 128, __nv_bfloat16) DR_DEC(128, 128, __nv_bfloat16)
  } else {
    DR_DEC(64, 64, float) DR_DEC(128, 64, float)
    DR_DEC(64, 128, float) DR_DEC(128, 128, float)
  }
#undef DR_DEC
  return cudaErrorInvalidValue;
}

}  // namespace dr
