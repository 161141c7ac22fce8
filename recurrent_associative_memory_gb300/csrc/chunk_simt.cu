// chunk_simt.cu — fused chunkwise forward on fp32 CUDA cores (all variants).
//
// One CTA of 256 threads owns one (b, h, 32-column slice of dv) and walks the
// sequence chunk by chunk, keeping its dk x 32 slice of S in shared memory.
// Within a chunk of C <= 64 tokens (KLA notes section 2.5, Eqs. (7)-(9),
// generalised to a write matrix W as in the PDN notes section 2.6):
//
//   prep   k^, q^ (optional L2 norm), cumulative log-decay g, write vectors W
//          (GDN/KLA scalars; PGDN statistic scan; KDN variance scan, carried
//          across chunks per channel in registers)
//   Gram   L = strict_lower((K W^T) . exp(g_i - g_j)),  P = lower((Q W^T) . exp(...))
//   solve  T = (I + L)^-1 by 16x16 block forward substitution
//   carry  R = V - (Gamma.K) S ;  E = T R ;  O = (Gamma.Q) S + P E
//          S <- diag(gamma_C) S + (exp(g_C - g_j).W)^T E
//
// Decay ratios are always formed from log differences (KDN notes section 6,
// numerics).  With per-channel decay (KDN) the Gram cannot factor as a single
// matrix product; the chunk is cut into 16-token sub-chunks and each block
// (I, J) of the Gram uses a reference point r with every factor bounded:
//   J < I : k_i exp(g_i - g_b) * w_j exp(g_e(J) - g_j) * exp(g_b - g_e(J)),
//           b = last token of sub-chunk I-1, e(J) = last token of sub-chunk J
//           (all three factors <= 1);
//   J = I : the same with the mid token of the sub-chunk as reference, so the
//           two growing factors stay below exp(decay over 8 tokens).
// This path serves the fp32 mode (tolerance 1e-4) and any shape the
// tensor-core path does not take.
#include "dr_common.cuh"

namespace dr {

namespace {

constexpr int kThreads = 256;
constexpr int CM = 64;      // max chunk handled on chip
constexpr int NV = 32;      // dv columns per CTA
constexpr int CS = CM + 4;  // row stride of token-minor (transposed) buffers
constexpr int NSM = CM / 16;

template <int DK>
struct SimtSmem {
  static constexpr int kKt = DK * CS;          // K^T  [DK][CS]  (k^, then scaled copies)
  static constexpr int kQt = DK * CS;          // Q^T  [DK][CS]
  static constexpr int kW = CM * DK;           // W    [CM][DK]
  static constexpr int kS = DK * NV;           // S    [DK][NV]
  static constexpr int kV = CM * NV;           // V / R [CM][NV]
  static constexpr int kE = CM * NV;           // E    [CM][NV]
  static constexpr int kL = CM * CS;           // L^T  [CM][CS]
  static constexpr int kP = CM * CS;           // P^T  [CM][CS]
  static constexpr int kX = (CM * DK > CM * CS) ? CM * DK : CM * CS;  // g | W^T | T^T
  static constexpr int kF = (NSM * NSM + 4 * NSM) * DK;  // decay factor vectors
  static constexpr int kVec = 8 * CM + DK;
  static constexpr int total = kKt + kQt + kW + kS + kV + kE + kL + kP + kX + kF + kVec;
};

__device__ __forceinline__ long tok_index(const FwdArgs& a, int b, int t, int h) {
  return ((long)b * a.T + t) * a.H + h;
}

template <typename Tin>
__device__ __forceinline__ float ldg_in(const void* p, long i) {
  return to_f<Tin>(static_cast<const Tin*>(p)[i]);
}

template <int DK, typename Tin>
__global__ void __launch_bounds__(kThreads, 1) chunk_simt_kernel(FwdArgs a, int C) {
  using SM = SimtSmem<DK>;
  extern __shared__ __align__(16) float sm[];
  float* sKt = sm;
  float* sQt = sKt + SM::kKt;
  float* sW = sQt + SM::kQt;
  float* sS = sW + SM::kW;
  float* sV = sS + SM::kS;
  float* sE = sV + SM::kV;
  float* sLt = sE + SM::kE;
  float* sPt = sLt + SM::kL;
  float* sX = sPt + SM::kP;
  float* sF = sX + SM::kX;
  float* sg = sF + SM::kF;        // [CM] scalar cumulative log-decay
  float* sb1 = sg + CM;           // [CM] beta (GDN/KLA), eta (PGDN), r (KDN)
  float* sb2 = sb1 + CM;          // [CM] alphaP
  float* sb3 = sb2 + CM;          // [CM] betaP
  float* sz = sb3 + CM;           // [CM] KDN sum p^ k^2
  float* sgC = sz + CM;           // [DK] gamma_C per channel (scalar: [0])

  const int ntile = a.dv / NV;
  const int tile = blockIdx.x % ntile;
  const int bh = blockIdx.x / ntile;
  const int b = bh / a.H, h = bh % a.H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool kdn = (a.variant == DR_KDN);
  const bool pgdn = (a.variant == DR_PGDN);

  // factor vectors inside sF
  float* fOff = sF;                       // [NSM*NSM][DK]  exp(g_b(I) - g_e(J)), J < I
  float* fDa = fOff + NSM * NSM * DK;     // [NSM][DK]      exp(g_b(I) - g_m(I))
  float* fDb = fDa + NSM * DK;            // [NSM][DK]      exp(g_m(I) - g_e(I))
  float* fGb = fDb + NSM * DK;            // [NSM][DK]      exp(g_b(I))  (b(0): chunk start, 1)
  float* fWc = fGb + NSM * DK;            // [NSM][DK]      exp(g_e(last) - g_e(I))

  // state tile
  for (int e = tid; e < DK * NV; e += kThreads) {
    const int c = e / NV, n = e % NV;
    sS[e] = a.S0 ? a.S0[((long)bh * DK + c) * a.dv + tile * NV + n] : 0.f;
  }
  // per-channel carried gain state: PGDN A / KDN p
  float carry = 0.f;
  if (tid < DK) {
    if (pgdn) carry = a.aux0 ? a.aux0[(long)bh * DK + tid] : 0.f;
    if (kdn) carry = a.aux0 ? a.aux0[(long)bh * DK + tid] : 1.f;
  }
  const float mu_h = pgdn ? a.mu[h] : 0.f;
  bool bad = false;

  for (int t0 = 0; t0 < a.T; t0 += C) {
    const int Cc = min(C, a.T - t0);
    const int Cp = (Cc + 15) & ~15;
    const int NS = Cp / 16;
    __syncthreads();

    // ---- 1. loads (rows Cc..Cp-1 are padding: zero inputs, no decay)
    for (int e = tid; e < Cp * DK; e += kThreads) {
      const int i = e / DK, c = e % DK;
      float kv = 0.f, qv = 0.f;
      if (i < Cc) {
        const long ti = tok_index(a, b, t0 + i, h) * DK + c;
        kv = ldg_in<Tin>(a.k, ti);
        qv = ldg_in<Tin>(a.q, ti);
      }
      sKt[c * CS + i] = kv;
      sQt[c * CS + i] = qv;
      if (kdn) {
        const long ti = tok_index(a, b, t0 + i, h) * DK + c;
        sX[i * DK + c] = (i < Cc) ? a.log_alpha[ti] : 0.f;
        sW[i * DK + c] = (i < Cc) ? a.omega[ti] : 0.f;
      }
    }
    for (int e = tid; e < Cp * NV; e += kThreads) {
      const int i = e / NV, n = e % NV;
      sV[e] = (i < Cc) ? ldg_in<Tin>(a.v, tok_index(a, b, t0 + i, h) * a.dv + tile * NV + n) : 0.f;
    }
    if (tid < Cp) {
      const int i = tid;
      const bool real = i < Cc;
      const long ti = real ? tok_index(a, b, t0 + i, h) : 0;
      if (!kdn) {
        sg[i] = real ? a.log_alpha[ti] : 0.f;
        sb1[i] = real ? a.eta[ti] : 0.f;
      } else {
        sb1[i] = real ? a.r[ti] : 1.f;
      }
      if (pgdn) {
        sb2[i] = real ? a.alphaP[ti] : 1.f;
        sb3[i] = real ? a.betaP[ti] : 0.f;
      }
    }
    __syncthreads();

    // ---- 2. L2 norms (in place) and the GDN/KLA write scale
    for (int i = warp; i < Cp; i += kThreads / 32) {
      float kk = 0.f, qq = 0.f;
      for (int c = lane; c < DK; c += 32) {
        const float kv = sKt[c * CS + i], qv = sQt[c * CS + i];
        kk += kv * kv;
        qq += qv * qv;
      }
      kk = warp_sum(kk);
      qq = warp_sum(qq);
      const float kn = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
      const float qn = a.q_l2norm ? 1.f / fmaxf(sqrtf(qq), 1e-30f) : 1.f;
      for (int c = lane; c < DK; c += 32) {
        sKt[c * CS + i] *= kn;
        sQt[c * CS + i] *= qn;
      }
      if (lane == 0) {
        const float kk_eff = kk * kn * kn;
        if (a.variant == DR_KLA) sb1[i] = sb1[i] / (kk_eff + a.eps);
      }
    }
    __syncthreads();

    // ---- 3. cumulative decay and write vectors
    if (!kdn) {
      if (warp == 0) {  // inclusive scan of log-alpha over Cp <= 64 tokens, 2 per lane
        const float x0 = (2 * lane < Cp) ? sg[2 * lane] : 0.f;
        const float x1 = (2 * lane + 1 < Cp) ? sg[2 * lane + 1] : 0.f;
        float s = x0 + x1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, s, o);
          if (lane >= o) s += y;
        }
        const float base = s - (x0 + x1);
        if (2 * lane < Cp) sg[2 * lane] = base + x0;
        if (2 * lane + 1 < Cp) sg[2 * lane + 1] = s;
      }
      if (pgdn) {
        if (tid < DK) {  // statistic scan for channel c, carried across chunks
          const int c = tid;
          float A = carry;
          for (int i = 0; i < Cp; ++i) {
            const float kv = sKt[c * CS + i];
            A = sb2[i] * A + sb3[i] * kv * kv;
            const float rr = logf(fmaxf(A, a.log_floor)) - mu_h;
            const float s = rr / (1.f + fabsf(rr));
            sW[i * DK + c] = sb1[i] * expf(-a.ln_x * s) * kv;
          }
          carry = A;
        }
      } else {
        for (int e = tid; e < Cp * DK; e += kThreads) {
          const int i = e / DK, c = e % DK;
          sW[e] = sb1[i] * sKt[c * CS + i];
        }
      }
      __syncthreads();
    } else {
      if (tid < DK) {  // variance scan (predict -> update) and cumulative decay, channel c
        const int c = tid;
        float p = carry, g = 0.f;
        for (int i = 0; i < Cp; ++i) {
          const float la = sX[i * DK + c];
          const float al = expf(la);
          const float p_hat = al * al * p + sW[i * DK + c];
          const float kv = sKt[c * CS + i];
          const float u = (a.info_scale / sb1[i]) * kv * kv;
          sW[i * DK + c] = p_hat;
          p = p_hat / (1.f + u * p_hat);
          g += la;
          sX[i * DK + c] = g;
        }
        carry = p;
      }
      __syncthreads();
      for (int i = warp; i < Cp; i += kThreads / 32) {
        float z = 0.f;
        for (int c = lane; c < DK; c += 32) {
          const float kv = sKt[c * CS + i];
          z += sW[i * DK + c] * kv * kv;
        }
        z = warp_sum(z);
        if (lane == 0) sz[i] = z;
      }
      __syncthreads();
      for (int e = tid; e < Cp * DK; e += kThreads) {
        const int i = e / DK, c = e % DK;
        sW[e] = sW[e] * sKt[c * CS + i] / (sb1[i] + sz[i]);
      }
      __syncthreads();
      // factor vectors from the per-channel g (g_{-1} = 0 at the chunk start)
      for (int e = tid; e < NS * DK; e += kThreads) {
        const int I = e / DK, c = e % DK;
        const float gb = (I == 0) ? 0.f : sX[(16 * I - 1) * DK + c];
        const float gm = sX[(16 * I + 7) * DK + c];
        const float ge = sX[(16 * I + 15) * DK + c];
        fDa[I * DK + c] = expf(gb - gm);
        fDb[I * DK + c] = expf(gm - ge);
        fGb[I * DK + c] = expf(gb);
        fWc[I * DK + c] = expf(sX[(Cp - 1) * DK + c] - ge);
        for (int J = 0; J < I; ++J)
          fOff[(I * NSM + J) * DK + c] = expf(gb - sX[(16 * J + 15) * DK + c]);
      }
      if (tid < DK) sgC[tid] = expf(sX[(Cp - 1) * DK + tid]);
      // scale K, Q to their sub-chunk's previous boundary and W to its own end
      for (int e = tid; e < Cp * DK; e += kThreads) {
        const int i = e / DK, c = e % DK, I = i / 16;
        const float gi = sX[i * DK + c];
        const float gb = (I == 0) ? 0.f : sX[(16 * I - 1) * DK + c];
        const float ge = sX[(16 * I + 15) * DK + c];
        const float fk = expf(gi - gb);
        sKt[c * CS + i] *= fk;
        sQt[c * CS + i] *= fk;
        sW[e] *= expf(ge - gi);
      }
      __syncthreads();
    }

    // ---- 4. Gram matrices L^T, P^T (token-minor transposed layout)
    {
      float* sWt = sX;  // W^T [DK][CS]; the per-channel g above is no longer needed
      // (KDN: g is dead after the scaling pass; scalar decay never used sX)
      for (int e = tid; e < Cp * DK; e += kThreads) {
        const int i = e / DK, c = e % DK;
        sWt[c * CS + i] = sW[e];
      }
      __syncthreads();
      const int nt = Cp / 4;
      if (tid < nt * nt) {
        const int ti = tid / nt, tj = tid % nt;
        float ak[4][4], aq[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) ak[x][y] = aq[x][y] = 0.f;
        if (tj <= ti) {
          const int I = (4 * ti) / 16, J = (4 * tj) / 16;
          const float* fo = (kdn && J < I) ? fOff + (I * NSM + J) * DK : nullptr;
          const float* fa = (kdn && J == I) ? fDa + I * DK : nullptr;
          const float* fb = (kdn && J == I) ? fDb + I * DK : nullptr;
          for (int c = 0; c < DK; ++c) {
            float4 k4 = *reinterpret_cast<const float4*>(sKt + c * CS + 4 * ti);
            float4 q4 = *reinterpret_cast<const float4*>(sQt + c * CS + 4 * ti);
            float4 w4 = *reinterpret_cast<const float4*>(sWt + c * CS + 4 * tj);
            if (kdn) {
              if (J < I) {
                const float f = fo[c];
                w4.x *= f; w4.y *= f; w4.z *= f; w4.w *= f;
              } else {
                const float fA = fa[c], fB = fb[c];
                k4.x *= fA; k4.y *= fA; k4.z *= fA; k4.w *= fA;
                q4.x *= fA; q4.y *= fA; q4.z *= fA; q4.w *= fA;
                w4.x *= fB; w4.y *= fB; w4.z *= fB; w4.w *= fB;
              }
            }
            const float kx[4] = {k4.x, k4.y, k4.z, k4.w};
            const float qx[4] = {q4.x, q4.y, q4.z, q4.w};
            const float wx[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
              for (int y = 0; y < 4; ++y) {
                ak[x][y] += kx[x] * wx[y];
                aq[x][y] += qx[x] * wx[y];
              }
          }
        }
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int j = 4 * tj + y;
          float lv[4], pv[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int i = 4 * ti + x;
            const float f = kdn ? 1.f : expf(sg[i] - sg[min(j, i)]);
            lv[x] = (j < i) ? ak[x][y] * f : 0.f;
            pv[x] = (j <= i) ? aq[x][y] * f : 0.f;
          }
          *reinterpret_cast<float4*>(sLt + j * CS + 4 * ti) = make_float4(lv[0], lv[1], lv[2], lv[3]);
          *reinterpret_cast<float4*>(sPt + j * CS + 4 * ti) = make_float4(pv[0], pv[1], pv[2], pv[3]);
        }
      }
      __syncthreads();
    }

    // ---- 5. operands of the carry: Gamma.K, Gamma.Q, exp(g_C - g_j).W, gamma_C
    if (kdn) {
      // K, Q carry exp(g_i - g_b(I)); multiply by exp(g_b(I)).  W carries
      // exp(g_e(J) - g_j); multiply by exp(g_C - g_e(J)) = gamma_C / exp(g_e(J)).
      for (int e = tid; e < Cp * DK; e += kThreads) {
        const int i = e / DK, c = e % DK, I = i / 16;
        const float gb = fGb[I * DK + c];
        sKt[c * CS + i] *= gb;
        sQt[c * CS + i] *= gb;
        sW[e] *= fWc[I * DK + c];
      }
    } else {
      const float gC = sg[Cp - 1];
      for (int e = tid; e < Cp * DK; e += kThreads) {
        const int i = e / DK, c = e % DK;
        const float gi = expf(sg[i]);
        sKt[c * CS + i] *= gi;
        sQt[c * CS + i] *= gi;
        sW[e] *= expf(gC - sg[i]);
      }
      if (tid == 0) sgC[0] = expf(gC);
    }

    // ---- 6. T = (I + L)^-1, stored transposed in sX: T(i,j) = sTt[j*CS + i]
    float* sTt = sX;
    for (int e = tid; e < Cp * CS; e += kThreads) sTt[e] = 0.f;
    __syncthreads();
    if (tid < NS * 16) {  // diagonal 16x16 blocks, one column per thread
      const int I = tid / 16, j = tid;  // global column
      float* col = sTt + j * CS;
      col[j] = 1.f;
      for (int i = j + 1; i < 16 * I + 16; ++i) {
        float s = 0.f;
        for (int l = j; l < i; ++l) s += sLt[l * CS + i] * col[l];
        col[i] = -s;
      }
    }
    __syncthreads();
    for (int d = 1; d < NS; ++d) {
      const int nb = NS - d;  // blocks (I, J = I - d), I = d .. NS-1
      for (int e = tid; e < nb * 256; e += kThreads) {  // X = sum_K L_IK T_KJ
        const int blk = e / 256, ii = (e / 16) % 16, jj = e % 16;
        const int I = d + blk, J = blk;
        const int gi = 16 * I + ii, gj = 16 * J + jj;
        float s = 0.f;
        for (int l = 16 * J; l < 16 * I; ++l) s += sLt[l * CS + gi] * sTt[gj * CS + l];
        sE[e] = s;
      }
      __syncthreads();
      for (int e = tid; e < nb * 256; e += kThreads) {  // T_IJ = -T_II X
        const int blk = e / 256, ii = (e / 16) % 16, jj = e % 16;
        const int I = d + blk, J = blk;
        const int gi = 16 * I + ii, gj = 16 * J + jj;
        float s = 0.f;
        for (int ll = 0; ll <= ii; ++ll) s += sTt[(16 * I + ll) * CS + gi] * sE[blk * 256 + ll * 16 + jj];
        sTt[gj * CS + gi] = -s;
      }
      __syncthreads();
    }

    // ---- 7. R = V - (Gamma.K) S   (rows i in 4-blocks, columns n in pairs)
    const int ti = tid / 16, tn = tid % 16;  // 16 x 16 thread grid: 4 rows x 2 cols each
    const bool rowok = 4 * ti < Cp;
    float acc[4][2];
    if (rowok) {
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
    }
    __syncthreads();
    // E = T R
    if (rowok) {
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
#pragma unroll
      for (int x = 0; x < 4; ++x)
        *reinterpret_cast<float2*>(sE + (4 * ti + x) * NV + 2 * tn) = make_float2(acc[x][0], acc[x][1]);
    }
    __syncthreads();
    // O = (Gamma.Q) S + P E  -> global
    if (rowok) {
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
        const float2 e2 = *reinterpret_cast<const float2*>(sE + j * NV + 2 * tn);
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
      const int tc = tid / 8, tv = tid % 8;  // 32 x 8 grid over (DK/4? ) channels, 4 columns each
      for (int cb = tc; cb < DK / 4; cb += 32) {
        float s4[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int c = 4 * cb + x;
          const float gcf = kdn ? sgC[c] : sgC[0];
          const float4 old = *reinterpret_cast<const float4*>(sS + c * NV + 4 * tv);
          s4[x][0] = gcf * old.x; s4[x][1] = gcf * old.y; s4[x][2] = gcf * old.z; s4[x][3] = gcf * old.w;
        }
        for (int j = 0; j < Cp; ++j) {
          const float4 w4 = *reinterpret_cast<const float4*>(sW + j * DK + 4 * cb);
          const float4 e4 = *reinterpret_cast<const float4*>(sE + j * NV + 4 * tv);
          const float wx[4] = {w4.x, w4.y, w4.z, w4.w};
          const float ex[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
          for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) s4[x][y] += wx[x] * ex[y];
        }
        __syncwarp();
#pragma unroll
        for (int x = 0; x < 4; ++x)
          *reinterpret_cast<float4*>(sS + (4 * cb + x) * NV + 4 * tv) =
              make_float4(s4[x][0], s4[x][1], s4[x][2], s4[x][3]);
      }
    }
  }
  __syncthreads();

  // final state and aux
  if (a.S) {
    for (int e = tid; e < DK * NV; e += kThreads) {
      const int c = e / NV, n = e % NV;
      const float v = sS[e];
      a.S[((long)bh * DK + c) * a.dv + tile * NV + n] = v;
      if (a.check_finite) bad |= !finite_f(v);
    }
  }
  if (a.aux && tile == 0 && tid < DK && (pgdn || kdn)) a.aux[(long)bh * DK + tid] = carry;
  if (bad) set_status(DR_ERR_NONFINITE);
}

}  // namespace

size_t simt_smem_bytes(int dk) {
  return sizeof(float) * (dk == 64 ? SimtSmem<64>::total : SimtSmem<128>::total);
}

cudaError_t launch_chunk_simt(const FwdArgs& a, int dtype, cudaStream_t st) {
  const int C = a.chunk > CM ? CM : a.chunk;
  const int grid = a.B * a.H * (a.dv / NV);
  const size_t smem = simt_smem_bytes(a.dk);
#define DR_SIMT(DK_, T_)                                                                   \
  if (a.dk == DK_) {                                                                       \
    cudaError_t err = cudaFuncSetAttribute(chunk_simt_kernel<DK_, T_>,                     \
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                                           (int)smem);                                     \
    if (err != cudaSuccess) return err;                                                    \
    chunk_simt_kernel<DK_, T_><<<grid, kThreads, smem, st>>>(a, C);                        \
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
