// chunk_bwd.cu — backward of the chunkwise forward for the scalar-decay write
// rules GDN (w = eta k^) and KLA (w = eta k^ / (||k^||^2 + eps)): bf16 q/k/v,
// fp32 gates and state, dk = dv = 128, chunk 64.  Gradients are fp32.
//
// Per chunk (local index i, j; KLA notes section 2.5, Eqs. (7)-(9), with the
// write matrix of the PDN notes section 2.6), with S_c the chunk-start state:
//
//   R = V - (Gamma.K^) S_c,  (I + L) E = R,  O = (Gamma.Q^) S_c + P E,
//   S_{c+1} = gamma S_c + Wbar^T E,  Wbar_j = e^{G - g_j} w_j,
//   L_ij = (k^_i . w_j) e^{g_i - g_j} (j < i),  P_ij = (q^_i . w_j) e^{g_i - g_j} (j <= i).
//
// Differentiating line by line, in reverse chunk order (dS = dL/dS_{c+1}):
//
//   dE = P^T dO + Wbar dS,  dR = (I + L)^-T dE = T^T dE,  dV = dR,
//   dS_c = gamma dS + (Gamma.Q^)^T dO - (Gamma.K^)^T dR,
//
// and, per chunk, the local gradients: dP = dO E^T (j <= i), dL = -dR E^T (j < i),
// dq^ = e^g (dO S_c^T) + (dP.D) W,  dk^ = -e^g (dR S_c^T) + (dL.D) W,
// dw = (dP.D)^T Q^ + (dL.D)^T K^ + e^{G-g} (E dS^T),  D_ij = e^{g_i - g_j},
// the decay terms (every entry X_ij . dX_ij of P and L adds to dg_i and takes
// from dg_j; e^g (dO S_c^T) . q^ and -e^g (dR S_c^T) . k^ add to dg_i;
// -e^{G-g_j} w_j . (E dS^T)_j to dg_j and its sum plus gamma <dS, S_c> to dG),
// then d log alpha_t = sum_{i >= t} dg_i with dG on the chunk's last token; the
// write gain (d beta = dw . k^, dk^ += beta dw; KLA: d eta = d beta / (s + eps),
// dk^ -= 2 d beta eta / (s + eps)^2 k^) and the L2 norms (dx = (dx^ - x^ (x^ . dx^)) / ||x||).
//
// PGDN's write vector w = eta B(A) . k^ comes from the key statistic A_t =
// alphaP A_{t-1} + betaP k^.k^ (PDN notes Eq. (9)): the chunk part collects
// dL/dw with the record's explicit write keys in place of eta k^, and
// `pgdn_gain_bwd` carries the statistic's adjoint dA backwards (dA_{t-1} =
// alphaP_t dA_t plus each token's own term through B: affine per chunk, so each
// chunk's map, a scan over the row's chunks, then every chunk at once), giving
// the gradients of k^, beta, alphaP, betaP, mu and A_0.
//
// Kernels (after the forward's prep and carry, which saves S_c and E per chunk):
//   bwd_carry   one CTA per (b, h, 64 columns of dv), chunks in reverse: dE, dR
//               (written as dV) and dS_c on tcgen05 (dL/dS in registers), saving
//               dS = dL/dS_{c+1} per chunk.
//   bwd_state   a persistent CTA per SM over the chunks: dO S_c^T, dR S_c^T, E dS^T,
//               dO E^T, dR E^T on tcgen05.
//   bwd_local   GDN, KLA, PGDN: a persistent CTA per SM, the Grams and the products
//               with W, Q^, K^ on tcgen05, then the decay terms, the gain and norm
//               backward, d log alpha; bwd_local_pc (per-channel decay): one CTA per
//               chunk, block rows on warp-level products.
#include "chain.cuh"
#include "dr_common.cuh"
#include "tc_common.cuh"

namespace dr {

cudaError_t launch_chunk_tc_split(const FwdArgs& a, void* workspace, cudaStream_t st);
cudaError_t launch_kdn_split(const FwdArgs& a, int dtype, void* workspace, cudaStream_t st);

namespace {

using namespace tc;

constexpr int kBwdThreads = 256;
constexpr uint64_t kWait = 2000000000ull;   // 2 s per bounded wait

int bwd_sm_count() {
  static int count[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!count[dev]) cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev);
  return count[dev];
}
// The workspace: the forward's chunk records, then per record the saved state, E,
// dS_{c+1}, E dS^T, dO E^T, dR E^T and gamma <dS, S_c> (one array each, record-major)
constexpr size_t kRecF = 66560;                 // the forward's GDN / KLA chunk record (tc_split)
constexpr size_t kRecFP = 101376;               // the forward's PGDN chunk record
constexpr uint32_t rWF = 66560, rAuxF = 99328;    // PGDN record: write keys, statistic
// the forward record's vectors (floats after rVecF): e^g qn, e^{G-g} c, gamma, e^g cr
constexpr size_t rVecF = 65536;
constexpr uint32_t rTF = 0, rPF = 49152;
// the per-channel-decay record (tensor-core prep): W'^T [128 c][64 j] hi | lo, and
// (Gamma.Q), Wbar as [64 tok][128] (two 64-column blocks) hi | lo; gamma_C per
// channel at float 128 of the vectors; the gain state at the chunk start
constexpr size_t kRecPC = 135168;
constexpr uint32_t rWpPC = 16384, rQPC = 66560, rWbPC = 99328, rP0PC = 134144;

// workspace layouts: scalar decay (GDN, KLA), PGDN (+ dL/dw, key norms, d mu
// parts), per-channel decay (KDA: + the forward's write vectors, dG per channel),
// Diagonal KDN (+ dL/dw)
// (BW_GAIN: Diagonal KDN, PKDA, isotropic KDN, whose gain kernels take dL/dw, each
// chunk's affine map of the gain adjoint and its value at the chunk's end; PKDA
// also each chunk's part of dL/dmu)
enum { BW_SCALAR = 0, BW_PGDN = 1, BW_PC = 2, BW_GAIN = 3 };
inline int bwd_mode(int variant) {
  if (variant == DR_PGDN) return BW_PGDN;
  if (variant == DR_KDA) return BW_PC;
  if (variant == DR_KDN || variant == DR_PKDA || variant == DR_IKDN) return BW_GAIN;
  return BW_SCALAR;
}

struct BwdWs {
  uint8_t* rec;   // [n] x kRecF
  // S, E and dS are stored as [32 column quads][rows][4] per chunk: the carries
  // (one thread per row) write a warp's rows as one 512-byte piece
  float* S;       // [n][32][128][4]  S_c
  float* E;       // [n][32][64][4]   E
  float* dS;      // [n][32][128][4]  dL/dS_{c+1}
  float* XW;      // [n][64][128]   E dS^T
  float* dP;      // [n][64][64]    dO E^T
  float* dL;      // [n][64][64]    dR E^T
  float* SS;      // [n]            gamma <dS, S_c>  (per-channel decay: [n][128])
  float* DW;      // PGDN, KDN [n][64][128]  dL/dw
  float* CR;      // PGDN [n][64]       key-norm factors
  float* MU;      // PGDN / PKDA [n]     each chunk's part of dL/dmu
  float* Wf;      // per-channel decay [n][64][128]  the forward's write vectors
  float* GM;      // gain variants and PGDN [n][2][128]  each chunk's affine map of the gain adjoint
  float* GE;      // gain variants and PGDN [n][128]     the gain adjoint at each chunk's end
  size_t recb;    // bytes of one forward record
};

// Every array starts on a 256-byte boundary (the 16-byte copies need 16).
inline size_t al256(size_t bytes) { return (bytes + 255) / 256 * 256; }

// Lays the arrays out from `base` (null: only the size), returns the bytes used.
size_t bwd_layout(void* base, long n, int rows, int mode, BwdWs* w) {
  const bool pgdn = mode == BW_PGDN, pc = mode >= BW_PC, gain = mode == BW_GAIN;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* q = p ? p + off : nullptr;
    off += al256(bytes);
    return q;
  };
  BwdWs v{};
  v.recb = pgdn ? kRecFP : (pc ? kRecPC : kRecF);
  // (per-channel decay: the forward's hand-over flags follow its records)
  v.rec = take((size_t)n * v.recb + (pc ? chain_bytes(n) : 0));
  v.S = reinterpret_cast<float*>(take((size_t)n * 16384 * 4));
  v.E = reinterpret_cast<float*>(take((size_t)n * 8192 * 4));
  v.dS = reinterpret_cast<float*>(take((size_t)n * 16384 * 4));
  v.XW = reinterpret_cast<float*>(take((size_t)n * 8192 * 4));
  v.dP = reinterpret_cast<float*>(take((size_t)n * 4096 * 4));
  v.dL = reinterpret_cast<float*>(take((size_t)n * 4096 * 4));
  v.SS = reinterpret_cast<float*>(take((size_t)n * (pc ? 128 : 1) * 4));
  if (pgdn || gain) v.DW = reinterpret_cast<float*>(take((size_t)n * 8192 * 4));
  if (pgdn) v.CR = reinterpret_cast<float*>(take((size_t)n * 64 * 4));
  if (pgdn || gain) v.MU = reinterpret_cast<float*>(take((size_t)n * 4));
  if (pc) v.Wf = reinterpret_cast<float*>(take((size_t)n * 8192 * 4));
  if (pgdn || gain) {
    v.GM = reinterpret_cast<float*>(take((size_t)n * 256 * 4));
    v.GE = reinterpret_cast<float*>(take((size_t)n * 128 * 4));
  }
  if (w) *w = v;
  return off;
}

BwdWs bwd_ws(void* base, long n, int rows, int mode) {
  BwdWs w;
  bwd_layout(base, n, rows, mode, &w);
  return w;
}

// ---- warp-level tensor-core products on fp32 shared-memory operands: each value
// split into bf16 hi + lo (x = hi + lo to ~2^-17 of |x|) and three m16n8k16
// products hi.hi + lo.hi + hi.lo, accumulated in fp32.
// A element (m, k) = TA ? A[k lda + m] : A[m lda + k];
// B element (k, n) = TB ? B[n ldb + k] : B[k ldb + n].
// NT tiles side by side: D_j (16 x 8) += op(A)[16 x 8K] op(B)[8K x 8] at B columns
// 8 j .. 8 j + 8 (K = KSTEPS x 8, KSTEPS even).  The A fragment is split once per
// k-step for all NT tiles, and each tile keeps its three products in separate
// accumulators, so 3 NT independent chains are in flight per warp.  The fragment's
// k slots (2t, 2t+1, 2t+8, 2t+9) of lane (g, t) hold k0 + t + (0, 4, 8, 12) in A
// and B alike (a sum over k is order-free), so a lane reads the same
// bank-conflict-free addresses as an 8-wide step per 8 of K.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32"
      " {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// (x0, x1) -> packed bf16x2 hi = bf16(x) and lo = bf16(x - hi)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x0, x1);
  lo = pack_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xFFFF0000u));
}

template <int NT, int KSTEPS, bool TA, bool TB>
__device__ __forceinline__ void mm3x(float (&d)[NT][4], const float* A, int lda, const float* B,
                                     int ldb, int lane) {
  static_assert(KSTEPS % 2 == 0, "K must be a multiple of 16");
  const int g = lane >> 2, t = lane & 3;
  float c1[NT][4], c2[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) c1[j][i] = c2[j][i] = 0.f;
  auto ae = [&](int m, int k) { return TA ? A[k * lda + m] : A[m * lda + k]; };
  auto be = [&](int k, int n) { return TB ? B[n * ldb + k] : B[k * ldb + n]; };
#pragma unroll 2
  for (int ks = 0; ks < KSTEPS / 2; ++ks) {
    const int k0 = 16 * ks + t;
    uint32_t ah[4], al[4];
    split2(ae(g, k0), ae(g, k0 + 4), ah[0], al[0]);
    split2(ae(g + 8, k0), ae(g + 8, k0 + 4), ah[1], al[1]);
    split2(ae(g, k0 + 8), ae(g, k0 + 12), ah[2], al[2]);
    split2(ae(g + 8, k0 + 8), ae(g + 8, k0 + 12), ah[3], al[3]);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int n = 8 * j + g;
      uint32_t bh[2], bl[2];
      split2(be(k0, n), be(k0 + 4, n), bh[0], bl[0]);
      split2(be(k0 + 8, n), be(k0 + 12, n), bh[1], bl[1]);
      mma16816(d[j], ah, bh);
      mma16816(c1[j], al, bh);
      mma16816(c2[j], ah, bl);
    }
  }
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) d[j][i] += c1[j][i] + c2[j][i];
}

// fragment element e of a 16 x 8 tile: row and column within the tile
__device__ __forceinline__ int frag_row(int lane, int e) { return (lane >> 2) + ((e >> 1) << 3); }
__device__ __forceinline__ int frag_col(int lane, int e) { return 2 * (lane & 3) + (e & 1); }

// 16-byte asynchronous copy global -> shared; src_bytes 0 fills zeros
__device__ __forceinline__ void cpa16(void* dst, const void* src, int src_bytes = 16) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(umma::smem_u32(dst)),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cpa_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ long tok(const FwdArgs& a, int b, int t, int h) {
  return ((long)b * a.T + t) * a.H + h;
}

struct BwdArgs {
  const void* d_out;         // [B,T,H,dv] bf16
  const float* dS_final;     // [B,H,dk,dv] or null
  float* dq;                 // [B,T,H,dk] fp32
  float* dk;
  float* dv;                 // [B,T,H,dv]
  float* dla;                // [B,T,H]
  float* deta;               // [B,T,H]
  float* dS0;                // [B,H,dk,dv] or null
  float* daP;                // PGDN [B,T,H]
  float* dbP;                // PGDN [B,T,H]
  float* dmu;                // PGDN [H]
  float* daux0;              // PGDN / KDN [B,H,dk] or null
  const float* daux_T;       // PGDN / KDN [B,H,dk] or null
  float* domega;             // KDN [B,T,H,dk]
  float* dr;                 // KDN [B,T,H]
  BwdWs w;
};

// ================================================================= bwd_carry_tc
// The reverse carry of the scalar-decay variants (GDN, KLA) on tcgen05: one CTA
// per (b, h, dv half), chunks in reverse, dL/dS (128 x 64 fp32) in registers.
// Per chunk, with the record's P and T images (bf16 hi | lo), the raw K and Q rows
// (bf16, exact) and the row vectors sq = e^g qn, u = e^{G-g} c, sk = e^g cr, gamma:
//   G1  D1 = [P_hi ; P_lo]^T dO                 (A MN-major, M = 128)
//   G2  D2 = [K ; Q] [dS_hi | dS_lo]            (the Q rows are not used)
//   G4a D4 = Q^T [dO'_hi | dO'_lo],  dO' = sq . dO
//   dE  = D1 (both halves) + u . (K dS_hi + K dS_lo)
//   G3  D3 = [T_hi ; T_lo]^T [dE_hi | dE_lo],    dR = dV = hi.hi + hi.lo + lo.hi
//   G4b D4 -= K^T [dR'_hi | dR'_lo],  dR' = sk . dR
//   dS <- gamma dS + D4 (both halves)
// G1, G2 and G4a are issued together; the chain is G2 -> dE -> G3 -> dR -> G4b -> dS.
// The M = 128 halves of D1 and D3 meet through shared memory (the quadrant of lanes
// 64-127 hands its rows to the quadrant of lanes 0-63).  The next chunk's operands
// arrive by asynchronous copies under the current chunk's dR and dS steps.
constexpr uint32_t kcKQ = 0;            // 2 buffers x [K kb0 | Q kb0 | K kb1 | Q kb1] (8 KB each)
constexpr uint32_t kcP = 65536;         // P hi | P lo (the record's images)
constexpr uint32_t kcT = kcP + 16384;   // T hi | T lo
constexpr uint32_t kcO = kcT + 16384;   // dO [64 j][64 n] bf16 (MN-major B)
constexpr uint32_t kcVec = kcO + 8192;  // 2 x fp32 [256]: sq [0, 64), u [64, 128), gamma, sk [192, 256)
constexpr uint32_t kcS = kcVec + 2048;  // dS hi | dS lo: [128 c][64 n] each (16 KB)
constexpr uint32_t kcE = kcS + 32768;   // dE hi | dE lo [64][64] (8 KB each); then the dR exchange
constexpr uint32_t kcR = kcE + 16384;   // dR' hi | lo; before it, the dE exchange
constexpr uint32_t kcO2 = kcR + 16384;  // dO' hi | lo
constexpr uint32_t kcW = kcO2 + 16384;  // PGDN: the record's write keys as [hi kb0 | lo kb0 | hi kb1 | lo kb1]
constexpr uint32_t kCarryTcSmem = kcO2 + 16384 + 1024;
constexpr uint32_t kCarryTcSmemPG = kcW + 32768 + 1024;
constexpr uint32_t tcD1 = 0, tcD2 = 64, tcD3 = 192, tcD4 = 320, kCarryTcTmem = 512;
constexpr uint32_t I_C1 = idesc_bf16(128, 64, 1, 1);
constexpr uint32_t I_C2 = idesc_bf16(128, 128, 0, 1);
constexpr uint32_t I_C3 = idesc_bf16(128, 128, 1, 1);
constexpr uint32_t I_C4N = idesc_bf16(128, 128, 1, 1, 1);

__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// 32 fp32 values of one row -> bf16 hi / lo at columns col0 .. col0 + 31 of a
// 128B-swizzled image with 128-byte rows (hi at base, lo at base + lo_off)
__device__ __forceinline__ void put_row32(uint8_t* base, uint32_t lo_off, int row, int col0,
                                          const float (&v)[32]) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = v[8 * m + e];
    uint4 hi, lo;
    split8(x, hi, lo);
    const uint32_t o = sw128_offset(row, col0 + 8 * m);
    *reinterpret_cast<uint4*>(base + o) = hi;
    *reinterpret_cast<uint4*>(base + o + lo_off) = lo;
  }
}

// PG (PGDN): W is explicit (the record's write keys, hi / lo), so G2 takes
// [W_hi ; W_lo] in place of [K ; Q] and dE adds u . (hi.hi + hi.lo + lo.hi).
template <bool PG>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_carry_tc_kernel(FwdArgs a, BwdArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bars[3];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, hc = warp >> 2, trow = 32 * q4 + lane;   // TMEM lane = trow
  const int bh = blockIdx.x >> 1, cb = blockIdx.x & 1, n0 = 64 * cb;
  const int b = bh / a.H, h = bh % a.H;
  const int NC = (a.T + 63) / 64;
  const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(g.d_out);
  float* xch = reinterpret_cast<float*>(sm + kcR);    // dE exchange [64][64], XOR-swizzled
  float* xch2 = reinterpret_cast<float*>(sm + kcE);   // dR exchange

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, kCarryTcTmem);
  // chunk c's operands: P, T, dO, vectors, and K / Q into buffer kq (one commit group)
  auto load = [&](int c, int kq) {
    const uint8_t* rec = g.w.rec + ((size_t)bh * NC + c) * g.w.recb;
    const int t0 = 64 * c, Cc = min(64, a.T - t0);
    for (int e = tid; e < 2048; e += kBwdThreads) {   // P, T images: 16 KB each
      const uint32_t o = 16 * e;
      cpa16(sm + (o < 16384 ? kcP + o : kcT + o - 16384),
            rec + (o < 16384 ? rPF + o : rTF + o - 16384));
    }
    for (int e = tid; e < 64 * 8; e += kBwdThreads) {   // dO rows: 8 16-byte pieces of 64 columns
      const int j = e >> 3, p = e & 7;
      const bool live = j < Cc;
      cpa16(sm + kcO + sw128_offset(j, 8 * p), dO + tok(a, b, t0 + (live ? j : 0), h) * 128 + n0 + 8 * p,
            live ? 16 : 0);
    }
    for (int e = tid; e < 64 * 32; e += kBwdThreads) {   // K and Q rows: 16 pieces of 128 channels each
      const int j = e >> 5, isq = (e >> 4) & 1, p = e & 15, kb = p >> 3;
      const bool live = j < Cc;
      cpa16(sm + kcKQ + kq * 32768 + kb * 16384 + isq * 8192 + sw128_offset(j, 8 * (p & 7)),
            (isq ? Q : K) + tok(a, b, t0 + (live ? j : 0), h) * 128 + 8 * p, live ? 16 : 0);
    }
    for (int e = tid; e < 64; e += kBwdThreads) {   // vectors: sq, u, gamma at 128, sk at 192
      const float* rv = reinterpret_cast<const float*>(rec + rVecF);
      cpa16(sm + kcVec + (c & 1) * 1024 + 16 * e, rv + 4 * e);
    }
    for (int e = tid; PG && e < 2048; e += kBwdThreads) {   // PGDN write keys, rearranged per k-block
      const uint32_t o = 16 * e, piece = o >> 13;
      cpa16(sm + kcW + (piece & 1) * 16384 + (piece >> 1) * 8192 + (o & 8191), rec + rWF + o);
    }
    cpa_commit();
  };
  // dS = dL/dS_T (or 0): rows c = trow, columns 32 hc .. + 31 of this half
  float ds[32];
#pragma unroll
  for (int e = 0; e < 32; ++e)
    ds[e] = g.dS_final ? g.dS_final[((size_t)bh * 128 + trow) * 128 + n0 + 32 * hc + e] : 0.f;
  load(NC - 1, (NC - 1) & 1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
  int nA = 0, nB = 0, nC = 0;

  for (int c = NC - 1; c >= 0; --c) {
    const int it = NC - 1 - c, kq = c & 1;
    const size_t ri = (size_t)bh * NC + c;
    const int t0 = 64 * c, Cc = min(64, a.T - t0);
    // dL/dS_{c+1} for the local gradients; its hi / lo image for G2
    {
      float* sv = g.w.dS + ri * 16384 + 4 * trow;
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4*>(sv + (size_t)((n0 + 32 * hc + e) >> 2) * 512) =
            make_float4(ds[e], ds[e + 1], ds[e + 2], ds[e + 3]);
      put_row32(sm + kcS, 16384, trow, 32 * hc, ds);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();   // chunk c's operands landed (every thread's copies)
    const float* vec = reinterpret_cast<const float*>(sm + kcVec + (c & 1) * 1024);
    // dO' = sq . dO (hi / lo): row j, 8 columns per unit
    for (int e = tid; e < 64 * 8; e += kBwdThreads) {
      const int j = e >> 3, p = e & 7;
      const uint32_t o = sw128_offset(j, 8 * p);
      float x[8];
      unpack8(*reinterpret_cast<const uint4*>(sm + kcO + o), x);
      const float s = vec[j];
#pragma unroll
      for (int f = 0; f < 8; ++f) x[f] *= s;
      uint4 hi, lo;
      split8(x, hi, lo);
      *reinterpret_cast<uint4*>(sm + kcO2 + o) = hi;
      *reinterpret_cast<uint4*>(sm + kcO2 + 8192 + o) = lo;
    }
    fence_proxy_async();
    __syncthreads();
    const uint32_t kqb = smem_u32(sm + kcKQ + kq * 32768);
    if (tid == 0) {
      tc_fence_after();
      const uint32_t pb = smem_u32(sm + kcP), ob = smem_u32(sm + kcO), o2 = smem_u32(sm + kcO2);
      const uint32_t sb = smem_u32(sm + kcS);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)   // G1: K = 64 tokens
        mma_bf16(tmem + tcD1, desc_sw128(pb + ks * 2048, 8192, 1024), desc_sw128(ob + ks * 2048, 8192, 1024),
                 I_C1, ks > 0);
      const uint32_t ab = PG ? smem_u32(sm + kcW) : kqb;   // [W_hi ; W_lo] or [K ; Q]
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)   // G2: K = 128 channels
        mma_bf16(tmem + tcD2, desc_sw128(ab + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                 desc_sw128(sb + ks * 2048, 16384, 1024), I_C2, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)   // G4a: K = 64 tokens, A = Q^T (MN-major)
        mma_bf16(tmem + tcD4, desc_sw128(kqb + 8192 + ks * 2048, 16384, 1024),
                 desc_sw128(o2 + ks * 2048, 8192, 1024), I_C3, ks > 0);
      mma_commit(&bars[0]);
      ++nA;
    }
    if (!mbar_wait(&bars[0], it & 1, kWait)) s_abort = 1;
    __syncthreads();
    if (s_abort) break;
    tc_fence_after();
    // ---- dE: lanes 64-127 hand D1's lo rows (PGDN: and u . W_lo dS_hi) over; lanes
    //      0-63 sum and write dE hi / lo
    if (trow >= 64) {
      float v[32], w[32];
      tmem_ld16(tl + tcD1 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tcD1 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      if (PG) {
        tmem_ld16(tl + tcD2 + 32 * hc, *reinterpret_cast<float(*)[16]>(w));
        tmem_ld16(tl + tcD2 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(w + 16));
      }
      tmem_ld_wait();
      const int i = trow - 64;
      const float u = PG ? vec[64 + i] : 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) xch[i * 64 + ((32 * hc + e) ^ (i & 31))] = PG ? fmaf(u, w[e], v[e]) : v[e];
    }
    __syncthreads();
    if (trow < 64) {
      float v[32], k0[32], k1[32];
      tmem_ld16(tl + tcD1 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tcD1 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      tmem_ld16(tl + tcD2 + 32 * hc, *reinterpret_cast<float(*)[16]>(k0));
      tmem_ld16(tl + tcD2 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(k0 + 16));
      tmem_ld16(tl + tcD2 + 64 + 32 * hc, *reinterpret_cast<float(*)[16]>(k1));
      tmem_ld16(tl + tcD2 + 64 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(k1 + 16));
      tmem_ld_wait();
      const int i = trow;
      const float u = vec[64 + i];
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] += xch[i * 64 + ((32 * hc + e) ^ (i & 31))] + u * (k0[e] + k1[e]);
      put_row32(sm + kcE, 8192, i, 32 * hc, v);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {   // G3: dR = T^T dE
      tc_fence_after();
      const uint32_t tb = smem_u32(sm + kcT), eb = smem_u32(sm + kcE);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + tcD3, desc_sw128(tb + ks * 2048, 8192, 1024), desc_sw128(eb + ks * 2048, 8192, 1024),
                 I_C3, ks > 0);
      mma_commit(&bars[1]);
      ++nB;
    }
    if (!mbar_wait(&bars[1], it & 1, kWait)) s_abort = 1;
    __syncthreads();
    if (s_abort) break;
    tc_fence_after();
    // the next chunk's operands (G1, G3 are done with P, T, dO; the other K/Q buffer
    // was last read by the previous chunk)
    if (c > 0) load(c - 1, (c - 1) & 1);
    // ---- dR = T_hi^T dE_hi + T_hi^T dE_lo + T_lo^T dE_hi; dV out; dR' = sk . dR
    if (trow >= 64) {
      float v[32];
      tmem_ld16(tl + tcD3 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tcD3 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      tmem_ld_wait();
      const int i = trow - 64;
#pragma unroll
      for (int e = 0; e < 32; ++e) xch2[i * 64 + ((32 * hc + e) ^ (i & 31))] = v[e];
    }
    __syncthreads();
    if (trow < 64) {
      float v[32], w[32];
      tmem_ld16(tl + tcD3 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tcD3 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      tmem_ld16(tl + tcD3 + 64 + 32 * hc, *reinterpret_cast<float(*)[16]>(w));
      tmem_ld16(tl + tcD3 + 64 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(w + 16));
      tmem_ld_wait();
      const int i = trow;
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] += w[e] + xch2[i * 64 + ((32 * hc + e) ^ (i & 31))];
      if (i < Cc) {
        float* dv = g.dv + tok(a, b, t0 + i, h) * 128 + n0 + 32 * hc;
#pragma unroll
        for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4*>(dv + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
      const float sk = vec[192 + i];
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] *= sk;
      put_row32(sm + kcR, 8192, i, 32 * hc, v);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {   // G4b: D4 -= K^T dR'
      tc_fence_after();
      const uint32_t rb = smem_u32(sm + kcR);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + tcD4, desc_sw128(kqb + ks * 2048, 16384, 1024), desc_sw128(rb + ks * 2048, 8192, 1024),
                 I_C4N, true);
      mma_commit(&bars[2]);
      ++nC;
    }
    if (!mbar_wait(&bars[2], it & 1, kWait)) s_abort = 1;
    __syncthreads();
    if (s_abort) break;
    tc_fence_after();
    {   // ---- dS_c = gamma dS + D4 (both halves); lane = state row
      float v[32], w[32];
      tmem_ld16(tl + tcD4 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tcD4 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      tmem_ld16(tl + tcD4 + 64 + 32 * hc, *reinterpret_cast<float(*)[16]>(w));
      tmem_ld16(tl + tcD4 + 64 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(w + 16));
      tmem_ld_wait();
      const float gam = vec[128];
#pragma unroll
      for (int e = 0; e < 32; ++e) ds[e] = fmaf(gam, ds[e], v[e] + w[e]);
    }
    tc_fence_before();
    __syncthreads();   // every buffer of this chunk read before the next one's writes
  }
  if (s_abort) {
    if (tid == 0) {   // drain: no MMA may still write TMEM after the dealloc
      set_status(DR_ERR_TIMEOUT);
      if (nA > 0) mbar_wait(&bars[0], (nA - 1) & 1, kWait / 4);
      if (nB > 0) mbar_wait(&bars[1], (nB - 1) & 1, kWait / 4);
      if (nC > 0) mbar_wait(&bars[2], (nC - 1) & 1, kWait / 4);
    }
  } else if (g.dS0) {
    float* d0 = g.dS0 + ((size_t)bh * 128 + trow) * 128 + n0 + 32 * hc;
#pragma unroll
    for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4*>(d0 + e) = make_float4(ds[e], ds[e + 1], ds[e + 2], ds[e + 3]);
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kCarryTcTmem);
}

// The per-channel-decay variants' reverse carry on tcgen05 (KDA, Diagonal /
// isotropic KDN, PKDA): the record holds (Gamma.Q), Wbar and W'^T as bf16 hi / lo
// images and gamma per state row, and dS_c = gamma . dS + (Gamma.Q)^T dO - W'^T dE
// ((Gamma.K)^T dR = (T Gamma.K)^T dE), so the dS step needs dE only:
//   G1  D1 = [P_hi ; P_lo]^T dO,   G2  D2 = [Wbar_hi ; Wbar_lo] [dS_hi | dS_lo]
//   dE  = D1 (both halves) + hi.hi + hi.lo + lo.hi of D2
//   G3  D3 = [T_hi ; T_lo]^T [dE_hi | dE_lo]       (dR = dV)
//   G4  D4 = -W'^T_hi [dE_hi | dE_lo] - W'^T_lo dE_hi + (Gamma.Q)^T_hi dO + (Gamma.Q)^T_lo dO
// G3 and G4 are issued together once dE is written.
constexpr uint32_t kpW = 0;             // Wbar as [hi kb0 | lo kb0 | hi kb1 | lo kb1] (8 KB each)
constexpr uint32_t kpQ = 32768;         // (Gamma.Q) hi kb0 | hi kb1 | lo kb0 | lo kb1 (the record's order)
constexpr uint32_t kpWp = 65536;        // W'^T hi | lo [128 c][64 j]
constexpr uint32_t kpP = 98304;         // P hi | lo
constexpr uint32_t kpT = 114688;        // T hi | lo
constexpr uint32_t kpO = 131072;        // 2 x dO [64 j][64 n] bf16
constexpr uint32_t kpVec = 147456;      // 2 x fp32 [256]: gamma per state row at [128, 256)
constexpr uint32_t kpS = 149504;        // dS hi | lo [128 c][64 n]
constexpr uint32_t kpE = kpS + 32768;   // dE hi | lo; then the dR exchange
constexpr uint32_t kpX = kpE + 16384;   // the dE exchange [64][64] fp32
constexpr uint32_t kCarryPcSmem = kpX + 16384 + 1024;
constexpr uint32_t I_P4N = idesc_bf16(128, 128, 0, 1, 1);
constexpr uint32_t I_P4N64 = idesc_bf16(128, 64, 0, 1, 1);

__global__ void __launch_bounds__(kBwdThreads, 1) bwd_carry_tc_pc_kernel(FwdArgs a, BwdArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bars[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, hc = warp >> 2, trow = 32 * q4 + lane;
  const int bh = blockIdx.x >> 1, cb = blockIdx.x & 1, n0 = 64 * cb;
  const int b = bh / a.H, h = bh % a.H;
  const int NC = (a.T + 63) / 64;
  const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(g.d_out);
  float* xch = reinterpret_cast<float*>(sm + kpX);
  float* xch2 = reinterpret_cast<float*>(sm + kpE);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, kCarryTcTmem);
  // chunk c's first group: P, Wbar, dO (slot c & 1), vectors (slot c & 1)
  auto load_a = [&](int c) {
    const uint8_t* rec = g.w.rec + ((size_t)bh * NC + c) * g.w.recb;
    const int t0 = 64 * c, Cc = min(64, a.T - t0);
    for (int e = tid; e < 1024; e += kBwdThreads) {   // P (16 KB)
      cpa16(sm + kpP + 16 * e, rec + rPF + 16 * e);
    }
    for (int e = tid; e < 2048; e += kBwdThreads) {   // Wbar (32 KB), rearranged per k-block
      const uint32_t o = 16 * e, piece = o >> 13;
      cpa16(sm + kpW + (piece & 1) * 16384 + (piece >> 1) * 8192 + (o & 8191), rec + rWbPC + o);
    }
    for (int e = tid; e < 64 * 8; e += kBwdThreads) {
      const int j = e >> 3, p = e & 7;
      const bool live = j < Cc;
      cpa16(sm + kpO + (c & 1) * 8192 + sw128_offset(j, 8 * p),
            dO + tok(a, b, t0 + (live ? j : 0), h) * 128 + n0 + 8 * p, live ? 16 : 0);
    }
    for (int e = tid; e < 64; e += kBwdThreads)
      cpa16(sm + kpVec + (c & 1) * 1024 + 16 * e, rec + rVecF + 16 * e);
    cpa_commit();
  };
  // the second group: (Gamma.Q), T, W'^T
  auto load_b = [&](int c) {
    const uint8_t* rec = g.w.rec + ((size_t)bh * NC + c) * g.w.recb;
    for (int e = tid; e < 2048; e += kBwdThreads) cpa16(sm + kpQ + 16 * e, rec + rQPC + 16 * e);
    for (int e = tid; e < 1024; e += kBwdThreads) cpa16(sm + kpT + 16 * e, rec + rTF + 16 * e);
    for (int e = tid; e < 2048; e += kBwdThreads) cpa16(sm + kpWp + 16 * e, rec + rWpPC + 16 * e);
    cpa_commit();
  };
  float ds[32];
#pragma unroll
  for (int e = 0; e < 32; ++e)
    ds[e] = g.dS_final ? g.dS_final[((size_t)bh * 128 + trow) * 128 + n0 + 32 * hc + e] : 0.f;
  load_a(NC - 1);
  load_b(NC - 1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
  int nA = 0, nB = 0;

  for (int c = NC - 1; c >= 0; --c) {
    const int it = NC - 1 - c;
    const size_t ri = (size_t)bh * NC + c;
    const int t0 = 64 * c, Cc = min(64, a.T - t0);
    {
      float* sv = g.w.dS + ri * 16384 + 4 * trow;
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4*>(sv + (size_t)((n0 + 32 * hc + e) >> 2) * 512) =
            make_float4(ds[e], ds[e + 1], ds[e + 2], ds[e + 3]);
      put_row32(sm + kpS, 16384, trow, 32 * hc, ds);
    }
    asm volatile("cp.async.wait_group 1;" ::: "memory");   // this chunk's first group
    fence_proxy_async();
    __syncthreads();
    const float* vec = reinterpret_cast<const float*>(sm + kpVec + (c & 1) * 1024);
    const uint32_t ob = smem_u32(sm + kpO + (c & 1) * 8192);
    if (tid == 0) {
      tc_fence_after();
      const uint32_t pb = smem_u32(sm + kpP), wb = smem_u32(sm + kpW), sb = smem_u32(sm + kpS);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)   // G1
        mma_bf16(tmem + tcD1, desc_sw128(pb + ks * 2048, 8192, 1024), desc_sw128(ob + ks * 2048, 8192, 1024),
                 I_C1, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)   // G2
        mma_bf16(tmem + tcD2, desc_sw128(wb + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                 desc_sw128(sb + ks * 2048, 16384, 1024), I_C2, ks > 0);
      mma_commit(&bars[0]);
      ++nA;
    }
    if (!mbar_wait(&bars[0], it & 1, kWait)) s_abort = 1;
    __syncthreads();
    if (s_abort) break;
    tc_fence_after();
    if (c > 0) load_a(c - 1);   // P and Wbar are read; dO and the vectors take the other slot
    // ---- dE
    if (trow >= 64) {
      float v[32], w[32];
      tmem_ld16(tl + tcD1 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tcD1 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      tmem_ld16(tl + tcD2 + 32 * hc, *reinterpret_cast<float(*)[16]>(w));
      tmem_ld16(tl + tcD2 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(w + 16));
      tmem_ld_wait();
      const int i = trow - 64;
#pragma unroll
      for (int e = 0; e < 32; ++e) xch[i * 64 + ((32 * hc + e) ^ (i & 31))] = v[e] + w[e];
    }
    __syncthreads();
    if (trow < 64) {
      float v[32], k0[32], k1[32];
      tmem_ld16(tl + tcD1 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tcD1 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      tmem_ld16(tl + tcD2 + 32 * hc, *reinterpret_cast<float(*)[16]>(k0));
      tmem_ld16(tl + tcD2 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(k0 + 16));
      tmem_ld16(tl + tcD2 + 64 + 32 * hc, *reinterpret_cast<float(*)[16]>(k1));
      tmem_ld16(tl + tcD2 + 64 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(k1 + 16));
      tmem_ld_wait();
      const int i = trow;
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] += k0[e] + k1[e] + xch[i * 64 + ((32 * hc + e) ^ (i & 31))];
      put_row32(sm + kpE, 8192, i, 32 * hc, v);
    }
    if (c > 0)   // this chunk's second group (the next chunk's first one may still fly)
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    else
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {   // G3 and G4
      tc_fence_after();
      const uint32_t tb = smem_u32(sm + kpT), eb = smem_u32(sm + kpE), wp = smem_u32(sm + kpWp);
      const uint32_t qb = smem_u32(sm + kpQ);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + tcD3, desc_sw128(tb + ks * 2048, 8192, 1024), desc_sw128(eb + ks * 2048, 8192, 1024),
                 I_C3, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + tcD4, desc_sw128(wp + ks * 32, 16, 1024), desc_sw128(eb + ks * 2048, 8192, 1024),
                 I_P4N, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + tcD4, desc_sw128(wp + 16384 + ks * 32, 16, 1024), desc_sw128(eb + ks * 2048, 8192, 1024),
                 I_P4N64, true);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tmem + tcD4, desc_sw128(qb + ks * 2048, 8192, 1024), desc_sw128(ob + ks * 2048, 8192, 1024),
                 I_C1, true);
        mma_bf16(tmem + tcD4, desc_sw128(qb + 16384 + ks * 2048, 8192, 1024),
                 desc_sw128(ob + ks * 2048, 8192, 1024), I_C1, true);
      }
      mma_commit(&bars[1]);
      ++nB;
    }
    if (!mbar_wait(&bars[1], it & 1, kWait)) s_abort = 1;
    __syncthreads();
    if (s_abort) break;
    tc_fence_after();
    if (c > 0) load_b(c - 1);   // (Gamma.Q), T and W'^T are read
    // ---- dR = dV: lanes 64-127 hand over T_lo^T dE_hi
    if (trow >= 64) {
      float v[32];
      tmem_ld16(tl + tcD3 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tcD3 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      tmem_ld_wait();
      const int i = trow - 64;
#pragma unroll
      for (int e = 0; e < 32; ++e) xch2[i * 64 + ((32 * hc + e) ^ (i & 31))] = v[e];
    }
    {   // ---- dS_c = gamma . dS + D4 (both halves); lane = state row
      float v[32], w[32];
      tmem_ld16(tl + tcD4 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tcD4 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      tmem_ld16(tl + tcD4 + 64 + 32 * hc, *reinterpret_cast<float(*)[16]>(w));
      tmem_ld16(tl + tcD4 + 64 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(w + 16));
      tmem_ld_wait();
      const float gam = vec[128 + trow];
#pragma unroll
      for (int e = 0; e < 32; ++e) ds[e] = fmaf(gam, ds[e], v[e] + w[e]);
    }
    __syncthreads();
    if (trow < 64) {
      float v[32], w[32];
      tmem_ld16(tl + tcD3 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tcD3 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      tmem_ld16(tl + tcD3 + 64 + 32 * hc, *reinterpret_cast<float(*)[16]>(w));
      tmem_ld16(tl + tcD3 + 64 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(w + 16));
      tmem_ld_wait();
      const int i = trow;
      if (i < Cc) {
        float* dv = g.dv + tok(a, b, t0 + i, h) * 128 + n0 + 32 * hc;
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(dv + e) =
              make_float4(v[e] + w[e] + xch2[i * 64 + ((32 * hc + e) ^ (i & 31))],
                          v[e + 1] + w[e + 1] + xch2[i * 64 + ((32 * hc + e + 1) ^ (i & 31))],
                          v[e + 2] + w[e + 2] + xch2[i * 64 + ((32 * hc + e + 2) ^ (i & 31))],
                          v[e + 3] + w[e + 3] + xch2[i * 64 + ((32 * hc + e + 3) ^ (i & 31))]);
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (s_abort) {
    if (tid == 0) {
      set_status(DR_ERR_TIMEOUT);
      if (nA > 0) mbar_wait(&bars[0], (nA - 1) & 1, kWait / 4);
      if (nB > 0) mbar_wait(&bars[1], (nB - 1) & 1, kWait / 4);
    }
  } else if (g.dS0) {
    float* d0 = g.dS0 + ((size_t)bh * 128 + trow) * 128 + n0 + 32 * hc;
#pragma unroll
    for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4*>(d0 + e) = make_float4(ds[e], ds[e + 1], ds[e + 2], ds[e + 3]);
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kCarryTcTmem);
}

// ================================================================= bwd_state
// Per chunk, five products over the dv index v (all fp32 data, K = 128):
//   X_Q = dO S_c^T, X_K = dR S_c^T (64 x 128, raw dq / dk for bwd_local),
//   dO E^T, dR E^T (64 x 64) and X_W = E dS^T (64 x 128),
// plus gamma <dS, S_c> (per-channel decay: per state row).  On tcgen05 (M = 128,
// fp32 in TMEM) as three MMA groups on bf16 hi/lo images (hi.hi + lo.hi + hi.lo):
//   G1  A = [dO ; dR] (128 rows),  B = S_c (128 rows)  -> D1 = [X_Q ; X_K]
//   G2  A = [dO ; dR],             B = E (64 rows)     -> D2 = [dO E^T ; dR E^T]
//   G3  A = dS (128 rows),         B = E               -> D3 = X_W^T
// (dO is bf16, so its lo rows are zero).  A persistent CTA of 16 warps per SM
// takes tasks (b, h, chunk) in turn: the fp32 blocks are read with coalesced
// 16-byte loads and split into 128B-swizzled K-major images, G1 and G2 run while
// dS is read (and <dS, S_c> formed from registers), dS's image replaces S_c's
// once G1 is done, and the readouts of D1 / D2 overlap G3.
constexpr int kStateThreads = 512;
constexpr uint32_t sAh = 0;           // [dO ; dR] hi, 2 k-blocks x 128 rows x 128 B
constexpr uint32_t sAl = 32768;       // [0 ; dR] lo
constexpr uint32_t sBh = 65536;       // S_c hi, then dS hi
constexpr uint32_t sBl = 98304;       // S_c lo, then dS lo
constexpr uint32_t sEh = 131072;      // E hi, 2 k-blocks x 64 rows x 128 B
constexpr uint32_t sEl = 147456;      // E lo
constexpr uint32_t kStateSmem = 163840 + 1024;
constexpr uint32_t tD1 = 0, tD2 = 128, tD3 = 192, kStateTmem = 256;
constexpr uint32_t I_S128 = idesc_bf16(128, 128, 0, 0);
constexpr uint32_t I_S64 = idesc_bf16(128, 64, 0, 0);

// 4 fp32 -> bf16 hi (8 bytes) and lo (8 bytes) at a swizzled K-major position
__device__ __forceinline__ void put4(uint8_t* hi, uint8_t* lo, uint32_t off, const float4& x) {
  const float f[4] = {x.x, x.y, x.z, x.w};
  uint32_t h[2], l[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    h[i] = pack_bf16(f[2 * i], f[2 * i + 1]);
    l[i] = pack_bf16(f[2 * i] - __uint_as_float(h[i] << 16),
                     f[2 * i + 1] - __uint_as_float(h[i] & 0xFFFF0000u));
  }
  *reinterpret_cast<uint2*>(hi + off) = make_uint2(h[0], h[1]);
  *reinterpret_cast<uint2*>(lo + off) = make_uint2(l[0], l[1]);
}

__global__ void __launch_bounds__(kStateThreads, 1)
    bwd_state_kernel(FwdArgs a, BwdArgs g, long n) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bars[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ float s_red[kStateThreads / 32];
  __shared__ float s_rowp[kStateThreads / 32][128];
  __shared__ volatile int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NC = (a.T + 63) / 64;
  const bool pc = a.variant == DR_KDA || a.variant == DR_KDN || a.variant == DR_PKDA ||
                  a.variant == DR_IKDN;
  const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(g.d_out);
  // this thread's 4 columns of v in every 128-wide row: k-block and swizzled column
  const uint32_t kb = lane >> 4, col = 4 * (lane & 15);

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, kStateTmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t a_h = smem_u32(sm + sAh), a_l = smem_u32(sm + sAl);
  const uint32_t b_h = smem_u32(sm + sBh), b_l = smem_u32(sm + sBl);
  const uint32_t e_h = smem_u32(sm + sEh), e_l = smem_u32(sm + sEl);
  int it = 0, n1 = 0, n2 = 0;   // tasks done; groups committed (thread 0)

  for (long task = blockIdx.x; task < n; task += gridDim.x, ++it) {
    const int bh = (int)(task / NC), c = (int)(task % NC);
    const int b = bh / a.H, h = bh % a.H;
    const int t0 = 64 * c, Cc = min(64, a.T - t0);
    const float* Sc = g.w.S + (size_t)task * 16384;
    const float* Ec = g.w.E + (size_t)task * 8192;
    const float* dSc = g.w.dS + (size_t)task * 16384;
    // ---- images: dO (bf16, copied as is; its lo rows zero, rewritten every task since
    //      the previous task's outputs passed through them), dR, S_c and E (hi / lo)
    for (int e = tid; e < 64 * 16; e += kStateThreads) {
      const int r = e >> 4, cz = e & 15;
      *reinterpret_cast<uint4*>(sm + sAl + (cz >> 3) * 16384 + r * 128 + (cz & 7) * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    for (int e = tid; e < 64 * 16; e += kStateThreads) {
      const int r = e >> 4, cc = e & 15;
      cpa16(sm + sAh + (cc >> 3) * 16384 + sw128_offset(r, 8 * (cc & 7)),
            dO + tok(a, b, t0 + min(r, Cc - 1), h) * 128 + 8 * cc, r < Cc ? 16 : 0);
    }
    // S_c, E, dS in [column quad][row][4] order: element j of this thread is column
    // quad warp + 16 (j >> 2) (k-block j >> 2, columns 4 warp ..) of row lane + 32 (j & 3)
    float4 sv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      sv[j] = *reinterpret_cast<const float4*>(Sc + ((warp + 16 * (j >> 2)) * 128 + lane + 32 * (j & 3)) * 4);
    {
      float4 ev[4], rv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ev[j] = *reinterpret_cast<const float4*>(Ec + ((warp + 16 * (j >> 1)) * 64 + lane + 32 * (j & 1)) * 4);
        const int r = 16 * j + warp;
        rv[j] = r < Cc ? *reinterpret_cast<const float4*>(g.dv + tok(a, b, t0 + r, h) * 128 + 4 * lane)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = 16 * j + warp;
        put4(sm + sEh + (j >> 1) * 8192, sm + sEl + (j >> 1) * 8192, sw128_offset(lane + 32 * (j & 1), 4 * warp),
             ev[j]);
        put4(sm + sAh + kb * 16384, sm + sAl + kb * 16384, sw128_offset(64 + r, col), rv[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      put4(sm + sBh + (j >> 2) * 16384, sm + sBl + (j >> 2) * 16384, sw128_offset(lane + 32 * (j & 3), 4 * warp),
           sv[j]);
    cpa_wait_all();
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {   // G1 and G2
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32, oe = (ks >> 2) * 8192 + (ks & 3) * 32;
        const uint64_t ah = desc_sw128(a_h + o, 16, 1024), al = desc_sw128(a_l + o, 16, 1024);
        const uint64_t bh_ = desc_sw128(b_h + o, 16, 1024), bl = desc_sw128(b_l + o, 16, 1024);
        const uint64_t eh = desc_sw128(e_h + oe, 16, 1024), el = desc_sw128(e_l + oe, 16, 1024);
        mma_bf16(tmem + tD1, ah, bh_, I_S128, ks > 0);
        mma_bf16(tmem + tD1, al, bh_, I_S128, true);
        mma_bf16(tmem + tD1, ah, bl, I_S128, true);
        mma_bf16(tmem + tD2, ah, eh, I_S64, ks > 0);
        mma_bf16(tmem + tD2, al, eh, I_S64, true);
        mma_bf16(tmem + tD2, ah, el, I_S64, true);
      }
      mma_commit(&bars[0]);
      ++n1;
    }
    // ---- dS into registers; gamma <dS, S_c> from the S_c values already held
    float4 dv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      dv[j] = *reinterpret_cast<const float4*>(dSc + ((warp + 16 * (j >> 2)) * 128 + lane + 32 * (j & 3)) * 4);
    const float* rvec = reinterpret_cast<const float*>(g.w.rec + (size_t)task * g.w.recb + rVecF);
    float part = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // rows lane + 32 j: column quads warp and warp + 16
      const float p = dv[j].x * sv[j].x + dv[j].y * sv[j].y + dv[j].z * sv[j].z + dv[j].w * sv[j].w +
                      dv[j + 4].x * sv[j + 4].x + dv[j + 4].y * sv[j + 4].y + dv[j + 4].z * sv[j + 4].z +
                      dv[j + 4].w * sv[j + 4].w;
      if (pc) s_rowp[warp][lane + 32 * j] = p;
      part += p;
    }
    if (!pc) {
      part = warp_sum(part);
      if (lane == 0) s_red[warp] = part;
    }
    if (!mbar_wait(&bars[0], it & 1, kWait)) s_abort = 1;
    __syncthreads();
    if (s_abort) break;
    if (!pc && tid == 0) {
      float tsum = 0.f;
      for (int w = 0; w < kStateThreads / 32; ++w) tsum += s_red[w];
      g.w.SS[task] = rvec[128] * tsum;
    }
    if (pc && tid < 128) {   // gamma_c <dS, S_c>_c per state row: the 16 warps' parts
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kStateThreads / 32; ++w) t += s_rowp[w][tid];
      g.w.SS[(size_t)task * 128 + tid] = rvec[128 + tid] * t;
    }
    // ---- dS's image over S_c's (G1 has read it), then G3
#pragma unroll
    for (int j = 0; j < 8; ++j)
      put4(sm + sBh + (j >> 2) * 16384, sm + sBl + (j >> 2) * 16384, sw128_offset(lane + 32 * (j & 3), 4 * warp),
           dv[j]);
    fence_proxy_async();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t o = (ks >> 2) * 16384 + (ks & 3) * 32, oe = (ks >> 2) * 8192 + (ks & 3) * 32;
        const uint64_t dh = desc_sw128(b_h + o, 16, 1024), dl = desc_sw128(b_l + o, 16, 1024);
        const uint64_t eh = desc_sw128(e_h + oe, 16, 1024), el = desc_sw128(e_l + oe, 16, 1024);
        mma_bf16(tmem + tD3, dh, eh, I_S64, ks > 0);
        mma_bf16(tmem + tD3, dl, eh, I_S64, true);
        mma_bf16(tmem + tD3, dh, el, I_S64, true);
      }
      mma_commit(&bars[1]);
      ++n2;
    }
    // ---- D1, D2 out: warp (quadrant q, column quarter cq); lane = TMEM row.  The rows
    //      go out row-contiguously through shared memory: D1 through the [dO ; dR]
    //      images (G1 and G2 have read them), D2 through the E images once G3 has
    //      read those (16-byte pieces XOR-swizzled by row against bank conflicts)
    const int q = warp & 3, cq = warp >> 2, row = 32 * q + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
    float z[16];
    {
      float x[16], y[16];
      tmem_ld16(tl + tD1 + 32 * cq, x);
      tmem_ld16(tl + tD1 + 32 * cq + 16, y);
      tmem_ld16(tl + tD2 + 16 * cq, z);
      tmem_ld_wait();
      uint8_t* st1 = sm + sAh + row * 512;
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        const int ch = 8 * cq + e / 4;
        *reinterpret_cast<float4*>(st1 + ((ch ^ (row & 31)) << 4)) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
        *reinterpret_cast<float4*>(st1 + (((ch + 4) ^ (row & 31)) << 4)) =
            make_float4(y[e], y[e + 1], y[e + 2], y[e + 3]);
      }
    }
    __syncthreads();
    for (int u = tid; u < 128 * 32; u += kStateThreads) {   // X_Q / X_K rows out
      const int r = u >> 5, ch = u & 31, i = r & 63;
      if (i < Cc)
        *reinterpret_cast<float4*>((r < 64 ? g.dq : g.dk) + tok(a, b, t0 + i, h) * 128 + 4 * ch) =
            *reinterpret_cast<const float4*>(sm + sAh + r * 512 + ((ch ^ (r & 31)) << 4));
    }
    if (!mbar_wait(&bars[1], it & 1, kWait)) s_abort = 1;
    __syncthreads();
    if (s_abort) break;
    tc_fence_after();
    {
      uint8_t* st2 = sm + sEh + row * 256;
#pragma unroll
      for (int e = 0; e < 16; e += 4)
        *reinterpret_cast<float4*>(st2 + (((4 * cq + e / 4) ^ (row & 15)) << 4)) =
            make_float4(z[e], z[e + 1], z[e + 2], z[e + 3]);
    }
    {   // D3 = X_W^T: lane = state row n, column = token j -> X_W[j][n] (coalesced in n)
      float z[16];
      tmem_ld16(tl + tD3 + 16 * cq, z);
      tmem_ld_wait();
      float* xw = g.w.XW + (size_t)task * 8192 + row;
#pragma unroll
      for (int e = 0; e < 16; ++e) xw[(16 * cq + e) * 128] = z[e];
    }
    __syncthreads();
    for (int u = tid; u < 128 * 16; u += kStateThreads) {   // dO E^T / dR E^T rows out
      const int r = u >> 4, ch = u & 15;
      *reinterpret_cast<float4*>((r < 64 ? g.w.dP : g.w.dL) + (size_t)task * 4096 + (r & 63) * 64 + 4 * ch) =
          *reinterpret_cast<const float4*>(sm + sEh + r * 256 + ((ch ^ (r & 15)) << 4));
    }
    tc_fence_before();
    __syncthreads();   // TMEM read and every image consumed before the next task
  }
  if (s_abort && tid == 0) {   // drain: no MMA may still write TMEM after the dealloc
    set_status(DR_ERR_TIMEOUT);
    if (n1 > 0) mbar_wait(&bars[0], (n1 - 1) & 1, kWait / 4);
    if (n2 > 0) mbar_wait(&bars[1], (n2 - 1) & 1, kWait / 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kStateTmem);
}

// ================================================================= bwd_local
constexpr int cLDK = 132;   // K^, Q^, W, staging [64][132]
constexpr int cLDM = 68;    // M_P, M_L [64][68]
// Scalar decay (GDN, KLA, PGDN): a persistent CTA per SM takes tasks (b, h, chunk).
// The chunk's products run on tcgen05 (M = 128, fp32 in TMEM) over three bf16 hi/lo
// images (hi.hi + lo.hi + hi.lo):
//   IA = [Q^ ; K^] (128 rows i, K-major in c),  IW = W (64 rows j),
//   IM = [M_P ; M_L] (128 rows i, K-major in j),  M_P = dP.D (j <= i),
//   M_L = -dL.D (j < i), D_ij = e^{g_i - g_j},
// and three MMA groups issued together:
//   G1 = IA IW^T            -> [Q^ W^T ; K^ W^T]   (the Grams, for the decay terms)
//   G2 = IA^T IM (MN-major) -> dw^T = Q^^T M_P + K^^T M_L   (lane = channel)
//   G3 = IM IW  (MN-major)  -> [M_P W ; M_L W] = [dq^_P ; dk^_L]  (lane = token)
// Every Gram entry X_ij = M_P,ij (Q^W^T)_ij + M_L,ij (K^W^T)_ij adds to dg_i and takes
// from dg_j; dw = dw_G2 + e^{G-g} X_W; the rows then add e^g X_Q / -e^g X_K (the
// raw dO S_c^T, dR S_c^T that bwd_state left in dq / dk), the write gain (GDN eta,
// KLA eta / (s + eps)) and the norms; d log alpha is dg's reverse cumulative sum
// with dG = gamma <dS, S_c> + sum_j e^{G-g_j} X_W,j . w_j on the chunk's last token.
// PGDN takes W from the record's explicit write keys, keeps dL/dw and the memory
// part of dL/dk^ (and the key norms) for pgdn_gain_bwd.
constexpr uint32_t lA = 0;            // IA hi (2 k-blocks x 128 rows x 128 B) | lo at +32 KB
constexpr uint32_t lW = 65536;        // IW hi (2 k-blocks x 64 rows) | lo at +16 KB
constexpr uint32_t lM = 98304;        // IM hi (128 rows x 64 j) | lo at +16 KB
constexpr uint32_t lD = 131072;       // fp32 dw [64 j][cLDK]
constexpr uint32_t lX = lD + 64 * cLDK * 4;   // fp32 Gram terms X [64 i][65]
constexpr uint32_t lR = lX + 64 * 65 * 4;     // raw k | q rows, bf16 [64][cKR] each
constexpr int cKR = 136;
constexpr uint32_t kLocalSmem = lR + 2 * 64 * cKR * 2 + 1024;
constexpr uint32_t tG1 = 0, tG2 = 64, tG3 = 128, kLocalTmem = 256;
constexpr uint32_t I_L1 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t I_L2 = idesc_bf16(128, 64, 1, 1);
constexpr uint32_t I_L3 = idesc_bf16(128, 128, 0, 1);

template <int VARIANT>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_local_kernel(FwdArgs a, BwdArgs g, long n) {
  constexpr bool PG = VARIANT == DR_PGDN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  float* sD = reinterpret_cast<float*>(sm + lD);
  float* sX = reinterpret_cast<float*>(sm + lX);
  float* sX2 = reinterpret_cast<float*>(sm + lW);   // scalar decay: after the products, IW is free
  uint16_t* sKr = reinterpret_cast<uint16_t*>(sm + lR);
  uint16_t* sQr = sKr + 64 * cKR;
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int s_abort;
  __shared__ float s_g[64], s_cr[64], s_qn[64], s_beta[64], s_s[64], s_eta[64], s_ew[64];
  __shared__ float s_dgx[64], s_dgr[64], s_dgq[64], s_dgk[64], s_dbeta[64], s_dGt[64];
  __shared__ float s_dot[2][128], s_xd[2][128], s_p1[4][64], s_p2[4][64];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NC = (a.T + 63) / 64;
  const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(a.k);
  const __nv_bfloat16* Qp = static_cast<const __nv_bfloat16*>(a.q);
  auto bf = [](uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); };
  // element (row, col) of a bf16 hi/lo image with 128-byte rows (one 64-wide block)
  auto hl = [&](uint32_t base, uint32_t lo_off, int row, int col) {
    const uint32_t o = base + sw128_offset(row, col);
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + o)) +
           __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + o + lo_off));
  };

  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) tmem_alloc(&tmem_base_s, kLocalTmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const int q4 = warp & 3, hc = warp >> 2, trow = 32 * q4 + lane;
  const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
  int it = 0, nc = 0;

  // L2 prefetch (one bulk hint per contiguous block): this task's X_W, read after its
  // products, and the next task's dP / dL (and PGDN's write keys)
  auto prefetch = [&](long tk, bool now) {
    if (tk >= n || tid != 0) return;
    if (now) {
      l2_prefetch(g.w.XW + (size_t)tk * 8192, 32768);
    } else {
      l2_prefetch(g.w.dP + (size_t)tk * 4096, 16384);
      l2_prefetch(g.w.dL + (size_t)tk * 4096, 16384);
      if (PG) l2_prefetch(g.w.rec + (size_t)tk * g.w.recb + rWF, 32768);
    }
  };
  prefetch(blockIdx.x, false);

  for (long task = blockIdx.x; task < n; task += gridDim.x, ++it) {
    const int bh = (int)(task / NC), c = (int)(task % NC);
    const int b = bh / a.H, h = bh % a.H;
    const int t0 = 64 * c, Cc = min(64, a.T - t0);
    prefetch(task, true);
    prefetch(task + gridDim.x, false);
    // ---- raw rows, gates, dP / dL (every load issued before the first shared-memory
    //      store, which could otherwise alias them), PGDN's write-key images
    float4 mp[4][2];   // dP / dL, used by the images below
    {
      uint4 rk[4], rq[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int e = tid + r * kBwdThreads, j = e >> 4, c0 = 8 * (e & 15);
        const bool live = j < Cc;
        const long o = tok(a, b, t0 + (live ? j : 0), h) * 128 + c0;
        rk[r] = live ? *reinterpret_cast<const uint4*>(K + o) : make_uint4(0u, 0u, 0u, 0u);
        rq[r] = live ? *reinterpret_cast<const uint4*>(Qp + o) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int u = tid + r * kBwdThreads, row = u >> 3, j0 = 8 * (u & 7);
        const float4* src = reinterpret_cast<const float4*>((row >= 64 ? g.w.dL : g.w.dP) +
                                                            (size_t)task * 4096 + (row & 63) * 64 + j0);
        mp[r][0] = src[0];
        mp[r][1] = src[1];
      }
      float lg = 0.f, et = 0.f;
      if (tid < Cc) {
        lg = a.log_alpha[tok(a, b, t0 + tid, h)];
        et = a.eta[tok(a, b, t0 + tid, h)];
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int e = tid + r * kBwdThreads, j = e >> 4, c0 = 8 * (e & 15);
        *reinterpret_cast<uint4*>(sKr + j * cKR + c0) = rk[r];
        *reinterpret_cast<uint4*>(sQr + j * cKR + c0) = rq[r];
      }
      if (tid < 64) {
        s_g[tid] = lg;
        s_eta[tid] = et;
      }
    }
    if (PG) {
      const uint8_t* rw = g.w.rec + (size_t)task * g.w.recb + rWF;
      for (int e = tid; e < 32768 / 16; e += kBwdThreads) cpa16(sm + lW + 16 * e, rw + 16 * e);
    }
    __syncthreads();
    {   // norms: four threads per row
      const int j = tid >> 2, part = tid & 3;
      float kk = 0.f, qq = 0.f;
#pragma unroll 8
      for (int c0 = 32 * part; c0 < 32 * part + 32; ++c0) {
        const float x = bf(sKr[j * cKR + c0]), y = bf(sQr[j * cKR + c0]);
        kk += x * x;
        qq += y * y;
      }
      kk += __shfl_xor_sync(0xffffffffu, kk, 1);
      kk += __shfl_xor_sync(0xffffffffu, kk, 2);
      qq += __shfl_xor_sync(0xffffffffu, qq, 1);
      qq += __shfl_xor_sync(0xffffffffu, qq, 2);
      if (part == 0) {
        const float cr = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
        const float qn = a.q_l2norm ? 1.f / fmaxf(sqrtf(qq), 1e-30f) : 1.f;
        const float s = kk * cr * cr;
        s_cr[j] = cr;
        s_qn[j] = qn;
        s_s[j] = s;
        s_beta[j] = VARIANT == DR_KLA ? s_eta[j] / (s + a.eps) : s_eta[j];
        if (PG && j < Cc) g.w.CR[(size_t)task * 64 + j] = cr;
      }
    }
    if (warp == 0) {   // inclusive cumulative log-decay (two tokens per lane)
      const float x0 = s_g[2 * lane], x1 = s_g[2 * lane + 1];
      float s = x0 + x1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      __syncwarp();
      s_g[2 * lane] = s - x1;
      s_g[2 * lane + 1] = s;
    }
    __syncthreads();
    const float G = s_g[Cc - 1];
    if (tid < 64) s_ew[tid] = tid < Cc ? __expf(G - s_g[tid]) : 0.f;
    // ---- images: IA = [q^ ; k^], IW = beta k^ (PGDN: copied above), IM = [M_P ; M_L]
#pragma unroll 2
    for (int r = 0; r < 8; ++r) {
      const int u = tid + r * kBwdThreads, row = u >> 4, cg = u & 15, kb = cg >> 3, c8 = (cg & 7) * 8;
      const bool isk = row >= 64;
      const int j = row & 63;
      const uint16_t* src = (isk ? sKr : sQr) + j * cKR + 64 * kb + c8;
      const uint4 raw = *reinterpret_cast<const uint4*>(src);
      float x[8];
      unpack8(raw, x);
      const float sc = isk ? s_cr[j] : s_qn[j];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= sc;
      uint4 hi, lo;
      split8(x, hi, lo);
      const uint32_t o = lA + kb * 16384 + sw128_offset(row, c8);
      *reinterpret_cast<uint4*>(sm + o) = hi;
      *reinterpret_cast<uint4*>(sm + o + 32768) = lo;
      if (!PG && isk) {
        const float bt = s_beta[j];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= bt;
        split8(x, hi, lo);
        const uint32_t ow = lW + kb * 8192 + sw128_offset(j, c8);
        *reinterpret_cast<uint4*>(sm + ow) = hi;
        *reinterpret_cast<uint4*>(sm + ow + 16384) = lo;
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int u = tid + r * kBwdThreads, row = u >> 3, j0 = 8 * (u & 7);
      const bool isl = row >= 64;
      const int i = row & 63;
      const float4 v0 = mp[r][0], v1 = mp[r][1];
      const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      const float gi = s_g[i];
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = j0 + e;
        const bool keep = isl ? j < i : j <= i;
        x[e] = keep ? (isl ? -v[e] : v[e]) * __expf(gi - s_g[j]) : 0.f;
      }
      uint4 hi, lo;
      split8(x, hi, lo);
      const uint32_t o = lM + sw128_offset(row, j0);
      *reinterpret_cast<uint4*>(sm + o) = hi;
      *reinterpret_cast<uint4*>(sm + o + 16384) = lo;
    }
    cpa_wait_all();
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t ah = smem_u32(sm + lA), al = ah + 32768;
      const uint32_t wh = smem_u32(sm + lW), wl = wh + 16384;
      const uint32_t mh = smem_u32(sm + lM), ml = mh + 16384;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {   // G1: K = 128 channels (K-major A and B)
        const uint32_t oa = (ks >> 2) * 16384 + (ks & 3) * 32, ow = (ks >> 2) * 8192 + (ks & 3) * 32;
        const uint64_t dah = desc_sw128(ah + oa, 16, 1024), dal = desc_sw128(al + oa, 16, 1024);
        const uint64_t dwh = desc_sw128(wh + ow, 16, 1024), dwl = desc_sw128(wl + ow, 16, 1024);
        mma_bf16(tmem + tG1, dah, dwh, I_L1, ks > 0);
        mma_bf16(tmem + tG1, dal, dwh, I_L1, true);
        mma_bf16(tmem + tG1, dah, dwl, I_L1, true);
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {   // G2: K = 128 rows i (A = IA^T and B = IM, MN-major)
        const uint32_t o = ks * 2048;
        const uint64_t dah = desc_sw128(ah + o, 16384, 1024), dal = desc_sw128(al + o, 16384, 1024);
        const uint64_t dmh = desc_sw128(mh + o, 16384, 1024), dml = desc_sw128(ml + o, 16384, 1024);
        mma_bf16(tmem + tG2, dah, dmh, I_L2, ks > 0);
        mma_bf16(tmem + tG2, dal, dmh, I_L2, true);
        mma_bf16(tmem + tG2, dah, dml, I_L2, true);
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {   // G3: K = 64 tokens j (A = IM K-major, B = IW MN-major)
        const uint64_t dmh = desc_sw128(mh + ks * 32, 16, 1024), dml = desc_sw128(ml + ks * 32, 16, 1024);
        const uint64_t dwh = desc_sw128(wh + ks * 2048, 8192, 1024);
        const uint64_t dwl = desc_sw128(wl + ks * 2048, 8192, 1024);
        mma_bf16(tmem + tG3, dmh, dwh, I_L3, ks > 0);
        mma_bf16(tmem + tG3, dml, dwh, I_L3, true);
        mma_bf16(tmem + tG3, dmh, dwl, I_L3, true);
      }
      mma_commit(&bar);
      ++nc;
    }
    if (!mbar_wait(&bar, it & 1, kWait)) s_abort = 1;
    __syncthreads();
    if (s_abort) break;
    tc_fence_after();
    // X_Q (rows 0-63) and X_K (64-127) staged into the consumed IA images for G3:
    // row-contiguous copies here, then each thread reads its own row (16-byte pieces
    // XOR-swizzled by row, so a warp's 32 rows fall on distinct banks)
    for (int u = tid; u < 128 * 32; u += kBwdThreads) {
      const int r = u >> 5, ch = u & 31, i = r & 63;
      const bool live = i < Cc;
      const float* src = (r < 64 ? g.dq : g.dk) + tok(a, b, t0 + (live ? i : 0), h) * 128 + 4 * ch;
      cpa16(sm + lA + r * 512 + ((ch ^ (r & 31)) << 4), src, live ? 16 : 0);
    }
    // ---- G1: X_ij = M_P,ij (Q^W^T)_ij + M_L,ij (K^W^T)_ij (query rows first, then key rows)
    {
      float v[32];
      tmem_ld16(tl + tG1 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tG1 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      tmem_ld_wait();
      const int i = trow & 63;
      float m[32];   // this row's 32 IM entries, hi + lo, eight per 16-byte read
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t o = lM + sw128_offset(trow, 32 * hc + 8 * q);
        float mh[8], ml[8];
        unpack8(*reinterpret_cast<const uint4*>(sm + o), mh);
        unpack8(*reinterpret_cast<const uint4*>(sm + o + 16384), ml);
#pragma unroll
        for (int e = 0; e < 8; ++e) m[8 * q + e] = mh[e] + ml[e];
      }
      if (!PG) {   // query rows into sX, key rows into sX2 (the consumed IW images)
        float* dst = (trow < 64 ? sX : sX2) + i * 65 + 32 * hc;
#pragma unroll
        for (int e = 0; e < 32; ++e) dst[e] = m[e] * v[e];
      } else {     // PGDN reads its IW images below: the halves meet in sX in turn
        if (trow < 64) {
#pragma unroll
          for (int e = 0; e < 32; ++e) sX[i * 65 + 32 * hc + e] = m[e] * v[e];
        }
        __syncthreads();
        if (trow >= 64) {
#pragma unroll
          for (int e = 0; e < 32; ++e) sX[i * 65 + 32 * hc + e] += m[e] * v[e];
        }
      }
    }
    // ---- G2: dw_jc = (dw^T)_cj + e^{G-g_j} X_W,jc, transposed into sD (lane = channel);
    //      per token j the sums over channels d beta_j = dw_j . k^_j and X_W,j . w_j, by
    //      a butterfly over the warp's lanes (lane l ends with token 32 hc + l) and the
    //      four quadrants' parts in shared memory
    {
      float v[32], xv[32];
      const float* xw = g.w.XW + (size_t)task * 8192 + trow;
#pragma unroll
      for (int e = 0; e < 32; ++e) xv[e] = xw[(32 * hc + e) * 128];
      tmem_ld16(tl + tG2 + 32 * hc, *reinterpret_cast<float(*)[16]>(v));
      tmem_ld16(tl + tG2 + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int j = 32 * hc + e;
        const float dw = v[e] + s_ew[j] * xv[e];
        sD[j * cLDK + trow] = dw;
        if (PG) g.w.DW[(size_t)task * 8192 + j * 128 + trow] = dw;
        const float kh = bf(sKr[j * cKR + trow]) * s_cr[j];
        const float w = PG ? hl(lW + (trow >> 6) * 8192, 16384, j, trow & 63) : s_beta[j] * kh;
        v[e] = dw * kh;
        xv[e] = xv[e] * w;
      }
#pragma unroll
      for (int st = 16; st >= 1; st >>= 1) {
        const bool up = (lane & st) != 0;
#pragma unroll
        for (int i = 0; i < st; ++i) {
          const float s1 = up ? v[i] : v[i + st], s2 = up ? xv[i] : xv[i + st];
          const float r1 = __shfl_xor_sync(0xffffffffu, s1, st);
          const float r2 = __shfl_xor_sync(0xffffffffu, s2, st);
          v[i] = (up ? v[i + st] : v[i]) + r1;
          xv[i] = (up ? xv[i + st] : xv[i]) + r2;
        }
      }
      s_p1[q4][32 * hc + lane] = v[0];
      s_p2[q4][32 * hc + lane] = xv[0];
    }
    __syncthreads();
    if (tid < 64) {   // each Gram entry adds to dg of its row and takes from dg of its column
      float r = 0.f;
      for (int j = 0; j < 64; ++j) r += PG ? sX[tid * 65 + j] : sX[tid * 65 + j] + sX2[tid * 65 + j];
      s_dgr[tid] = r;
    } else if (tid < 128) {
      const int j = tid - 64;
      float cs = 0.f;
      for (int i = 0; i < 64; ++i) cs += PG ? sX[i * 65 + j] : sX[i * 65 + j] + sX2[i * 65 + j];
      s_dgx[j] = cs;
    } else if (tid < 192) {   // d beta_j and e^{G-g_j} X_W,j . w_j from the quadrants' parts
      const int j = tid - 128;
      const float dwk = s_p1[0][j] + s_p1[1][j] + s_p1[2][j] + s_p1[3][j];
      const float xww = s_p2[0][j] + s_p2[1][j] + s_p2[2][j] + s_p2[3][j];
      s_dbeta[j] = j < Cc ? dwk : 0.f;
      s_dGt[j] = s_ew[j] * xww;
    }
    cpa_wait_all();
    __syncthreads();
    // ---- G3: rows of dq^ (TMEM rows 0-63) and dk^ (64-127); warp half hc takes 64 columns
    {
      const bool isk = trow >= 64;
      const int i = trow & 63;
      const bool live = i < Cc;
      const float eg = __expf(s_g[i]);
      float* xrow = reinterpret_cast<float*>(sm + lA + trow * 512);   // staged X_Q / X_K, out
      auto xpiece = [&](int ch) { return reinterpret_cast<float4*>(xrow + 4 * (ch ^ (trow & 31))); };
      const uint16_t* rr = (isk ? sKr : sQr) + i * cKR + 64 * hc;
      const float sc = isk ? s_cr[i] : s_qn[i];
      const float bgain = (PG || !isk) ? 0.f : s_beta[i];
      const float se = s_s[i] + a.eps, db = s_dbeta[i];
      const float ds2 = (VARIANT == DR_KLA && isk) ? -2.f * db * s_eta[i] / (se * se) : 0.f;
      float d[64];
      float dot = 0.f, xd = 0.f;
#pragma unroll
      for (int p = 0; p < 2; ++p) {   // 32 columns: the raw row's loads first, then TMEM
        float4 x4[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x4[e] = *xpiece(16 * hc + 8 * p + e);
        float v[32];
        tmem_ld16(tl + tG3 + 64 * hc + 32 * p, *reinterpret_cast<float(*)[16]>(v));
        tmem_ld16(tl + tG3 + 64 * hc + 32 * p + 16, *reinterpret_cast<float(*)[16]>(v + 16));
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; ++e) {   // four columns: the raw row and dw as 8- and 16-byte reads
          const float xs[4] = {x4[e].x, x4[e].y, x4[e].z, x4[e].w};
          const uint2 r2 = *reinterpret_cast<const uint2*>(rr + 32 * p + 4 * e);
          const float xr[4] = {__uint_as_float(r2.x << 16), __uint_as_float(r2.x & 0xFFFF0000u),
                               __uint_as_float(r2.y << 16), __uint_as_float(r2.y & 0xFFFF0000u)};
          const float4 sd4 = isk ? *reinterpret_cast<const float4*>(sD + i * cLDK + 64 * hc + 32 * p + 4 * e)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
          const float sdv[4] = {sd4.x, sd4.y, sd4.z, sd4.w};
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            const int cc = 32 * p + 4 * e + f;
            const float xh = xr[f] * sc;
            const float val = isk ? v[4 * e + f] - eg * xs[f] + bgain * sdv[f] + ds2 * xh
                                  : v[4 * e + f] + eg * xs[f];
            d[cc] = val;
            dot += val * xh;
            xd += xs[f] * xh;
          }
        }
      }
      s_dot[hc][trow] = dot;
      s_xd[hc][trow] = xd;
      __syncthreads();
      dot = s_dot[0][trow] + s_dot[1][trow];
      if (live) {
        const bool norm = isk ? (a.k_l2norm && !PG) : a.q_l2norm;
#pragma unroll
        for (int cc = 0; cc < 64; cc += 4) {
          float o4[4];
          const uint2 r2 = *reinterpret_cast<const uint2*>(rr + cc);
          const float xr[4] = {__uint_as_float(r2.x << 16), __uint_as_float(r2.x & 0xFFFF0000u),
                               __uint_as_float(r2.y << 16), __uint_as_float(r2.y & 0xFFFF0000u)};
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            const float xh = xr[f] * sc;
            o4[f] = norm ? (d[cc + f] - xh * dot) * sc : d[cc + f];
          }
          *xpiece(16 * hc + cc / 4) = make_float4(o4[0], o4[1], o4[2], o4[3]);
        }
        if (hc == 0) {
          const float x = s_xd[0][trow] + s_xd[1][trow];
          if (isk) {
            s_dgk[i] = -eg * x;
            if (!PG) g.deta[tok(a, b, t0 + i, h)] = VARIANT == DR_KLA ? db / se : db;
          } else {
            s_dgq[i] = eg * x;
          }
        }
      } else if (hc == 0) {
        if (isk) s_dgk[i] = 0.f; else s_dgq[i] = 0.f;
      }
    }
    tc_fence_before();
    __syncthreads();
    for (int u = tid; u < 128 * 32; u += kBwdThreads) {   // dq^, dk^ rows out (coalesced)
      const int r = u >> 5, ch = u & 31, i = r & 63;
      if (i < Cc)
        *reinterpret_cast<float4*>((r < 64 ? g.dq : g.dk) + tok(a, b, t0 + i, h) * 128 + 4 * ch) =
            *reinterpret_cast<const float4*>(sm + lA + r * 512 + ((ch ^ (r & 31)) << 4));
    }
    // ---- d log alpha: reverse cumulative sum of dg, dG (+ gamma <dS, S_c>) on the last token
    if (warp == 0) {
      float x[2];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int t = 63 - 2 * lane - m;
        x[m] = s_dgr[t] - s_dgx[t] - s_dGt[t] + s_dgq[t] + s_dgk[t];
      }
      float dG = 0.f;
      for (int j = lane; j < 64; j += 32) dG += s_dGt[j];
      dG = warp_sum(dG) + g.w.SS[task];
      if (63 - 2 * lane == Cc - 1) x[0] += dG;
      if (62 - 2 * lane == Cc - 1) x[1] += dG;
      float s = x[0] + x[1];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      const int ta = 63 - 2 * lane, tb = 62 - 2 * lane;
      if (ta < Cc) g.dla[tok(a, b, t0 + ta, h)] = s - x[1];
      if (tb < Cc) g.dla[tok(a, b, t0 + tb, h)] = s;
    }
    __syncthreads();   // every buffer read before the next task writes it
  }
  if (s_abort && tid == 0) {   // drain: no MMA may still write TMEM after the dealloc
    set_status(DR_ERR_TIMEOUT);
    if (nc > 0) mbar_wait(&bar, (nc - 1) & 1, kWait / 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kLocalTmem);
}

// ================================================================= bwd_local_pc
// Per-channel decay (KDA; the chunk part of Diagonal KDN): one CTA per (b, h,
// chunk).  With D_ijc = exp(g_ic - g_jc) per channel the Gram gradients do not
// factor into whole-chunk products; each 16-token block row I takes its middle
// token m(I) as reference, as the forward's Gram does (every factor bounded by the
// decay over 8 tokens or <= 1):
//   dq^_i += e^{g_i - g_m(I)} . sum_j (M_P)_ij [w_j e^{g_m(I) - g_j}]     (i in I, j <= i)
//   dk^_i += e^{g_i - g_m(I)} . sum_j (M_L)_ij [w_j e^{g_m(I) - g_j}]
//   dw_j  += sum_{I >= J} e^{g_m(I) - g_j} . sum_{i in I} ((M_P)_ij q~_i + (M_L)_ij k~_i),
//            q~_i = q^_i e^{g_i - g_m(I)},  k~ likewise,
// with M_P = dP (j <= i) and M_L = -dR E^T (j < i), on TF32x3 tiles.  Every Gram
// entry adds x_ic dx_ic to dg_ic and takes w_jc dw_jc from dg_jc, so per channel
//   dg = q^ . dq^_P + k^ . dk^_L - w . dw_{P,L} + e^g (X_Q . q^ - X_K . k^) - Wbar . X_W,
// dG_c = gamma_c <dS_c, S_c> + sum_j Wbar_jc X_W,jc on the chunk's last token, and
// d log alpha = the reverse cumulative sum of dg per channel.  dq^ and dk^ gather
// in the gradient arrays (bwd_state left X_Q = dO S_c^T, X_K = dR S_c^T there).
// KDA's gain (w = eta k^): d eta = dw . k^, dk^ += eta dw, then the L2 norms;
// Diagonal KDN, PKDA and isotropic KDN keep dw and dk^ for their gain kernels.
constexpr int cKRS = 136;   // raw k, q rows (bf16): 272 bytes, 4 banks apart
constexpr int kPcLocalSmem = (4 * 64 * cLDK + 2 * 64 * cLDM + 2 * 16 * cLDK) * 4 + 2 * 64 * cKRS * 2;

constexpr int kLT = 512;   // bwd_local_pc: 16 warps
constexpr int kLW = kLT / 32;

template <int VARIANT>
__global__ void __launch_bounds__(kLT, 1)
    bwd_local_pc_kernel(FwdArgs a, BwdArgs g) {
  // every variant but KDA finishes its gain (and the key norm) in a gain kernel
  constexpr bool kGainK = VARIANT != DR_KDA;
  extern __shared__ __align__(16) float smf[];
  float* sW = smf;                   // w [j][c]
  float* sG = sW + 64 * cLDK;        // cumulative log-decay g [j][c]
  float* sMP = sG + 64 * cLDK;       // M_P [i][j]
  float* sML = sMP + 64 * cLDM;      // M_L [i][j]
  float* sWt = sML + 64 * cLDM;      // w~ of block row I [j][c]
  float* sAq = sWt + 64 * cLDK;      // q~ of block row I [16][c]
  float* sAk = sAq + 16 * cLDK;      // k~
  float* sDW = sAk + 16 * cLDK;      // dw, Gram part [j][c]
  uint16_t* sKr = reinterpret_cast<uint16_t*>(sDW + 64 * cLDK);   // raw k, q (bf16) [j][cKRS]
  uint16_t* sQr = sKr + 64 * cKRS;
  __shared__ float s_cr[64], s_qn[64], s_eta[64];
  __shared__ float s_scan[4][128], s_scan2[4][128];   // channel scans: the parts' totals

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NC = (a.T + 63) / 64;
  const long task = blockIdx.x;
  const int bh = (int)(task / NC), c = (int)(task % NC);
  const int b = bh / a.H, h = bh % a.H;
  const int t0 = 64 * c, Cc = min(64, a.T - t0);
  auto bf = [](uint16_t x) { return __uint_as_float(static_cast<uint32_t>(x) << 16); };

  // ---- raw rows (loaded ahead of the copies, stored after them: a store first could
  //      alias the loads), w, log-decay, dP and dR E^T
  constexpr int kRR = 64 * 16 / kLT;
  uint4 rk[kRR], rq[kRR];
#pragma unroll
  for (int r = 0; r < kRR; ++r) {
    const int e = tid + r * kLT, j = e >> 4, c0 = 8 * (e & 15);
    const bool live = j < Cc;
    const long o = tok(a, b, t0 + (live ? j : 0), h) * 128 + c0;
    rk[r] = live ? *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.k) + o) : make_uint4(0u, 0u, 0u, 0u);
    rq[r] = live ? *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + o) : make_uint4(0u, 0u, 0u, 0u);
  }
  for (int e = tid; e < 64 * 32; e += kLT) {
    const int j = e >> 5, c4 = 4 * (e & 31);
    const bool live = j < Cc;
    cpa16(sW + j * cLDK + c4, g.w.Wf + (size_t)task * 8192 + j * 128 + c4);
    cpa16(sG + j * cLDK + c4, a.log_alpha + tok(a, b, t0 + (live ? j : 0), h) * 128 + c4, live ? 16 : 0);
  }
  for (int e = tid; e < 64 * 16; e += kLT) {
    const int i = e >> 4, c4 = 4 * (e & 15);
    cpa16(sMP + i * cLDM + c4, g.w.dP + (size_t)task * 4096 + i * 64 + c4);
    cpa16(sML + i * cLDM + c4, g.w.dL + (size_t)task * 4096 + i * 64 + c4);
  }
  if (tid < 64) s_eta[tid] = (!kGainK && tid < Cc) ? a.eta[tok(a, b, t0 + tid, h)] : 0.f;
  for (int e = tid; e < 64 * 128; e += kLT) sDW[(e >> 7) * cLDK + (e & 127)] = 0.f;
#pragma unroll
  for (int r = 0; r < kRR; ++r) {
    const int e = tid + r * kLT, j = e >> 4, c0 = 8 * (e & 15);
    *reinterpret_cast<uint4*>(sKr + j * cKRS + c0) = rk[r];
    *reinterpret_cast<uint4*>(sQr + j * cKRS + c0) = rq[r];
  }
  cpa_wait_all();
  __syncthreads();
  {   // norms: eight threads per row
    static_assert(kLT == 512, "eight threads per row");
    const int j = tid >> 3, part = tid & 7;
    float kk = 0.f, qq = 0.f;
    for (int c0 = 16 * part; c0 < 16 * part + 16; ++c0) {
      const float x = bf(sKr[j * cKRS + c0]), y = bf(sQr[j * cKRS + c0]);
      kk += x * x;
      qq += y * y;
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      kk += __shfl_xor_sync(0xffffffffu, kk, o);
      qq += __shfl_xor_sync(0xffffffffu, qq, o);
    }
    if (part == 0) {
      s_cr[j] = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
      s_qn[j] = a.q_l2norm ? 1.f / fmaxf(sqrtf(qq), 1e-30f) : 1.f;
    }
  }
  float gl[16];   // cumulative log-decay: four threads per channel, 16 tokens each
  const int sch = tid & 127, spart = tid >> 7;
  {
    float gg = 0.f;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      gg += sG[(16 * spart + q) * cLDK + sch];
      gl[q] = gg;
    }
    s_scan[spart][sch] = gg;
  }
  for (int e = tid; e < 64 * 64; e += kLT) {
    const int i = e >> 6, j = e & 63;
    sMP[i * cLDM + j] = (j <= i) ? sMP[i * cLDM + j] : 0.f;
    sML[i * cLDM + j] = (j < i) ? -sML[i * cLDM + j] : 0.f;
  }
  __syncthreads();
  {
    float off = 0.f;
    for (int p = 0; p < spart; ++p) off += s_scan[p][sch];
#pragma unroll
    for (int q = 0; q < 16; ++q) sG[(16 * spart + q) * cLDK + sch] = gl[q] + off;
  }
  __syncthreads();

  // ---- block rows I = 0..3
  for (int I = 0; I < 4; ++I) {
    const int nJ = 16 * (I + 1), m = 16 * I + 7;
    for (int e = tid; e < nJ * 32; e += kLT) {   // w~ = w e^{g_m(I) - g}, rows j < 16 (I + 1)
      const int j = e >> 5, c4 = 4 * (e & 31);
      const float4 w4 = *reinterpret_cast<const float4*>(sW + j * cLDK + c4);
      const float4 g4 = *reinterpret_cast<const float4*>(sG + j * cLDK + c4);
      const float4 m4 = *reinterpret_cast<const float4*>(sG + m * cLDK + c4);
      *reinterpret_cast<float4*>(sWt + j * cLDK + c4) =
          make_float4(w4.x * __expf(m4.x - g4.x), w4.y * __expf(m4.y - g4.y),
                      w4.z * __expf(m4.z - g4.z), w4.w * __expf(m4.w - g4.w));
    }
    for (int e = tid; e < 16 * 32; e += kLT) {   // q~, k~ of the block's rows
      const int r = e >> 5, c4 = 4 * (e & 31), i = 16 * I + r;
      const float4 g4 = *reinterpret_cast<const float4*>(sG + i * cLDK + c4);
      const float4 m4 = *reinterpret_cast<const float4*>(sG + m * cLDK + c4);
      const uint2 kr = *reinterpret_cast<const uint2*>(sKr + i * cKRS + c4);
      const uint2 qr = *reinterpret_cast<const uint2*>(sQr + i * cKRS + c4);
      const float f[4] = {__expf(g4.x - m4.x), __expf(g4.y - m4.y), __expf(g4.z - m4.z),
                          __expf(g4.w - m4.w)};
      const float kf[4] = {__uint_as_float(kr.x << 16), __uint_as_float(kr.x & 0xFFFF0000u),
                           __uint_as_float(kr.y << 16), __uint_as_float(kr.y & 0xFFFF0000u)};
      const float qf[4] = {__uint_as_float(qr.x << 16), __uint_as_float(qr.x & 0xFFFF0000u),
                           __uint_as_float(qr.y << 16), __uint_as_float(qr.y & 0xFFFF0000u)};
      const float cr = s_cr[i], qn = s_qn[i];
      *reinterpret_cast<float4*>(sAq + r * cLDK + c4) =
          make_float4(qf[0] * qn * f[0], qf[1] * qn * f[1], qf[2] * qn * f[2], qf[3] * qn * f[3]);
      *reinterpret_cast<float4*>(sAk + r * cLDK + c4) =
          make_float4(kf[0] * cr * f[0], kf[1] * cr * f[1], kf[2] * cr * f[2], kf[3] * cr * f[3]);
    }
    __syncthreads();
    {   // dq^_P, dk^_L of the block's 16 rows (warp: columns kCW warp .. + kCW)
      constexpr int kCW = 128 / kLW, kNT = kCW / 8;
      float dq2[kNT][4] = {}, dk2[kNT][4] = {};
      for (int kk = 0; kk <= I; ++kk) {
        mm3x<kNT, 2, false, false>(dq2, sMP + 16 * I * cLDM + 16 * kk, cLDM,
                                   sWt + 16 * kk * cLDK + kCW * warp, cLDK, lane);
        mm3x<kNT, 2, false, false>(dk2, sML + 16 * I * cLDM + 16 * kk, cLDM,
                                   sWt + 16 * kk * cLDK + kCW * warp, cLDK, lane);
      }
      // every raw X_Q / X_K value first (the stores below could alias them); a lane's
      // fragment elements e and e + 1 are adjacent columns of one row: 8-byte accesses
      float2 xqa[kNT][2], xka[kNT][2];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = 16 * I + frag_row(lane, 2 * hh), cc = kCW * warp + 8 * nt + frag_col(lane, 0);
          const long o = tok(a, b, t0 + (i < Cc ? i : 0), h) * 128 + cc;
          xqa[nt][hh] = i < Cc ? *reinterpret_cast<const float2*>(g.dq + o) : make_float2(0.f, 0.f);
          xka[nt][hh] = i < Cc ? *reinterpret_cast<const float2*>(g.dk + o) : make_float2(0.f, 0.f);
        }
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int i = 16 * I + frag_row(lane, 2 * hh), cc0 = kCW * warp + 8 * nt + frag_col(lane, 0);
          if (i < Cc) {
            float oq[2], ok[2];
#pragma unroll
            for (int f = 0; f < 2; ++f) {
              const int cc = cc0 + f;
              const float gi = sG[i * cLDK + cc];
              const float sc = __expf(gi - sG[m * cLDK + cc]), eg = __expf(gi);
              const float dqp = dq2[nt][2 * hh + f] * sc, dkl = dk2[nt][2 * hh + f] * sc;
              const float xq = f ? xqa[nt][hh].y : xqa[nt][hh].x, xk = f ? xka[nt][hh].y : xka[nt][hh].x;
              oq[f] = dqp + eg * xq;
              ok[f] = dkl - eg * xk;
            }
            const long o = tok(a, b, t0 + i, h) * 128 + cc0;
            *reinterpret_cast<float2*>(g.dq + o) = make_float2(oq[0], oq[1]);
            *reinterpret_cast<float2*>(g.dk + o) = make_float2(ok[0], ok[1]);
          }
        }
    }
    // dw of rows j < 16 (I + 1): M_P^T q~ + M_L^T k~ over the block's rows, times e^{g_m(I) - g_j}
    for (int pp = warp; pp < 8 * (I + 1); pp += kLW) {
      const int mt = pp >> 3, nt0 = 2 * (pp & 7);
      float d2[2][4] = {};
      mm3x<2, 2, true, false>(d2, sMP + 16 * I * cLDM + 16 * mt, cLDM, sAq + 8 * nt0, cLDK, lane);
      mm3x<2, 2, true, false>(d2, sML + 16 * I * cLDM + 16 * mt, cLDM, sAk + 8 * nt0, cLDK, lane);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {   // a lane's two adjacent columns as 8-byte accesses
          const int j = 16 * mt + frag_row(lane, 2 * hh), cc = 8 * (nt0 + nt) + frag_col(lane, 0);
          const float2 gm = *reinterpret_cast<const float2*>(sG + m * cLDK + cc);
          const float2 gj = *reinterpret_cast<const float2*>(sG + j * cLDK + cc);
          float2* dp = reinterpret_cast<float2*>(sDW + j * cLDK + cc);
          float2 dv = *dp;
          dv.x += d2[nt][2 * hh] * __expf(gm.x - gj.x);
          dv.y += d2[nt][2 * hh + 1] * __expf(gm.y - gj.y);
          *dp = dv;
        }
    }
    __syncthreads();
  }

  // ---- rows (eight threads per token, 16-byte pieces of the row side by side, two
  //      passes of 32 tokens): dw += e^{G - g} X_W, the column terms of dg, the write
  //      gain and the norms
  for (int pass = 0; pass < 64 * 8 / kLT; ++pass) {
    const int j = (kLT / 8) * pass + (tid >> 3), part = tid & 7;
    const bool live = j < Cc;
    const long o = tok(a, b, t0 + (live ? j : 0), h) * 128;
    const float* xw = g.w.XW + (size_t)task * 8192 + j * 128;
    const float cr = s_cr[j], qn = s_qn[j], eta = s_eta[j];
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float dkh[16], dqh[16], kh[16], qh[16], dwa[16], deta = 0.f, dotk = 0.f, dotq = 0.f;
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const int c0 = 4 * part + 32 * k4;
      const float4 g4 = *reinterpret_cast<const float4*>(sG + j * cLDK + c0);
      const float4 gC4 = *reinterpret_cast<const float4*>(sG + 63 * cLDK + c0);
      const float4 w4 = *reinterpret_cast<const float4*>(sW + j * cLDK + c0);
      const float4 d4 = *reinterpret_cast<const float4*>(sDW + j * cLDK + c0);
      const float4 x4 = live ? *reinterpret_cast<const float4*>(xw + c0) : z4;
      const float4 k4v = live ? *reinterpret_cast<const float4*>(g.dk + o + c0) : z4;
      const float4 q4v = live ? *reinterpret_cast<const float4*>(g.dq + o + c0) : z4;
      const uint2 kr = *reinterpret_cast<const uint2*>(sKr + j * cKRS + c0);
      const uint2 qr = *reinterpret_cast<const uint2*>(sQr + j * cKRS + c0);
      const float gg[4] = {g4.x, g4.y, g4.z, g4.w}, gc[4] = {gC4.x, gC4.y, gC4.z, gC4.w};
      const float ww[4] = {w4.x, w4.y, w4.z, w4.w}, dg4[4] = {d4.x, d4.y, d4.z, d4.w};
      const float xx[4] = {x4.x, x4.y, x4.z, x4.w};
      const float kk[4] = {k4v.x, k4v.y, k4v.z, k4v.w}, qq[4] = {q4v.x, q4v.y, q4v.z, q4v.w};
      const float kf[4] = {__uint_as_float(kr.x << 16), __uint_as_float(kr.x & 0xFFFF0000u),
                           __uint_as_float(kr.y << 16), __uint_as_float(kr.y & 0xFFFF0000u)};
      const float qf[4] = {__uint_as_float(qr.x << 16), __uint_as_float(qr.x & 0xFFFF0000u),
                           __uint_as_float(qr.y << 16), __uint_as_float(qr.y & 0xFFFF0000u)};
      float dwo[4], dgo[4], tgo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int q = 4 * k4 + e;
        const float ew = __expf(gc[e] - gg[e]);
        const float dw = dg4[e] + ew * xx[e];
        tgo[e] = live ? ww[e] * ew * xx[e] : 0.f;   // this token's part of dG_c
        kh[q] = kf[e] * cr;
        qh[q] = qf[e] * qn;
        dkh[q] = kk[e];
        dqh[q] = qq[e];
        if (!kGainK) {
          dkh[q] += eta * dw;
          deta += kh[q] * dw;
        }
        dwo[e] = dw;
        // the token's whole dg: the Gram's row terms and the state terms are
        // q^ . dq^ + k^ . dk^ of the block rows' dq^, dk^ (the Gram part and e^g X_Q,
        // -e^g X_K); kept here for the sums below
        dgo[e] = live ? qh[q] * qq[e] + kh[q] * kk[e] - ww[e] * dg4[e] - ww[e] * ew * xx[e] : 0.f;
        dotk += dkh[q] * kh[q];
        dotq += dqh[q] * qh[q];
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) dwa[4 * k4 + e] = dwo[e];
      *reinterpret_cast<float4*>(sDW + j * cLDK + c0) = make_float4(dgo[0], dgo[1], dgo[2], dgo[3]);
      *reinterpret_cast<float4*>(sWt + j * cLDK + c0) = make_float4(tgo[0], tgo[1], tgo[2], tgo[3]);
    }
    if (kGainK) {   // dL/dw for the gain kernel (after every load of the row above)
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4)
        *reinterpret_cast<float4*>(g.w.DW + (size_t)task * 8192 + j * 128 + 4 * part + 32 * k4) =
            make_float4(dwa[4 * k4], dwa[4 * k4 + 1], dwa[4 * k4 + 2], dwa[4 * k4 + 3]);
    }
#pragma unroll
    for (int o2 = 1; o2 < 8; o2 <<= 1) {
      deta += __shfl_xor_sync(0xffffffffu, deta, o2);
      dotk += __shfl_xor_sync(0xffffffffu, dotk, o2);
      dotq += __shfl_xor_sync(0xffffffffu, dotq, o2);
    }
    if (live) {
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const int c0 = 4 * part + 32 * k4;
        float dq4[4], dk4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int q = 4 * k4 + e;
          dq4[e] = a.q_l2norm ? (dqh[q] - qh[q] * dotq) * qn : dqh[q];
          dk4[e] = a.k_l2norm ? (dkh[q] - kh[q] * dotk) * cr : dkh[q];
        }
        *reinterpret_cast<float4*>(g.dq + o + c0) = make_float4(dq4[0], dq4[1], dq4[2], dq4[3]);
        // the gain kernels' variants keep dk^ of the memory part for them
        if (!kGainK)
          *reinterpret_cast<float4*>(g.dk + o + c0) = make_float4(dk4[0], dk4[1], dk4[2], dk4[3]);
      }
      if (!kGainK && part == 0) g.deta[tok(a, b, t0 + j, h)] = deta;
    }
  }
  __syncthreads();
  // ---- per channel: dG on the last token, then d log alpha = the reverse cumulative
  //      sum (four threads per channel, 16 tokens each; the tokens' parts of dG_c were
  //      left in the w~ buffer by the rows)
  {
    float dg[16], acc = 0.f, dGp = 0.f;
#pragma unroll
    for (int q = 15; q >= 0; --q) {
      const int j = 16 * spart + q;
      if (j < Cc) {
        acc += sDW[j * cLDK + sch];
        dGp += sWt[j * cLDK + sch];
      }
      dg[q] = acc;
    }
    s_scan[spart][sch] = acc;
    s_scan2[spart][sch] = dGp;
    __syncthreads();
    float off = g.w.SS[(size_t)task * 128 + sch];
    for (int p = 0; p < 4; ++p) {
      off += s_scan2[p][sch];
      if (p > spart) off += s_scan[p][sch];
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int j = 16 * spart + q;
      if (j < Cc) sDW[j * cLDK + sch] = dg[q] + off;
    }
  }
  __syncthreads();
  for (int e = tid; e < Cc * 32; e += kLT) {   // d log alpha out (coalesced)
    const int j = e >> 5, c4 = 4 * (e & 31);
    *reinterpret_cast<float4*>(g.dla + tok(a, b, t0 + j, h) * 128 + c4) =
        *reinterpret_cast<const float4*>(sDW + j * cLDK + c4);
  }
}

// ================================================================= pgdn_gain_bwd
// One CTA of 16 warps per chunk, four threads per key channel (16-token parts).  The
// statistic A_t is recomputed forward from its chunk-start value (the forward's
// record), then the tokens are walked backwards (PDN notes Eq. (9)):
//   r = ln max(A, floor) - mu,  B = exp(-ln(x) r / (1 + |r|)),  w = eta B . k^
//   d eta  = sum_i B k^ dw,   dr = -ln(x) B eta k^ dw / (1 + |r|)^2,
//   dA_t = dA + [A > floor] dr / A,   d mu -= [A > floor] dr,
//   d alphaP = sum_i A_{t-1} dA_t,   d betaP = sum_i k^2 dA_t,
//   dk^ += eta B dw + 2 betaP k^ dA_t,   dA <- alphaP dA_t (to token t-1),
// then the key norm.  The walk backwards is per channel (the chain through dA);
// the sums over channels follow per token, a warp per 16 tokens, A_{t-1}
// recomputed from the chunk start.  dA at the row start is dL/dA_0.  PC (PKDA, the
// same statistic with per-channel decay, which the statistic does not involve):
// the chunk-start statistic comes from the per-channel record and the key norms
// are formed here.
// The chain is affine in dA: token t maps dA_t's carry to alphaP_t (dA + y_t) with
// y_t = [A_t > floor] dr_t / A_t free of dA, so a chunk composes to dA_start =
// M dA_end + N per channel.  PHASE 0 (every chunk at once) forms (M, N);
// gain_scan walks each row's maps backwards (dA at every chunk's end, dL/dA_0);
// PHASE 1 (every chunk at once) runs the chunk backwards from it, writes the
// gradients and the chunk's part of dL/dmu.
constexpr int kGT = 512;                 // gain adjoints: four token parts of 16 per channel
constexpr int kGW = kGT / 32;
constexpr int kGainSmemF = 4 * 64 * 128 + 4 * 128 * 4 + 4 * 128;
constexpr int kGainMapSmemF = kGainSmemF;

template <bool PC, int PHASE>
__global__ void __launch_bounds__(kGT, 1) pgdn_gain_bwd_kernel(FwdArgs a, BwdArgs g) {
  extern __shared__ __align__(16) float smf[];
  float* sK = smf;                  // k^ [t][i]
  float* sDW = sK + 64 * 128;       // dL/dw [t][i]
  float* sA = sDW + 64 * 128;       // A_t [t][i], then dA_t
  float* sDK = sA + 64 * 128;       // dL/dk^ [t][i]: the memory part, then the total (PHASE 1)
  float4* sMap = reinterpret_cast<float4*>(sDK + 64 * 128);   // [4 parts][128] part maps
  float* sAs = reinterpret_cast<float*>(sMap + 4 * 128);      // [4 parts][128] A before each part
  __shared__ float s_aP[64], s_bP[64], s_eta[64], s_cr[64], s_mu[kGW];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = tid & 127, part = tid >> 7, t1 = 16 * part;   // channel, tokens t1 .. t1 + 15
  const int NC = (a.T + 63) / 64;
  const size_t ri = blockIdx.x;
  const int bh = (int)(ri / NC), c = (int)(ri % NC), b = bh / a.H, h = bh % a.H;
  const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(a.k);
  const float mu_h = a.mu[h];
  const int t0 = 64 * c, Cc = min(64, a.T - t0);
  float dmu = 0.f;
  if (tid < 64) {
    const bool live = tid < Cc;
    const long ti = tok(a, b, t0 + (live ? tid : 0), h);
    s_aP[tid] = live ? a.alphaP[ti] : 1.f;
    s_bP[tid] = live ? a.betaP[ti] : 0.f;
    s_eta[tid] = live ? a.eta[ti] : 0.f;
    if (!PC) s_cr[tid] = live ? g.w.CR[ri * 64 + tid] : 0.f;
  }
  uint4 rk[64 * 16 / kGT];   // the raw keys, in flight with the copies below
#pragma unroll
  for (int r = 0; r < 64 * 16 / kGT; ++r) {
    const int e = tid + r * kGT, t = e >> 4, c0 = 8 * (e & 15);
    rk[r] = t < Cc ? *reinterpret_cast<const uint4*>(K + tok(a, b, t0 + t, h) * 128 + c0) : make_uint4(0u, 0u, 0u, 0u);
  }
  for (int e = tid; e < 64 * 32; e += kGT) {   // dL/dw and the memory part of dL/dk^
    const int t = e >> 5, c4 = 4 * (e & 31);
    const bool live = t < Cc;
    cpa16(sDW + t * 128 + c4, g.w.DW + ri * 8192 + t * 128 + c4, live ? 16 : 0);
    if (PHASE == 1)
      cpa16(sDK + t * 128 + c4, g.dk + tok(a, b, t0 + (live ? t : 0), h) * 128 + c4, live ? 16 : 0);
  }
  cpa_wait_all();
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 64 * 16 / kGT; ++r) {   // k^ = k cr
    const int e = tid + r * kGT, t = e >> 4, c0 = 8 * (e & 15);
    float f[8];
    unpack8(rk[r], f);
#pragma unroll
    for (int q = 0; q < 8; ++q) sK[t * 128 + c0 + q] = PC ? f[q] : f[q] * s_cr[t];
  }
  __syncthreads();
  if (PC) {   // key norms (warp w: 4 tokens), then k^ = k cr
    for (int tt = 0; tt < 64 / kGW; ++tt) {
      const int t = (64 / kGW) * warp + tt;
      float kk = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float x = sK[t * 128 + lane + 32 * m];
        kk += x * x;
      }
      kk = warp_sum(kk);
      if (lane == 0) s_cr[t] = t < Cc ? (a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f) : 0.f;
    }
    __syncthreads();
    for (int e = tid; e < 64 * 128; e += kGT) sK[e] *= s_cr[e >> 7];
    __syncthreads();
  }
  // the statistic over the chunk from its chunk-start value: each part composes its
  // tokens' affine maps A <- alphaP A + betaP k^2, the earlier parts' maps give its start
  const float A0 =
      PC ? (c == 0 ? (a.aux0 ? a.aux0[(size_t)bh * 128 + i] : 0.f)
                   : reinterpret_cast<const float*>(g.w.rec + ri * g.w.recb + rP0PC)[i])
         : reinterpret_cast<const float*>(g.w.rec + ri * g.w.recb + rAuxF)[256 + i];
  {
    float Pm = 1.f, Pb = 0.f;
    for (int t = t1; t < t1 + 16 && t < Cc; ++t) {
      const float kv = sK[t * 128 + i];
      Pm = s_aP[t] * Pm;
      Pb = fmaf(s_aP[t], Pb, s_bP[t] * kv * kv);
    }
    sMap[part * 128 + i] = make_float4(Pm, Pb, 0.f, 0.f);
    __syncthreads();
    float A = A0;
    for (int q = 0; q < part; ++q) {
      const float4 M = sMap[q * 128 + i];
      A = fmaf(M.x, A, M.y);
    }
    sAs[part * 128 + i] = A;
    for (int t = t1; t < t1 + 16 && t < Cc; ++t) {
      const float kv = sK[t * 128 + i];
      A = s_aP[t] * A + s_bP[t] * kv * kv;
      sA[t * 128 + i] = A;
    }
  }
  // each part's affine map of the adjoint over its tokens, backwards:
  // dA_start = M dA_end + N (token t: dA <- alphaP_t (dA + y_t), y_t = [A_t > floor] dr_t / A_t)
  float M = 1.f, N = 0.f;
  for (int t = min(t1 + 15, Cc - 1); t >= t1; --t) {
    const float A = sA[t * 128 + i];
    const float rr = logf(fmaxf(A, a.log_floor)) - mu_h;
    const float den = 1.f + fabsf(rr);
    const float Bv = expf(-a.ln_x * rr / den);
    const float drr = -a.ln_x * Bv * (s_eta[t] * sK[t * 128 + i] * sDW[t * 128 + i]) / (den * den);
    const float y = A > a.log_floor ? __fdividef(drr, A) : 0.f;
    N = s_aP[t] * (N + y);
    M = s_aP[t] * M;
  }
  __syncthreads();   // every part's forward map read
  sMap[part * 128 + i] = make_float4(M, N, 0.f, 0.f);
  __syncthreads();
  if (PHASE == 0) {   // the chunk's map: the parts' maps composed from the last
    if (part == 0) {
      float Mc = 1.f, Nc = 0.f;
      for (int q = 3; q >= 0; --q) {
        const float4 Q = sMap[q * 128 + i];
        Nc = Q.x * Nc + Q.y;
        Mc = Q.x * Mc;
      }
      g.w.GM[ri * 256 + i] = Mc;
      g.w.GM[ri * 256 + 128 + i] = Nc;
    }
    return;
  }
  // the adjoint at this part's end: the chunk end's value through the later parts' maps
  float dA = g.w.GE[ri * 128 + i];
  for (int q = 3; q > part; --q) {
    const float4 Q = sMap[q * 128 + i];
    dA = Q.x * dA + Q.y;
  }
  // backwards over the part's tokens: per channel only (the chain through dA);
  // dA_t replaces A_t, and B k^ dw replaces dL/dw, for the sums over channels
  for (int t = min(t1 + 15, Cc - 1); t >= t1; --t) {
    const float A = sA[t * 128 + i];
    const float rr = logf(fmaxf(A, a.log_floor)) - mu_h;
    const float den = 1.f + fabsf(rr);
    const float Bv = expf(-a.ln_x * rr / den);
    const float dwv = sDW[t * 128 + i], kv = sK[t * 128 + i], et = s_eta[t];
    const float drr = -a.ln_x * Bv * (et * kv * dwv) / (den * den);
    const bool above = A > a.log_floor;
    const float dAt = dA + (above ? __fdividef(drr, A) : 0.f);
    if (above) dmu -= drr;
    sDK[t * 128 + i] += et * Bv * dwv + 2.f * s_bP[t] * kv * dAt;
    sDW[t * 128 + i] = Bv * kv * dwv;
    sA[t * 128 + i] = dAt;
    dA = s_aP[t] * dAt;
  }
  __syncthreads();
  // per token: d eta = sum B k^ dw, d alphaP = sum A_{t-1} dA_t, d betaP = sum k^2 dA_t,
  // and the key norm (dk = (dk^ - k^ (k^ . dk^)) cr); warp w takes 4 tokens of part
  // w / 4, a lane four channels, A_{t-1} recomputed from the part's start
  {
    const int tw = (64 / kGW) * warp, pw = tw >> 4;
    float Ap[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) Ap[m] = sAs[pw * 128 + lane + 32 * m];
    for (int t = 16 * pw; t < tw && t < Cc; ++t) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float kv = sK[t * 128 + lane + 32 * m];
        Ap[m] = s_aP[t] * Ap[m] + s_bP[t] * kv * kv;
      }
    }
    for (int tt = 0; tt < 64 / kGW; ++tt) {
      const int t = tw + tt;
      if (t >= Cc) break;
      float se = 0.f, sa = 0.f, sb = 0.f, dot = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int ch = lane + 32 * m;
        const float kv = sK[t * 128 + ch], dAt = sA[t * 128 + ch];
        se += sDW[t * 128 + ch];
        sa += Ap[m] * dAt;
        sb += kv * kv * dAt;
        dot += kv * sDK[t * 128 + ch];
        Ap[m] = s_aP[t] * Ap[m] + s_bP[t] * kv * kv;
      }
      se = warp_sum(se);
      sa = warp_sum(sa);
      sb = warp_sum(sb);
      dot = warp_sum(dot);
      if (lane == 0) {
        const long ti = tok(a, b, t0 + t, h);
        g.deta[ti] = se;
        g.daP[ti] = sa;
        g.dbP[ti] = sb;
      }
      const float cr = s_cr[t];
      float* dkrow = g.dk + tok(a, b, t0 + t, h) * 128;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int ch = lane + 32 * m;
        const float v = sDK[t * 128 + ch];
        dkrow[ch] = a.k_l2norm ? (v - sK[t * 128 + ch] * dot) * cr : v;
      }
    }
  }
  dmu = warp_sum(dmu);
  if (lane == 0) s_mu[warp] = dmu;
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
    for (int w = 0; w < kGW; ++w) s += s_mu[w];
    g.w.MU[ri] = s;
  }
}

// ================================================================= kdn_gain_bwd
// Diagonal KDN's write vector is the Kalman gain w = p^ . k^ / (r + sum_c p^ k^2)
// with the predicted variance p^_t = alpha_t^2 p_{t-1} + omega_t and the posterior
// p_t = p^_t / (1 + u_t p^_t), u_t = (mu / r_t) k^_t^2 (KDN notes Eq. (23) and
// section 5).  One CTA of 16 warps per chunk, four threads per key channel (16-token
// parts, each composing its tokens' maps before it walks them): p^ and p are recomputed over the chunk from its chunk-start variance (the
// forward's record), den_t = r_t + sum_c p^ k^2 and c_t = sum_c dw p^ k^ per token,
// then the tokens are walked backwards with the variance adjoint dp (from dL/dp_T):
//   dp^ = dw k^ / den - (c / den^2) k^2 + dp / q^2,  q = 1 + u p^,  du = -dp p^2 / q^2,
//   dk^ += dw p^ / den - 2 (c / den^2) p^ k^ + 2 (mu / r) k^ du,
//   d omega = dp^,  d log alpha += 2 alpha^2 p_{t-1} dp^,  dp <- alpha^2 dp^,
// and per token d r = -c / den^2 - (mu / r^2) sum_c k^2 du and the key norm.  dp at
// the row start is dL/dp_0.
// The chain is affine in dp: token t maps dL/dp_t to dL/dp_{t-1} = alpha^2 (X_t +
// dp / q^2) with X_t = dw k^ / den - (c / den^2) k^2, so each chunk composes to
// dp_start = A dp_end + B per channel.  PHASE 0 (every chunk at once) forms the
// chunk's (A, B); gain_scan walks each row's maps backwards and leaves dp at
// every chunk's end (and dL/dp_0); PHASE 1 (every chunk at once) runs the
// chunk's tokens backwards from it and writes the gradients.
constexpr int kKdnGainSmemF = 6 * 64 * 128 + 4 * 128 * 4;

template <int PHASE>
__global__ void __launch_bounds__(kGT, 1) kdn_gain_bwd_kernel(FwdArgs a, BwdArgs g) {
  extern __shared__ __align__(16) float smf[];
  float* sK = smf;                  // k^ [t][c]
  float* sDW = sK + 64 * 128;       // dL/dw, then k^2 du
  float* sDK = sDW + 64 * 128;      // dL/dk^: the memory part, then the total
  float* sA = sDK + 64 * 128;       // log-decay, then alpha
  float* sPh = sA + 64 * 128;       // omega, then p^
  float* sPo = sPh + 64 * 128;      // p (posterior)
  float4* sMap = reinterpret_cast<float4*>(sPo + 64 * 128);   // [4 parts][128] part maps
  __shared__ float s_r[64], s_mr[64], s_cr[64], s_den[64], s_cc[64], s_iden[64], s_cd2[64];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = tid & 127, part = tid >> 7, t1 = 16 * part;   // channel, tokens t1 .. t1 + 15
  const int NC = (a.T + 63) / 64;
  const size_t ri = blockIdx.x;
  const int bh = (int)(ri / NC), c = (int)(ri % NC), b = bh / a.H, h = bh % a.H;
  const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(a.k);
  const float mu = a.info_scale;
  const int t0 = 64 * c, Cc = min(64, a.T - t0);
  if (tid < 64) {
    s_r[tid] = tid < Cc ? a.r[tok(a, b, t0 + tid, h)] : 1.f;
    s_mr[tid] = mu / s_r[tid];
  }
  uint4 rk[64 * 16 / kGT];   // the raw keys, in flight with the copies below
#pragma unroll
  for (int r = 0; r < 64 * 16 / kGT; ++r) {
    const int e = tid + r * kGT, t = e >> 4, c0 = 8 * (e & 15);
    rk[r] = t < Cc ? *reinterpret_cast<const uint4*>(K + tok(a, b, t0 + t, h) * 128 + c0) : make_uint4(0u, 0u, 0u, 0u);
  }
  for (int e = tid; e < 64 * 32; e += kGT) {
    const int t = e >> 5, c4 = 4 * (e & 31);
    const bool live = t < Cc;
    const long o = tok(a, b, t0 + (live ? t : 0), h) * 128 + c4;
    cpa16(sDW + t * 128 + c4, g.w.DW + ri * 8192 + t * 128 + c4, live ? 16 : 0);
    if (PHASE == 1) cpa16(sDK + t * 128 + c4, g.dk + o, live ? 16 : 0);
    cpa16(sA + t * 128 + c4, a.log_alpha + o, live ? 16 : 0);
    cpa16(sPh + t * 128 + c4, a.omega + o, live ? 16 : 0);
  }
#pragma unroll
  for (int r = 0; r < 64 * 16 / kGT; ++r) {
    const int e = tid + r * kGT, t = e >> 4, c0 = 8 * (e & 15);
    float f[8];
    unpack8(rk[r], f);
#pragma unroll
    for (int q = 0; q < 8; ++q) sK[t * 128 + c0 + q] = f[q];
  }
  cpa_wait_all();
  __syncthreads();
  for (int tt = 0; tt < 64 / kGW; ++tt) {   // key norms: warp w takes 4 tokens
    const int t = (64 / kGW) * warp + tt;
    float kk = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float x = sK[t * 128 + lane + 32 * m];
      kk += x * x;
    }
    kk = warp_sum(kk);
    if (lane == 0) s_cr[t] = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
  }
  __syncthreads();
  // the variance over the chunk from its chunk-start value: each part composes its
  // tokens' maps of (n, d) (p = n / d; M = [[a^2, w], [u a^2, 1 + u w]], u = (mu / r) k^2),
  // the chunk start through the earlier parts' maps gives its start, then it walks
  const float p0 = c == 0 ? (a.aux0 ? a.aux0[(size_t)bh * 128 + i] : 1.f)
                          : reinterpret_cast<const float*>(g.w.rec + ri * g.w.recb + rP0PC)[i];
  {
    float P0 = 1.f, P1 = 0.f, P2 = 0.f, P3 = 1.f;
    for (int t = t1; t < t1 + 16 && t < Cc; ++t) {
      const float kh = sK[t * 128 + i] * s_cr[t];
      sK[t * 128 + i] = kh;
      const float al = __expf(sA[t * 128 + i]), x = al * al, om = sPh[t * 128 + i];
      sA[t * 128 + i] = al;
      const float y = s_mr[t] * kh * kh;
      const float q0 = fmaf(x, P0, om * P2), q1 = fmaf(x, P1, om * P3);
      P2 = fmaf(y, q0, P2);
      P3 = fmaf(y, q1, P3);
      P0 = q0;
      P1 = q1;
      const float sc = __uint_as_float(0x7f000000u - (__float_as_uint(fmaxf(P3, P2)) & 0x7f800000u));
      P0 *= sc;
      P1 *= sc;
      P2 *= sc;
      P3 *= sc;
    }
    sMap[part * 128 + i] = make_float4(P0, P1, P2, P3);
    __syncthreads();
    float n = p0, d = 1.f;
    for (int q = 0; q < part; ++q) {
      const float4 Q = sMap[q * 128 + i];
      const float n1 = fmaf(Q.x, n, Q.y * d), d1 = fmaf(Q.z, n, Q.w * d);
      const float sc = __uint_as_float(0x7f000000u - (__float_as_uint(d1) & 0x7f800000u));
      n = n1 * sc;
      d = d1 * sc;
    }
    float pv = __fdividef(n, d);
    for (int t = t1; t < t1 + 16 && t < Cc; ++t) {
      const float kh = sK[t * 128 + i], al = sA[t * 128 + i];
      const float ph = al * al * pv + sPh[t * 128 + i];
      pv = __fdividef(ph, 1.f + s_mr[t] * kh * kh * ph);
      sPh[t * 128 + i] = ph;
      sPo[t * 128 + i] = pv;
    }
  }
  __syncthreads();
  for (int tt = 0; tt < 64 / kGW; ++tt) {   // den_t and c_t (warp w: 4 tokens)
    const int t = (64 / kGW) * warp + tt;
    if (t >= Cc) break;
    float z = 0.f, cc = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int ch = lane + 32 * m;
      const float kh = sK[t * 128 + ch], ph = sPh[t * 128 + ch];
      z += ph * kh * kh;
      cc += sDW[t * 128 + ch] * ph * kh;
    }
    z = warp_sum(z);
    cc = warp_sum(cc);
    if (lane == 0) {
      const float den = s_r[t] + z;
      s_den[t] = den;
      s_cc[t] = cc;
      s_iden[t] = 1.f / den;
      s_cd2[t] = cc / (den * den);
    }
  }
  __syncthreads();
  // each part's affine map of the adjoint over its tokens, backwards: dp_start = A dp_end + B
  float A = 1.f, Bm = 0.f;
  for (int t = min(t1 + 15, Cc - 1); t >= t1; --t) {
    const float kh = sK[t * 128 + i], ph = sPh[t * 128 + i], al = sA[t * 128 + i];
    const float q1 = 1.f + s_mr[t] * kh * kh * ph;
    const float a2 = al * al, f = a2 * __fdividef(1.f, q1 * q1);
    const float x = sDW[t * 128 + i] * kh * s_iden[t] - s_cd2[t] * kh * kh;
    A = f * A;
    Bm = f * Bm + a2 * x;
  }
  __syncthreads();   // every part's map written over the forward maps' slots below
  sMap[part * 128 + i] = make_float4(A, Bm, 0.f, 0.f);
  __syncthreads();
  if (PHASE == 0) {   // the chunk's map: part 0's of parts 1, 2, 3 in turn
    if (part == 0) {
      float Ac = 1.f, Bc = 0.f;
      for (int q = 3; q >= 0; --q) {
        const float4 M = sMap[q * 128 + i];
        Bc = M.x * Bc + M.y;
        Ac = M.x * Ac;
      }
      g.w.GM[ri * 256 + i] = Ac;
      g.w.GM[ri * 256 + 128 + i] = Bc;
    }
    return;
  }
  // the adjoint at this part's end: the chunk end's value through the later parts' maps
  float dp = g.w.GE[ri * 128 + i];
  for (int q = 3; q > part; --q) {
    const float4 M = sMap[q * 128 + i];
    dp = M.x * dp + M.y;
  }
  // backwards over the part's tokens, per channel (the chain through dp)
  for (int t = min(t1 + 15, Cc - 1); t >= t1; --t) {
    const float kh = sK[t * 128 + i], ph = sPh[t * 128 + i], al = sA[t * 128 + i];
    const float dwv = sDW[t * 128 + i], iden = s_iden[t], cd2 = s_cd2[t], mr = s_mr[t];
    const float q1 = 1.f + mr * kh * kh * ph;
    const float iq2 = __fdividef(1.f, q1 * q1);
    const float dph = dwv * kh * iden - cd2 * kh * kh + dp * iq2;
    const float du = -dp * ph * ph * iq2;
    sDK[t * 128 + i] += dwv * ph * iden - 2.f * cd2 * ph * kh + 2.f * mr * kh * du;
    sDW[t * 128 + i] = kh * kh * du;
    const float prev = t > 0 ? sPo[(t - 1) * 128 + i] : p0;
    sA[t * 128 + i] = dph;                            // d omega
    sPh[t * 128 + i] = 2.f * al * al * prev * dph;    // d log alpha through alpha^2 p
    dp = al * al * dph;
  }
  __syncthreads();
  {   // d omega out, d log alpha updated (coalesced; every load before the stores)
    constexpr int kR = 64 * 32 / kGT;
    float4 la[kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      const int e = tid + kGT * r, t = e >> 5, c4 = 4 * (e & 31);
      la[r] = t < Cc ? *reinterpret_cast<const float4*>(g.dla + tok(a, b, t0 + t, h) * 128 + c4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int r = 0; r < kR; ++r) {
      const int e = tid + kGT * r, t = e >> 5, c4 = 4 * (e & 31);
      if (t >= Cc) continue;
      const long o = tok(a, b, t0 + t, h) * 128 + c4;
      *reinterpret_cast<float4*>(g.domega + o) = *reinterpret_cast<const float4*>(sA + t * 128 + c4);
      const float4 x = *reinterpret_cast<const float4*>(sPh + t * 128 + c4);
      la[r].x += x.x; la[r].y += x.y; la[r].z += x.z; la[r].w += x.w;
      *reinterpret_cast<float4*>(g.dla + o) = la[r];
    }
  }
  for (int tt = 0; tt < 64 / kGW; ++tt) {   // d r and the key norm, warp w: 4 tokens
    const int t = (64 / kGW) * warp + tt;
    if (t >= Cc) break;
    float su = 0.f, dot = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int ch = lane + 32 * m;
      su += sDW[t * 128 + ch];
      dot += sK[t * 128 + ch] * sDK[t * 128 + ch];
    }
    su = warp_sum(su);
    dot = warp_sum(dot);
    const float rt = s_r[t], den = s_den[t];
    if (lane == 0) g.dr[tok(a, b, t0 + t, h)] = -s_cc[t] / (den * den) - mu / (rt * rt) * su;
    const float cr = s_cr[t];
    float* dkrow = g.dk + tok(a, b, t0 + t, h) * 128;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int ch = lane + 32 * m;
      const float v = sDK[t * 128 + ch];
      dkrow[ch] = a.k_l2norm ? (v - sK[t * 128 + ch] * dot) * cr : v;
    }
  }
}

// Each row's chunk maps in reverse chunk order (one thread per channel, or one
// per row for a scalar adjoint, nch = 1): the adjoint at every chunk's end, from
// dL/d(final) (0 when absent), and at the row start dL/d(initial).
__global__ void gain_scan_kernel(FwdArgs a, BwdArgs g, int nch) {
  const int bh = blockIdx.x, i = threadIdx.x;
  if (i >= nch) return;
  const int NC = (a.T + 63) / 64;
  float dp = g.daux_T ? g.daux_T[(size_t)bh * nch + i] : 0.f;
  for (int c = NC - 1; c >= 0; --c) {
    const size_t ri = (size_t)bh * NC + c;
    g.w.GE[ri * 128 + i] = dp;
    dp = g.w.GM[ri * 256 + i] * dp + g.w.GM[ri * 256 + 128 + i];
  }
  if (g.daux0) g.daux0[(size_t)bh * nch + i] = dp;
}

// ================================================================= ikdn_gain_bwd
// Isotropic KDN keeps one variance b per head: b^_t = abar_t b_{t-1} + omega_t with
// abar_t = mean_c alpha_tc^2, w_t = beta_t k^_t, beta = b^ / (r + b^ s), s = ||k^||^2,
// b_t = b^ / (1 + u b^), u = mu s / (dk r) (KDN notes Eq. (40)).  One CTA per chunk:
// per token (in parallel) s, abar and d beta = k^ . dw; the
// scalar chain over the chunk's tokens (four lanes of warp 0, a 16-token part each
// composing its tokens' maps before it walks; b^ recomputed from the chunk-start
// variance of the record) with db (from dL/db_T):
//   db^ = d beta r / den^2 + db / q^2,  q = 1 + u b^,  du = -db b^2 / q^2,  den = r + b^ s,
//   d omega = db^,  db <- abar db^;
// then per (token, channel): dk^ += (b^ / den) dw + 2 ds k^ with
// ds = -d beta b^2 / den^2 + du mu / (dk r),  d r = -d beta b^ / den^2 - du mu s / (dk r^2),
// d log alpha += 2 alpha^2 b_{t-1} db^ / dk, and the key norm.  db at the row start
// is dL/db_0.  The chain is affine in db (db <- abar (d beta r / den^2 + db / q^2)),
// so, as for Diagonal KDN, PHASE 0 forms each chunk's map (M, N), gain_scan (one
// thread per row) the value at every chunk's end and PHASE 1 the gradients, all
// chunks at once.
constexpr int kIkdnGainSmemF = 3 * 64 * 128;

template <int PHASE>
__global__ void __launch_bounds__(kGT, 1) ikdn_gain_bwd_kernel(FwdArgs a, BwdArgs g) {
  extern __shared__ __align__(16) float smf[];
  float* sK = smf;                  // k^ [t][c]
  float* sDW = sK + 64 * 128;       // dL/dw [t][c]
  float* sA = sDW + 64 * 128;       // log-decay [t][c], then alpha^2
  __shared__ float s_r[64], s_om[64], s_cr[64], s_s[64], s_ab[64], s_db[64];
  __shared__ float s_bh[64], s_prev[64], s_dbh[64], s_du[64];
  const int i = threadIdx.x, warp = i >> 5, lane = i & 31;
  const int NC = (a.T + 63) / 64;
  const size_t ri = blockIdx.x;
  const int bh = (int)(ri / NC), c = (int)(ri % NC), b = bh / a.H, h = bh % a.H;
  const __nv_bfloat16* K = static_cast<const __nv_bfloat16*>(a.k);
  const float mu = a.info_scale;
  {
    const int t0 = 64 * c, Cc = min(64, a.T - t0);
    if (i < 64) {
      const bool live = i < Cc;
      const long ti = tok(a, b, t0 + (live ? i : 0), h);
      s_r[i] = live ? a.r[ti] : 1.f;
      s_om[i] = live ? a.omega[ti] : 0.f;
    }
    uint4 rk[64 * 16 / kGT];   // the raw keys, in flight with the copies below
#pragma unroll
    for (int r = 0; r < 64 * 16 / kGT; ++r) {
      const int e = i + r * kGT, t = e >> 4, c0 = 8 * (e & 15);
      rk[r] = t < Cc ? *reinterpret_cast<const uint4*>(K + tok(a, b, t0 + t, h) * 128 + c0) : make_uint4(0u, 0u, 0u, 0u);
    }
    for (int e = i; e < 64 * 32; e += kGT) {
      const int t = e >> 5, c4 = 4 * (e & 31);
      const bool live = t < Cc;
      const long o = tok(a, b, t0 + (live ? t : 0), h) * 128 + c4;
      cpa16(sDW + t * 128 + c4, g.w.DW + ri * 8192 + t * 128 + c4, live ? 16 : 0);
      cpa16(sA + t * 128 + c4, a.log_alpha + o, live ? 16 : 0);
    }
#pragma unroll
    for (int r = 0; r < 64 * 16 / kGT; ++r) {
      const int e = i + r * kGT, t = e >> 4, c0 = 8 * (e & 15);
      float f[8];
      unpack8(rk[r], f);
#pragma unroll
      for (int q = 0; q < 8; ++q) sK[t * 128 + c0 + q] = f[q];
    }
    cpa_wait_all();
    __syncthreads();
    for (int tt = 0; tt < 64 / kGW; ++tt) {   // per token: norm, s, abar, d beta (warp w: 4 tokens)
      const int t = (64 / kGW) * warp + tt;
      float kk = 0.f, a2 = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int ch = lane + 32 * m;
        const float x = sK[t * 128 + ch], al = expf(sA[t * 128 + ch]);
        kk += x * x;
        a2 += al * al;
        sA[t * 128 + ch] = al * al;
      }
      kk = warp_sum(kk);
      a2 = warp_sum(a2);
      const float cr = a.k_l2norm ? 1.f / fmaxf(sqrtf(kk), 1e-30f) : 1.f;
      float kd = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int ch = lane + 32 * m;
        const float kh = sK[t * 128 + ch] * cr;
        sK[t * 128 + ch] = kh;
        kd += kh * sDW[t * 128 + ch];
      }
      kd = warp_sum(kd);
      if (lane == 0) {
        s_cr[t] = t < Cc ? cr : 0.f;
        s_s[t] = kk * cr * cr;
        s_ab[t] = a2 * (1.f / 128.f);
        s_db[t] = kd;
      }
    }
    __syncthreads();
    if (warp == 0) {   // the chunk's variances forward, then the chain backwards, on
                       // lanes 0-3 (a 16-token part each): every part composes its
                       // tokens' maps, the earlier (later) parts' maps give its start
      const int part = lane & 3, t1 = 16 * part, t2 = min(t1 + 16, Cc);
      const float b0 = c == 0 ? (a.aux0 ? a.aux0[bh] : 1.f)
                              : reinterpret_cast<const float*>(g.w.rec + ri * g.w.recb + rP0PC)[0];
      // (n, d) -> [[ab, om], [u ab, 1 + u om]] (n, d), b = n / d, u = mu s / (dk r)
      float P0 = 1.f, P1 = 0.f, P2 = 0.f, P3 = 1.f;
      for (int t = t1; t < t2; ++t) {
        const float x = s_ab[t], om = s_om[t], y = mu * s_s[t] / (128.f * s_r[t]);
        const float q0 = fmaf(x, P0, om * P2), q1 = fmaf(x, P1, om * P3);
        P2 = fmaf(y, q0, P2);
        P3 = fmaf(y, q1, P3);
        P0 = q0;
        P1 = q1;
        const float sc = __uint_as_float(0x7f000000u - (__float_as_uint(fmaxf(P3, P2)) & 0x7f800000u));
        P0 *= sc;
        P1 *= sc;
        P2 *= sc;
        P3 *= sc;
      }
      float n = b0, d = 1.f;
      for (int q = 0; q < 3; ++q) {
        const float Q0 = __shfl_sync(0xffffffffu, P0, q), Q1 = __shfl_sync(0xffffffffu, P1, q);
        const float Q2 = __shfl_sync(0xffffffffu, P2, q), Q3 = __shfl_sync(0xffffffffu, P3, q);
        if (q < part) {
          const float n1 = fmaf(Q0, n, Q1 * d), d1 = fmaf(Q2, n, Q3 * d);
          const float sc = __uint_as_float(0x7f000000u - (__float_as_uint(d1) & 0x7f800000u));
          n = n1 * sc;
          d = d1 * sc;
        }
      }
      float bv = n / d;
      for (int t = t1; t < t2 && lane < 4; ++t) {
        s_prev[t] = bv;
        const float bhat = s_ab[t] * bv + s_om[t];
        s_bh[t] = bhat;
        bv = bhat / (1.f + mu * s_s[t] / (128.f * s_r[t]) * bhat);
      }
      // each part's affine map of the adjoint over its tokens, backwards
      float M = 1.f, N = 0.f;
      __syncwarp();
      for (int t = t2 - 1; t >= t1; --t) {
        const float bhat = s_bh[t], rt = s_r[t], st = s_s[t];
        const float den = rt + bhat * st, q1 = 1.f + mu * st / (128.f * rt) * bhat;
        const float iq2 = 1.f / (q1 * q1);
        N = s_ab[t] * (s_db[t] * rt / (den * den) + N * iq2);
        M = s_ab[t] * iq2 * M;
      }
      const float Ms[4] = {__shfl_sync(0xffffffffu, M, 0), __shfl_sync(0xffffffffu, M, 1),
                           __shfl_sync(0xffffffffu, M, 2), __shfl_sync(0xffffffffu, M, 3)};
      const float Ns[4] = {__shfl_sync(0xffffffffu, N, 0), __shfl_sync(0xffffffffu, N, 1),
                           __shfl_sync(0xffffffffu, N, 2), __shfl_sync(0xffffffffu, N, 3)};
      if (PHASE == 0) {   // the chunk's affine map db_start = M db_end + N
        if (lane == 0) {
          float Mc = 1.f, Nc = 0.f;
          for (int q = 3; q >= 0; --q) {
            Nc = Ms[q] * Nc + Ns[q];
            Mc = Ms[q] * Mc;
          }
          g.w.GM[ri * 256] = Mc;
          g.w.GM[ri * 256 + 128] = Nc;
        }
      } else if (lane < 4) {
        float db = g.w.GE[ri * 128];   // the adjoint at the chunk end, then at this part's
        for (int q = 3; q > part; --q) db = Ms[q] * db + Ns[q];
        for (int t = t2 - 1; t >= t1; --t) {
          const float bhat = s_bh[t], rt = s_r[t], st = s_s[t];
          const float den = rt + bhat * st, q1 = 1.f + mu * st / (128.f * rt) * bhat;
          const float iq2 = 1.f / (q1 * q1);
          const float dbh = s_db[t] * rt / (den * den) + db * iq2;
          s_du[t] = -db * bhat * bhat * iq2;
          s_dbh[t] = dbh;
          db = s_ab[t] * dbh;
        }
      }
    }
    __syncthreads();
    if (PHASE == 0) return;
    constexpr int kTW = 64 / kGW;   // tokens per warp
    float xk8[kTW][4], xl8[kTW][4];
#pragma unroll
    for (int tt = 0; tt < kTW; ++tt) {   // per (token, channel), warp w: tokens kTW w .. + kTW - 1
      const int t = kTW * warp + tt;
      if (t >= Cc) continue;
      if (tt == 0) {   // the warp's tokens' dk^ and d log alpha rows, before any store
#pragma unroll
        for (int u = 0; u < kTW; ++u) {
          const int tu = t + u;
          const long ou = tok(a, b, t0 + (tu < Cc ? tu : 0), h) * 128;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            xk8[u][m] = tu < Cc ? g.dk[ou + lane + 32 * m] : 0.f;
            xl8[u][m] = tu < Cc ? g.dla[ou + lane + 32 * m] : 0.f;
          }
        }
      }
      const float bhat = s_bh[t], rt = s_r[t], st = s_s[t], dbt = s_db[t], du = s_du[t];
      const float den = rt + bhat * st;
      const float ds = -dbt * bhat * bhat / (den * den) + du * mu / (128.f * rt);
      const long tt_ = tok(a, b, t0 + t, h);
      if (lane == 0) {
        g.domega[tt_] = s_dbh[t];
        g.dr[tt_] = -dbt * bhat / (den * den) - du * mu * st / (128.f * rt * rt);
      }
      const float fa = 2.f * s_prev[t] * s_dbh[t] / 128.f;
      float dkh[4], dot = 0.f;
      float* dkrow = g.dk + tt_ * 128;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int ch = lane + 32 * m;
        const float kh = sK[t * 128 + ch];
        dkh[m] = xk8[tt][m] + (bhat / den) * sDW[t * 128 + ch] + 2.f * ds * kh;
        dot += kh * dkh[m];
        g.dla[tt_ * 128 + ch] = xl8[tt][m] + fa * sA[t * 128 + ch];
      }
      dot = warp_sum(dot);
      const float cr = s_cr[t];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int ch = lane + 32 * m;
        dkrow[ch] = a.k_l2norm ? (dkh[m] - sK[t * 128 + ch] * dot) * cr : dkh[m];
      }
    }
  }
}

// dL/dmu_h: the chunks' parts summed over the batch and the chunks in order
__global__ void pgdn_dmu_kernel(FwdArgs a, BwdArgs g) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= a.H) return;
  const int NC = (a.T + 63) / 64;
  float s = 0.f;
  for (int b = 0; b < a.B; ++b)
    for (int c = 0; c < NC; ++c) s += g.w.MU[((size_t)b * a.H + h) * NC + c];
  g.dmu[h] = s;
}

}  // namespace

bool chunk_bwd_supported(int variant, int dtype, int dk, int dv, int chunk) {
  return (variant == DR_GDN || variant == DR_KLA || variant == DR_PGDN || variant == DR_KDA ||
          variant == DR_KDN || variant == DR_PKDA || variant == DR_IKDN) &&
         dtype == DR_BF16 && dk == 128 && dv == 128 && chunk == 64;
}

size_t chunk_bwd_workspace_bytes(int variant, int B, int T, int H) {
  const long n = (long)B * H * ((T + 63) / 64);
  return bwd_layout(nullptr, n, B * H, bwd_mode(variant), nullptr);
}

cudaError_t launch_chunk_bwd(const FwdArgs& fa, const void* d_out, const float* dS_final,
                             const dr_grads& gr, void* workspace, cudaStream_t st) {
  const long n = (long)fa.B * fa.H * ((fa.T + 63) / 64);
  const bool pg = fa.variant == DR_PGDN;
  const int mode = bwd_mode(fa.variant);
  const bool pc = mode >= BW_PC;
  BwdArgs g{d_out,      dS_final,    gr.dq,      gr.dk,      gr.dv,     gr.d_log_alpha,
            gr.d_eta,   gr.d_init_state, gr.d_alphaP, gr.d_betaP, gr.d_mu, gr.d_aux_init,
            gr.d_aux_final, gr.d_omega, gr.d_r, bwd_ws(workspace, n, fa.B * fa.H, mode)};
  // the forward again: the records, the state at every chunk start and E (no
  // output, no final state)
  FwdArgs a = fa;
  a.out = nullptr;
  a.S = nullptr;
  a.aux = nullptr;
  a.check_finite = 0;
  a.save_S = g.w.S;
  a.save_E = g.w.E;
  if (pc) a.save_W = g.w.Wf;
  cudaError_t e = pc ? launch_kdn_split(a, DR_BF16, workspace, st) : launch_chunk_tc_split(a, workspace, st);
  if (e != cudaSuccess) return e;
  const size_t s_smem = kStateSmem,
               l_smem = kLocalSmem, p_smem = (size_t)kGainSmemF * 4,
               pm_smem = (size_t)kGainMapSmemF * 4;
  if ((e = cudaFuncSetAttribute(bwd_carry_tc_kernel<false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCarryTcSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_carry_tc_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCarryTcSmemPG)) !=
          cudaSuccess ||

      (e = cudaFuncSetAttribute(bwd_carry_tc_pc_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCarryPcSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_local_pc_kernel<DR_KDA>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kPcLocalSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_local_pc_kernel<DR_KDN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kPcLocalSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(kdn_gain_bwd_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kKdnGainSmemF * 4)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(kdn_gain_bwd_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kKdnGainSmemF * 4)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_local_kernel<DR_PGDN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l_smem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(pgdn_gain_bwd_kernel<false, 0>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pm_smem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(pgdn_gain_bwd_kernel<false, 1>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p_smem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(pgdn_gain_bwd_kernel<true, 0>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pm_smem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(pgdn_gain_bwd_kernel<true, 1>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p_smem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_local_pc_kernel<DR_PKDA>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kPcLocalSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_local_pc_kernel<DR_IKDN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kPcLocalSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(ikdn_gain_bwd_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kIkdnGainSmemF * 4)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(ikdn_gain_bwd_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kIkdnGainSmemF * 4)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)s_smem)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_local_kernel<DR_GDN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l_smem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(bwd_local_kernel<DR_KLA>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l_smem)) !=
          cudaSuccess)
    return e;
  if (pg)
    bwd_carry_tc_kernel<true><<<fa.B * fa.H * 2, kBwdThreads, kCarryTcSmemPG, st>>>(fa, g);
  else if (pc)
    bwd_carry_tc_pc_kernel<<<fa.B * fa.H * 2, kBwdThreads, kCarryPcSmem, st>>>(fa, g);
  else
    bwd_carry_tc_kernel<false><<<fa.B * fa.H * 2, kBwdThreads, kCarryTcSmem, st>>>(fa, g);
  const int nsm = bwd_sm_count();
  if (nsm <= 0) return cudaErrorInvalidValue;
  bwd_state_kernel<<<(unsigned)(n < nsm ? n : nsm), kStateThreads, s_smem, st>>>(fa, g, n);
  const unsigned lgrid = (unsigned)(n < nsm ? n : nsm);
  if (fa.variant == DR_KDA) {
    bwd_local_pc_kernel<DR_KDA><<<(unsigned)n, kLT, kPcLocalSmem, st>>>(fa, g);
  } else if (fa.variant == DR_KDN) {
    bwd_local_pc_kernel<DR_KDN><<<(unsigned)n, kLT, kPcLocalSmem, st>>>(fa, g);
    kdn_gain_bwd_kernel<0><<<(unsigned)n, kGT, kKdnGainSmemF * 4, st>>>(fa, g);
    gain_scan_kernel<<<fa.B * fa.H, 128, 0, st>>>(fa, g, 128);
    kdn_gain_bwd_kernel<1><<<(unsigned)n, kGT, kKdnGainSmemF * 4, st>>>(fa, g);
  } else if (fa.variant == DR_PKDA) {
    bwd_local_pc_kernel<DR_PKDA><<<(unsigned)n, kLT, kPcLocalSmem, st>>>(fa, g);
    pgdn_gain_bwd_kernel<true, 0><<<(unsigned)n, kGT, pm_smem, st>>>(fa, g);
    gain_scan_kernel<<<fa.B * fa.H, 128, 0, st>>>(fa, g, 128);
    pgdn_gain_bwd_kernel<true, 1><<<(unsigned)n, kGT, p_smem, st>>>(fa, g);
    pgdn_dmu_kernel<<<(fa.H + 127) / 128, 128, 0, st>>>(fa, g);
  } else if (fa.variant == DR_IKDN) {
    bwd_local_pc_kernel<DR_IKDN><<<(unsigned)n, kLT, kPcLocalSmem, st>>>(fa, g);
    ikdn_gain_bwd_kernel<0><<<(unsigned)n, kGT, kIkdnGainSmemF * 4, st>>>(fa, g);
    gain_scan_kernel<<<fa.B * fa.H, 32, 0, st>>>(fa, g, 1);
    ikdn_gain_bwd_kernel<1><<<(unsigned)n, kGT, kIkdnGainSmemF * 4, st>>>(fa, g);
  } else if (fa.variant == DR_KLA) {
    bwd_local_kernel<DR_KLA><<<lgrid, kBwdThreads, l_smem, st>>>(fa, g, n);
  } else if (pg) {
    bwd_local_kernel<DR_PGDN><<<lgrid, kBwdThreads, l_smem, st>>>(fa, g, n);
    pgdn_gain_bwd_kernel<false, 0><<<(unsigned)n, kGT, pm_smem, st>>>(fa, g);
    gain_scan_kernel<<<fa.B * fa.H, 128, 0, st>>>(fa, g, 128);
    pgdn_gain_bwd_kernel<false, 1><<<(unsigned)n, kGT, p_smem, st>>>(fa, g);
    pgdn_dmu_kernel<<<(fa.H + 127) / 128, 128, 0, st>>>(fa, g);
  } else {
    bwd_local_kernel<DR_GDN><<<lgrid, kBwdThreads, l_smem, st>>>(fa, g, n);
  }
  return cudaGetLastError();
}

}  // namespace dr
