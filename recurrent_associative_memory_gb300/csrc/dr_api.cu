// dr_api.cu — the extern "C" entry points of libdr: argument checks, path
// selection and launches.  No device memory is allocated here; the only
// library-owned device storage is the sticky status word below.
#include <math.h>
#include <stdint.h>

#include "dr_common.cuh"

namespace dr {

__device__ int g_status = 0;
__device__ unsigned long long g_chain_wait_ns = 2000000000ull;
__device__ long long g_chain_withhold = -1;

cudaError_t launch_decode(const FwdArgs& a, int dtype, cudaStream_t st);
cudaError_t launch_chunk_simt(const FwdArgs& a, int dtype, cudaStream_t st);
cudaError_t launch_chunk_tc(const FwdArgs& a, cudaStream_t st);
bool chunk_tc_supported(int variant, int dtype, int dk, int dv, int chunk);
cudaError_t launch_chunk_tc_ws(const FwdArgs& a, cudaStream_t st);
bool chunk_tc_ws_supported(int variant, int dtype, int dk, int dv, int chunk);
cudaError_t launch_chunk_tc_split(const FwdArgs& a, void* workspace, cudaStream_t st);
bool chunk_tc_split_supported(int variant, int dtype, int dk, int dv, int chunk);
size_t chunk_tc_split_workspace_bytes(int variant, int B, int T, int H);
cudaError_t launch_kdn_split(const FwdArgs& a, int dtype, void* workspace, cudaStream_t st);
cudaError_t launch_kalman(const FwdArgs& a, int dtype, cudaStream_t st);
bool kdn_split_supported(int variant, int dtype, int dk, int dv, int chunk);
size_t kdn_split_workspace_bytes(int B, int T, int H);
bool chunk_bwd_supported(int variant, int dtype, int dk, int dv, int chunk);
size_t chunk_bwd_workspace_bytes(int variant, int B, int T, int H);
cudaError_t launch_chunk_bwd(const FwdArgs& fa, const void* d_out, const float* dS_final,
                             const dr_grads& g, void* workspace, cudaStream_t st);

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dim_ok(int d) { return d == 64 || d == 128; }

// Pointers the variant needs, shared by the forward and the decode step.
int check_gates(const dr_params* gp, int variant) {
  switch (variant) {
    case DR_GDN:
    case DR_KLA:
    case DR_KDA:
      if (!gp->eta) return DR_ERR_NULL;
      return DR_OK;
    case DR_PGDN:
    case DR_PKDA:
      if (!gp->eta || !gp->alphaP || !gp->betaP || !gp->mu) return DR_ERR_NULL;
      if (!(gp->x > 1.f) || !(gp->log_floor > 0.f)) return DR_ERR_ARG;
      return DR_OK;
    case DR_KDN:
    case DR_IKDN:
    case DR_EKDN:
      if (!gp->omega || !gp->r) return DR_ERR_NULL;
      if (!(gp->info_scale >= 0.f)) return DR_ERR_ARG;
      return DR_OK;
    default:
      return DR_ERR_UNSUPPORTED;
  }
}

FwdArgs make_args(const void* q, const void* k, const void* v, const float* log_alpha,
                  const dr_params* gp, int variant, float eps, int B, int T, int H, int dk,
                  int dv, int chunk) {
  FwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.log_alpha = log_alpha;
  a.eta = gp->eta;
  a.alphaP = gp->alphaP;
  a.betaP = gp->betaP;
  a.mu = gp->mu;
  a.omega = gp->omega;
  a.r = gp->r;
  a.B = B;
  a.T = T;
  a.H = H;
  a.dk = dk;
  a.dv = dv;
  a.chunk = chunk;
  a.variant = variant;
  a.q_l2norm = gp->q_l2norm ? 1 : 0;
  a.k_l2norm = gp->k_l2norm ? 1 : 0;
  a.check_finite = gp->check_finite ? 1 : 0;
  a.eps = eps;
  a.ln_x = (variant == DR_PGDN || variant == DR_PKDA) ? logf(gp->x) : 0.f;
  a.log_floor = gp->log_floor;
  a.info_scale = gp->info_scale;
  return a;
}

}  // namespace
}  // namespace dr

using namespace dr;

extern "C" {

void dr_params_init(dr_params* p) {
  if (!p) return;
  *p = dr_params{};
  p->dtype = DR_BF16;
  p->x = 1.5f;
  p->log_floor = 1e-12f;
  p->info_scale = 1.f;
}

const char* dr_status_string(int s) {
  switch (s) {
    case DR_OK: return "ok";
    case DR_ERR_NULL: return "a required pointer is NULL";
    case DR_ERR_SHAPE: return "unsupported size (B,T,H >= 1; dk,dv in {64,128}; chunk in {16,32,64,128})";
    case DR_ERR_DTYPE: return "dtype must be DR_FP32 or DR_BF16";
    case DR_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case DR_ERR_WORKSPACE: return "workspace missing or too small";
    case DR_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case DR_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    case DR_ERR_NONFINITE: return "non-finite value in an output or state";
    case DR_ERR_UNSUPPORTED: return "variant or option combination not supported";
    case DR_ERR_ARG: return "a scalar argument is out of range";
    default: return "unknown status";
  }
}

size_t dr_chunk_fwd_workspace_bytes(int variant, int dtype, int B, int T, int H, int dk, int dv,
                                    int chunk) {
  if (B < 1 || T < 1 || H < 1) return 0;
  // only the two-phase tensor-core path uses a workspace: one record per chunk
  if (chunk_tc_split_supported(variant, dtype, dk, dv, chunk))
    return chunk_tc_split_workspace_bytes(variant, B, T, H);
  if (kdn_split_supported(variant, dtype, dk, dv, chunk)) return kdn_split_workspace_bytes(B, T, H);
  return 0;
}

const char* dr_chunk_fwd_path(int variant, int dtype, int dk, int dv, int chunk) {
  if (variant == DR_EKDN) return "kalman";
  if (chunk_tc_split_supported(variant, dtype, dk, dv, chunk)) return "tc_split";
  if (kdn_split_supported(variant, dtype, dk, dv, chunk))
    return dtype == DR_BF16 ? "tc_pc_split" : "simt_split";
  if (chunk_tc_ws_supported(variant, dtype, dk, dv, chunk)) return "tc_ws";
  return chunk_tc_supported(variant, dtype, dk, dv, chunk) ? "tc" : "simt";
}

int dr_chunk_fwd(const void* q, const void* k, const void* v, const float* log_alpha,
                 const dr_params* gp, int variant, float eps, const float* init_state,
                 void* out, float* final_state, int B, int T, int H, int dk, int dv, int chunk,
                 dr_stream_t stream) {
  if (!gp || !q || !k || !v || !log_alpha || !out) return DR_ERR_NULL;
  if (gp->dtype != DR_FP32 && gp->dtype != DR_BF16) return DR_ERR_DTYPE;
  if (B < 1 || T < 1 || H < 1 || !dim_ok(dk) || !dim_ok(dv)) return DR_ERR_SHAPE;
  if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128) return DR_ERR_SHAPE;
  if ((long long)B * T * H * (dk > dv ? dk : dv) >= (1LL << 40)) return DR_ERR_SHAPE;
  if (!(eps >= 0.f)) return DR_ERR_ARG;
  int st = check_gates(gp, variant);
  if (st != DR_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(init_state) || !aligned16(final_state) || !aligned16(log_alpha))
    return DR_ERR_ALIGN;
  if ((variant == DR_KDN || variant == DR_EKDN) && !aligned16(gp->omega))
    return DR_ERR_ALIGN;   // copied in 16-byte pieces
  // per-channel log-decay is copied in 16-byte pieces too (checked above)

  FwdArgs a = make_args(q, k, v, log_alpha, gp, variant, eps, B, T, H, dk, dv, chunk);
  a.S0 = init_state;
  a.S = final_state;
  a.aux0 = gp->aux_init;
  a.aux = gp->aux_final;
  a.out = out;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  const bool kdn_split = kdn_split_supported(variant, gp->dtype, dk, dv, chunk);
  const size_t need = chunk_tc_split_supported(variant, gp->dtype, dk, dv, chunk)
                          ? chunk_tc_split_workspace_bytes(variant, B, T, H)
                          : (kdn_split ? kdn_split_workspace_bytes(B, T, H) : 0);
  const bool split = need > 0 && gp->workspace != nullptr;
  if (split && gp->workspace_bytes < need) return DR_ERR_WORKSPACE;
  if (split && (reinterpret_cast<uintptr_t>(gp->workspace) & 255u)) return DR_ERR_ALIGN;
  if (split && kdn_split)
    err = launch_kdn_split(a, gp->dtype, gp->workspace, s);   // per-channel decay: CUDA-core two phases
  else if (split)
    err = launch_chunk_tc_split(a, gp->workspace, s);   // GDN / KLA / PGDN: prep on every SM, then the carry
  else if (chunk_tc_ws_supported(variant, gp->dtype, dk, dv, chunk))
    err = launch_chunk_tc_ws(a, s);          // GDN / KLA: warp-specialised tensor-core kernel
  else if (chunk_tc_supported(variant, gp->dtype, dk, dv, chunk))
    err = launch_chunk_tc(a, s);             // PGDN: phase-sequential tensor-core kernel
  else if (variant == DR_EKDN)
    err = launch_kalman(a, gp->dtype, s);   // exact Kalman: token by token
  else
    err = launch_chunk_simt(a, gp->dtype, s);
  return err == cudaSuccess ? DR_OK : DR_ERR_CUDA;
}

int dr_decode_step(const void* q, const void* k, const void* v, const float* log_alpha,
                   const dr_params* gp, int variant, float eps, float* state, float* aux_state,
                   void* out, int B, int H, int dk, int dv, dr_stream_t stream) {
  if (!gp || !q || !k || !v || !log_alpha || !state || !out) return DR_ERR_NULL;
  if (gp->dtype != DR_FP32 && gp->dtype != DR_BF16) return DR_ERR_DTYPE;
  if (B < 1 || H < 1 || !dim_ok(dk) || !dim_ok(dv)) return DR_ERR_SHAPE;
  if (!(eps >= 0.f)) return DR_ERR_ARG;
  int st = check_gates(gp, variant);
  if (st != DR_OK) return st;
  if ((variant == DR_PGDN || variant == DR_KDN || variant == DR_PKDA || variant == DR_IKDN ||
       variant == DR_EKDN) &&
      !aux_state)
    return DR_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(state) || !aligned16(aux_state))
    return DR_ERR_ALIGN;
  FwdArgs a = make_args(q, k, v, log_alpha, gp, variant, eps, B, 1, H, dk, dv, 0);
  a.S = state;
  a.aux = aux_state;
  a.out = out;
  cudaError_t err;
  if (variant == DR_EKDN) {   // the exact filter's step: one CTA per head, S and P in place
    a.S0 = state;
    a.aux0 = aux_state;
    err = launch_kalman(a, gp->dtype, reinterpret_cast<cudaStream_t>(stream));
  } else {
    err = launch_decode(a, gp->dtype, reinterpret_cast<cudaStream_t>(stream));
  }
  return err == cudaSuccess ? DR_OK : DR_ERR_CUDA;
}

size_t dr_chunk_bwd_workspace_bytes(int variant, int dtype, int B, int T, int H, int dk, int dv,
                                    int chunk) {
  if (B < 1 || T < 1 || H < 1 || !chunk_bwd_supported(variant, dtype, dk, dv, chunk)) return 0;
  return chunk_bwd_workspace_bytes(variant, B, T, H);
}

int dr_chunk_bwd(const void* q, const void* k, const void* v, const float* log_alpha,
                 const dr_params* gp, int variant, float eps, const float* init_state,
                 const void* d_out, const float* d_final_state, const dr_grads* g, int B, int T,
                 int H, int dk_, int dv_, int chunk, dr_stream_t stream) {
  if (!gp || !g || !q || !k || !v || !log_alpha || !d_out || !g->dq || !g->dk || !g->dv ||
      !g->d_log_alpha)
    return DR_ERR_NULL;
  const bool kalman = variant == DR_KDN || variant == DR_IKDN;   // gains from a variance
  if (kalman ? (!g->d_omega || !g->d_r) : !g->d_eta) return DR_ERR_NULL;
  if (gp->dtype != DR_FP32 && gp->dtype != DR_BF16) return DR_ERR_DTYPE;
  if (B < 1 || T < 1 || H < 1 || !dim_ok(dk_) || !dim_ok(dv_)) return DR_ERR_SHAPE;
  if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128) return DR_ERR_SHAPE;
  if ((long long)B * T * H * (dk_ > dv_ ? dk_ : dv_) >= (1LL << 40)) return DR_ERR_SHAPE;
  if (!(eps >= 0.f)) return DR_ERR_ARG;
  int st = check_gates(gp, variant);
  if (st != DR_OK) return st;
  if (!chunk_bwd_supported(variant, gp->dtype, dk_, dv_, chunk)) return DR_ERR_UNSUPPORTED;
  if ((variant == DR_PGDN || variant == DR_PKDA) && (!g->d_alphaP || !g->d_betaP || !g->d_mu))
    return DR_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(log_alpha) ||
      !aligned16(d_out) || !aligned16(d_final_state) || !aligned16(g->dq) || !aligned16(g->dk) ||
      !aligned16(g->dv) || !aligned16(init_state) || !aligned16(g->d_init_state))
    return DR_ERR_ALIGN;
  if (variant == DR_KDN && !aligned16(gp->omega)) return DR_ERR_ALIGN;   // 16-byte copies
  const size_t need = chunk_bwd_workspace_bytes(variant, B, T, H);
  if (!gp->workspace || gp->workspace_bytes < need) return DR_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(gp->workspace) & 255u) return DR_ERR_ALIGN;
  FwdArgs a = make_args(q, k, v, log_alpha, gp, variant, eps, B, T, H, dk_, dv_, chunk);
  a.S0 = init_state;
  a.aux0 = gp->aux_init;
  cudaError_t err = launch_chunk_bwd(a, d_out, d_final_state, *g, gp->workspace,
                                     reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? DR_OK : DR_ERR_CUDA;
}

int dr_set_chain_fault_for_testing(long long withhold_flag, unsigned long long wait_ns) {
  if (withhold_flag < -1 || wait_ns == 0) return DR_ERR_ARG;
  if (cudaMemcpyToSymbol(g_chain_withhold, &withhold_flag, sizeof(withhold_flag)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_chain_wait_ns, &wait_ns, sizeof(wait_ns)) != cudaSuccess)
    return DR_ERR_CUDA;
  return DR_OK;
}

int dr_get_device_status(dr_stream_t stream) {
  int h = 0;
  const int zero = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyFromSymbolAsync(&h, g_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return DR_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return DR_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DR_ERR_CUDA;
  return h;
}

}  // extern "C"
