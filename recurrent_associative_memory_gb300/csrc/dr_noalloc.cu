// dr_noalloc.cu — dr_chunk_fwd_noalloc: the two-phase tensor-core forward with
// its per-chunk records kept in scratch that the library carries itself, for
// callers that cannot hand over device memory of their own.
//
// The scratch is one file-scope device array, created when the CUDA module is
// loaded on a device and held until the process exits.  Host code cannot pass
// the array's name to a kernel (on the host that name is only a stand-in for
// the device symbol), so the device address is looked up with
// cudaGetSymbolAddress, with that device current, and cached per device
// together with the context it was looked up in: a new context on the device
// (after cudaDeviceReset, say) reloads the module, and the address is looked up
// again there.
#include <cuda.h>

#include <mutex>

#include "dr_common.cuh"

namespace dr {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[DR_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
CUcontext g_scratch_ctx[kMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

// The current context (driver entry point cuCtxGetCurrent, via the runtime), or
// nullptr if it cannot be had.
CUcontext current_context() {
  using GetCtx = CUresult (*)(CUcontext*);
  static GetCtx fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<GetCtx>(nullptr);
    return reinterpret_cast<GetCtx>(p);
  }();
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of the scratch array on the current device (looked up on the
// first call per device and context), or nullptr if the lookup failed.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  const CUcontext ctx = current_context();   // null before the runtime's first call
  if (!g_scratch_addr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = current_context();
  }
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace dr

extern "C" int dr_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                    const float* log_alpha, const dr_params* gp, int variant,
                                    float eps, const float* init_state, void* out,
                                    float* final_state, int B, int T, int H, int dk, int dv,
                                    int chunk, dr_stream_t stream) {
  // the same argument checks as dr_chunk_fwd, in the same order, before the
  // workspace size is asked for, so one bad call gets one answer from both
  if (!gp || !q || !k || !v || !log_alpha || !out) return DR_ERR_NULL;
  if (gp->dtype != DR_FP32 && gp->dtype != DR_BF16) return DR_ERR_DTYPE;
  if (B < 1 || T < 1 || H < 1) return DR_ERR_SHAPE;
  const size_t need = dr_chunk_fwd_workspace_bytes(variant, gp->dtype, B, T, H, dk, dv, chunk);
  if (need == 0) return DR_ERR_UNSUPPORTED;                 // not the two-phase path's shapes
  if (need > (size_t)DR_NOALLOC_SCRATCH_BYTES) return DR_ERR_WORKSPACE;
  void* scratch = dr::scratch_address();
  if (!scratch) return DR_ERR_CUDA;
  // Nothing in the scratch has to start at zero: the prep kernel writes every
  // record the carry kernel reads, earlier in the same stream.
  dr_params p = *gp;
  p.workspace = scratch;
  p.workspace_bytes = DR_NOALLOC_SCRATCH_BYTES;
  return dr_chunk_fwd(q, k, v, log_alpha, &p, variant, eps, init_state, out, final_state, B, T,
                      H, dk, dv, chunk, stream);
}
