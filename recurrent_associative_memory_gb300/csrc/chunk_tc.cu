// chunk_tc.cu — tensor-core (tcgen05 / TMEM / TMA) chunkwise forward.
#include "dr_common.cuh"

namespace dr {

bool chunk_tc_supported(int variant, int dtype, int dk, int dv, int chunk) {
  (void)variant; (void)dtype; (void)dk; (void)dv; (void)chunk;
  return false;
}

cudaError_t launch_chunk_tc(const FwdArgs& a, cudaStream_t st) {
  (void)a; (void)st;
  return cudaErrorNotSupported;
}

}  // namespace dr
