// ua_prefill_d256.cu -- instantiations of the tensor-memory prefill kernel for head_dim 256.
#include "ua_prefill_wide.cuh"

namespace ua {

cudaError_t launch_prefill_d256(const PrefillParams& pp, dim3 grid, int kv, bool feat, int nq,
                                cudaStream_t s) {
  if (nq != 1) return cudaErrorInvalidValue;
  return launch_prefill_wide_dispatch<256>(pp, grid, kv, feat, s);
}

}  // namespace ua
