// ua_prefill_d256.cu -- instantiations of the tensor-memory prefill kernel for head_dim 256.
#include "ua_prefill.cuh"

namespace ua {

cudaError_t launch_prefill_d256(const PrefillParams& pp, dim3 grid, int kv, bool feat, int nq,
                                cudaStream_t s) {
  return launch_prefill_dispatch<256>(pp, grid, kv, feat, nq, s);
}

}  // namespace ua
