// ua_prefill_d64.cu -- instantiations of the tensor-memory prefill kernel for head_dim 64.
#include "ua_prefill_tm.cuh"

namespace ua {

cudaError_t launch_prefill_d64(const PrefillParams& pp, dim3 grid, int kv, bool feat, int nq,
                               cudaStream_t s) {
  return launch_prefill_tm_dispatch<64>(pp, grid, kv, feat, nq, s);
}

}  // namespace ua
