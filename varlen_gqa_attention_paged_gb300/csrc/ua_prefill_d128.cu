// ua_prefill_d128.cu -- instantiations of the tensor-memory prefill kernel for head_dim 128.
#include "ua_prefill_tm.cuh"

namespace ua {

cudaError_t launch_prefill_d128(const PrefillParams& pp, dim3 grid, int kv, bool feat, int nq,
                               cudaStream_t s) {
  return launch_prefill_tm_dispatch<128>(pp, grid, kv, feat, nq, s);
}

}  // namespace ua
