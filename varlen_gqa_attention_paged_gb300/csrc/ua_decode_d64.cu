// ua_decode_d64.cu -- instantiations of the key-major decode tile kernel for head_dim 64.
#include "ua_decode.cuh"

namespace ua {

cudaError_t launch_decode_d64(const TileParams& tp, dim3 grid, int kv, bool feat, int cluster_y,
                              int cluster_z, cudaStream_t s) {
  return launch_decode_dispatch<64>(tp, grid, kv, feat, cluster_y, cluster_z, s);
}

}  // namespace ua
