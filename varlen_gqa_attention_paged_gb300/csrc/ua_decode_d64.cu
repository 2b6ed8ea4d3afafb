// ua_decode_d64.cu -- instantiations of the key-major decode tile kernel for head_dim 64
// (four consumer warps).
#include "ua_decode.cuh"

namespace ua {

cudaError_t launch_decode_w4_d64(const TileParams& tp, dim3 grid, int kv, bool feat,
                                 int cluster_y, int cluster_z, cudaStream_t s) {
  return launch_decode_width<64, 4>(tp, grid, kv, feat, cluster_y, cluster_z, s);
}

}  // namespace ua
