// ua_tile_d64.cu -- instantiations of the attention tile kernel for head_dim 64.
#include "ua_tile.cuh"

namespace ua {

cudaError_t launch_tile_d64(const TileParams& tp, dim3 grid, int wm, int kv, bool feat, bool tma,
                             int cluster_y, int cluster_z, cudaStream_t s) {
  return launch_tile_dispatch<64>(tp, grid, wm, kv, feat, tma, cluster_y, cluster_z, s);
}

}  // namespace ua
