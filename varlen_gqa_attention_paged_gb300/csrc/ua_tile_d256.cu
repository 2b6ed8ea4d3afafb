// ua_tile_d256.cu -- instantiations of the attention tile kernel for head_dim 256.
#include "ua_tile.cuh"

namespace ua {

cudaError_t launch_tile_d256(const TileParams& tp, dim3 grid, int wm, int kv, bool feat, bool tma,
                             int cluster_y, int cluster_z, cudaStream_t s) {
  return launch_tile_dispatch<256>(tp, grid, wm, kv, feat, tma, cluster_y, cluster_z, s);
}

}  // namespace ua
