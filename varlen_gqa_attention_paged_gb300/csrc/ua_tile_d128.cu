// ua_tile_d128.cu -- instantiations of the attention tile kernel for head_dim 128.
#include "ua_tile.cuh"

namespace ua {

cudaError_t launch_tile_d128(const TileParams& tp, dim3 grid, int wm, int kv, bool feat, bool tma,
                             int cluster_y, int cluster_z, cudaStream_t s) {
  return launch_tile_dispatch<128>(tp, grid, wm, kv, feat, tma, cluster_y, cluster_z, s);
}

int tile_ctas_per_sm(int head_dim, int kv, int wm) {
  if (head_dim == 64) return tile_ctas_per_sm_d<64>(kv, wm);
  if (head_dim == 256) return tile_ctas_per_sm_d<256>(kv, wm);
  return tile_ctas_per_sm_d<128>(kv, wm);
}

}  // namespace ua
