// ua_tile_d256.cu -- instantiations of the attention tile kernel for head_dim 256.
#include "ua_tile.cuh"

namespace ua {

cudaError_t launch_tile_d256(const AttnParams& p, dim3 grid, int wm, int kv, bool feat,
                             cudaStream_t s) {
  return launch_tile_dispatch<256>(p, grid, wm, kv, feat, s);
}

}  // namespace ua
