// ua_tile_d64.cu -- instantiations of the attention tile kernel for head_dim 64.
#include "ua_tile.cuh"

namespace ua {

cudaError_t launch_tile_d64(const AttnParams& p, dim3 grid, int wm, int kv, bool feat,
                             cudaStream_t s) {
  return launch_tile_dispatch<64>(p, grid, wm, kv, feat, s);
}

}  // namespace ua
