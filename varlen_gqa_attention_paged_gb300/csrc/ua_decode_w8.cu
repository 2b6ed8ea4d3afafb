// ua_decode_w8.cu -- instantiations of the key-major decode tile kernel with eight consumer
// warps and 128-key stages (head_dim 64 and 128), for grids of at most one CTA per SM.
#include "ua_decode.cuh"

namespace ua {

cudaError_t launch_decode_w8_d64(const TileParams& tp, dim3 grid, int kv, bool feat,
                                 int cluster_y, int cluster_z, cudaStream_t s) {
  return launch_decode_width<64, 8>(tp, grid, kv, feat, cluster_y, cluster_z, s);
}

cudaError_t launch_decode_w8_d128(const TileParams& tp, dim3 grid, int kv, bool feat,
                                  int cluster_y, int cluster_z, cudaStream_t s) {
  return launch_decode_width<128, 8>(tp, grid, kv, feat, cluster_y, cluster_z, s);
}

int decode_cluster_capacity_w8(int head_dim, int kv, int cluster_y, int cluster_z) {
  return head_dim == 64 ? decode_cluster_capacity_d<64, 8>(kv, cluster_y, cluster_z)
                        : decode_cluster_capacity_d<128, 8>(kv, cluster_y, cluster_z);
}

}  // namespace ua
