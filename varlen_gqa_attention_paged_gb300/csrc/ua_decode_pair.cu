// ua_decode_pair.cu -- instantiations of the key-major decode tile kernel with two kv-heads
// per CTA (fp8 caches, head_dim 64 and 128, at most 4 rows per kv-head).
#include "ua_decode.cuh"

namespace ua {

cudaError_t launch_decode_pair_d64(const TileParams& tp, dim3 grid, bool feat, int cluster_y,
                                   int cluster_z, cudaStream_t s) {
  return launch_decode_pair<64>(tp, grid, feat, cluster_y, cluster_z, s);
}

cudaError_t launch_decode_pair_d128(const TileParams& tp, dim3 grid, bool feat, int cluster_y,
                                    int cluster_z, cudaStream_t s) {
  return launch_decode_pair<128>(tp, grid, feat, cluster_y, cluster_z, s);
}

int decode_cluster_capacity_pair(int head_dim, int cluster_y, int cluster_z) {
  return head_dim == 64 ? decode_cluster_capacity_t<64, KV_E4M3, 4, 2>(cluster_y, cluster_z)
                        : decode_cluster_capacity_t<128, KV_E4M3, 4, 2>(cluster_y, cluster_z);
}

int decode_pair_ctas_per_sm(int head_dim) {
  return head_dim == 64 ? DecCfg<64, KV_E4M3, 4, 2>::kMinBlocks
                        : DecCfg<128, KV_E4M3, 4, 2>::kMinBlocks;
}

}  // namespace ua
