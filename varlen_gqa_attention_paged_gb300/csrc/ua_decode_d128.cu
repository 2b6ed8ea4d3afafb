// ua_decode_d128.cu -- instantiations of the key-major decode tile kernel for head_dim 128
// (four consumer warps), and the decode tile's resource queries.
#include <array>
#include <map>
#include <mutex>

#include "ua_decode.cuh"

namespace ua {

cudaError_t launch_decode_w4_d128(const TileParams& tp, dim3 grid, int kv, bool feat,
                                  int cluster_y, int cluster_z, cudaStream_t s) {
  return launch_decode_width<128, 4>(tp, grid, kv, feat, cluster_y, cluster_z, s);
}

int decode_ctas_per_sm(int head_dim, int kv) {
  return head_dim == 64 ? decode_ctas_per_sm_d<64>(kv) : decode_ctas_per_sm_d<128>(kv);
}

int decode_cluster_capacity(int head_dim, int kv, bool wide, bool pair, int cluster_y,
                            int cluster_z) {
  static std::mutex mu;
  static std::map<std::array<int, 6>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  const std::array<int, 6> key = {dev, head_dim, kv == KV_E4M3 ? 1 : 0,
                                  pair ? 2 : wide ? 1 : 0, cluster_y, cluster_z};
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n;
  if (pair) n = decode_cluster_capacity_pair(head_dim, cluster_y, cluster_z);
  else if (wide) n = decode_cluster_capacity_w8(head_dim, kv, cluster_y, cluster_z);
  else n = head_dim == 64 ? decode_cluster_capacity_d<64, 4>(kv, cluster_y, cluster_z)
                          : decode_cluster_capacity_d<128, 4>(kv, cluster_y, cluster_z);
  cache.emplace(key, n);
  return n;
}

}  // namespace ua
