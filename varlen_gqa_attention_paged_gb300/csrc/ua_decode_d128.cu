// ua_decode_d128.cu -- instantiations of the key-major decode tile kernel for head_dim 128.
#include <array>
#include <map>
#include <mutex>

#include "ua_decode.cuh"

namespace ua {

cudaError_t launch_decode_d128(const TileParams& tp, dim3 grid, int kv, bool feat, int cluster_y,
                              int cluster_z, cudaStream_t s) {
  return launch_decode_dispatch<128>(tp, grid, kv, feat, cluster_y, cluster_z, s);
}

int decode_ctas_per_sm(int head_dim, int kv) {
  return head_dim == 64 ? decode_ctas_per_sm_d<64>(kv) : decode_ctas_per_sm_d<128>(kv);
}

int decode_cluster_capacity(int head_dim, int kv, int cluster_y, int cluster_z) {
  static std::mutex mu;
  static std::map<std::array<int, 5>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  const std::array<int, 5> key = {dev, head_dim, kv == KV_E4M3 ? 1 : 0, cluster_y, cluster_z};
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const int n = head_dim == 64 ? decode_cluster_capacity_d<64>(kv, cluster_y, cluster_z)
                               : decode_cluster_capacity_d<128>(kv, cluster_y, cluster_z);
  cache.emplace(key, n);
  return n;
}

}  // namespace ua
