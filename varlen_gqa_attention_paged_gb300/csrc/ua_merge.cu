// ua_merge.cu -- LSE merge of the split-KV partitions (the reduce kernel of the aiter
// PR #3962 "split-K long-context decode for shuffled fp8 SWA": per-partition max / sum /
// partial output in fp32 scratch, partitions whose sum is 0 skipped, rows that saw no
// key written as 0).
//
// One warp per output row (query token x head).  With m_z, l_z the base-2 running max
// and sum of partition z and acc_z its unnormalised output:
//   M = max_{z: l_z > 0} m_z,  L = sum_{z: l_z > 0} l_z 2^(m_z - M),
//   out = sum_{z: l_z > 0} acc_z 2^(m_z - M) / L   (0 when no partition has l_z > 0).
#include "ua_device.cuh"
#include "ua_internal.h"

#include "ua.h"

namespace ua {

template <int D>
__global__ void __launch_bounds__(256) ua_merge_kernel(const __grid_constant__ MergeParams p) {
  constexpr int kPer = D / 32;  // output elements per lane
  grid_dependency_wait();        // the partition kernel's scratch is complete
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  if (row >= p.rows) return;
  const int np = p.n_part;
  const float* m = p.ws_m + static_cast<size_t>(row) * np;
  const float* l = p.ws_l + static_cast<size_t>(row) * np;
  const float* a = p.ws_acc + static_cast<size_t>(row) * np * D + lane * kPer;

  // Partitions go 32 at a time, one per lane: max and sum loads are independent, the
  // row max and sum are warp reductions, and every partition's weight reaches the lanes
  // through a shuffle, so the partial-output loads of all partitions can be in flight
  // together.  Empty partitions (l = 0) get weight 0 and are selected away.
  float M = -INFINITY;
  for (int z0 = 0; z0 < np; z0 += 32) {
    const int z = z0 + lane;
    if (z < np && l[z] > 0.f) M = fmaxf(M, m[z]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float L = 0.f;
  if (M != -INFINITY) {
    for (int z0 = 0; z0 < np; z0 += 32) {
      const int z = z0 + lane;
      const float lz = z < np ? l[z] : 0.f;
      const float wz = lz > 0.f ? fast_exp2(m[z] - M) : 0.f;
      L += lz * wz;
      const int nz = min(32, np - z0);
#pragma unroll 8
      for (int k = 0; k < nz; ++k) {
        const float wt = __shfl_sync(0xffffffffu, wz, k);
        const float* az = a + static_cast<size_t>(z0 + k) * D;
#pragma unroll
        for (int e = 0; e < kPer; e += 2) {
          const float2 v = *reinterpret_cast<const float2*>(az + e);
          acc[e] += wt != 0.f ? v.x * wt : 0.f;
          acc[e + 1] += wt != 0.f ? v.y * wt : 0.f;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const size_t base = static_cast<size_t>(row) * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; e += 2) {
    const float x0 = acc[e] * inv, x1 = acc[e + 1] * inv;
    if (p.out_dtype == UA_DT_F32) {
      *reinterpret_cast<float2*>(static_cast<float*>(p.out) + base + e) = make_float2(x0, x1);
    } else {
      const uint32_t v = p.out_dtype == UA_DT_BF16 ? pack_bf16(x0, x1) : pack_f16(x0, x1);
      *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + base + e) = v;
    }
  }
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s) {
  if (p.rows <= 0) return cudaSuccess;
  const dim3 grid((p.rows + 7) / 8);
  switch (p.head_dim) {
    case 64: return launch_pdl(ua_merge_kernel<64>, grid, dim3(256), 0, s, 1, p);
    case 128: return launch_pdl(ua_merge_kernel<128>, grid, dim3(256), 0, s, 1, p);
    case 256: return launch_pdl(ua_merge_kernel<256>, grid, dim3(256), 0, s, 1, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ua
