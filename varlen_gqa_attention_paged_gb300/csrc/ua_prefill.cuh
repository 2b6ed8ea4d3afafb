// ua_prefill.cuh -- helpers shared by the tensor-memory prefill kernels of libua.so
// (ua_prefill_tm.cuh for head_dim <= 128, ua_prefill_wide.cuh for head_dim 256).
#pragma once

#include <cuda.h>

#include "ua_device.cuh"
#include "ua_internal.h"

namespace ua {

__device__ __forceinline__ void tma_load_3d_pf(void* dst, const CUtensorMap* map, int x, int y,
                                               int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// Bounded wait that also gives up at once when another warp of the CTA already did.
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        unsigned int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, DEV_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

// pf_wait for a whole warp: every lane waits, and the result is the same in every lane
// (a lane that gave up makes the warp give up), so the warp stays converged.
__device__ __forceinline__ bool pf_wait_warp(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, unsigned int* status) {
  return __all_sync(0xffffffffu, pf_wait(bar, parity, abort_flag, status));
}

// Sequence owning token-block slot x: the last b with floor(cu[b] / TQ) + b <= x.
__device__ __forceinline__ int pf_find_seq(const int32_t* __restrict__ cu, int num_seqs, int x,
                                           int tq) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) / tq + mid <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

}  // namespace ua
