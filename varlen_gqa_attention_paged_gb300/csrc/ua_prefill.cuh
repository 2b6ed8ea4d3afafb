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

// Sequence owning token-block slot x and its sizes, found by each warp on its own: lane i
// reads cu_seqlens_q[i], cu_seqlens_q[i + 1] and seq_lens_k[i] (32 sequences a round, the
// loads independent and coalesced), the owner is the last b with
// floor(cu[b] / tb) + b <= x (a ballot; the left side grows strictly with b), and its
// sizes reach every lane by shuffles.  One round of loads instead of the binary search's
// chain of dependent ones.
struct PfSeq {
  int b, q0, q_len, kv_len;
};
__device__ __forceinline__ PfSeq pf_seq_of_slot(const int32_t* __restrict__ cu,
                                                const int32_t* __restrict__ kvl, int num_seqs,
                                                int x, int tb) {
  const int lane = threadIdx.x & 31;
  PfSeq r{0, 0, 0, 0};
  for (int base = 0; base < num_seqs; base += 32) {
    const int i = base + lane;
    const bool in = i < num_seqs;
    const int c0 = in ? __ldg(cu + i) : 0;
    const int c1 = in ? __ldg(cu + i + 1) : 0;
    const int kv = in ? __ldg(kvl + i) : 0;
    const unsigned m = __ballot_sync(0xffffffffu, in && c0 / tb + i <= x);
    if (m != 0u) {
      const int src = 31 - __clz(m);
      r.b = base + src;
      r.q0 = __shfl_sync(0xffffffffu, c0, src);
      r.q_len = __shfl_sync(0xffffffffu, c1, src) - r.q0;
      r.kv_len = __shfl_sync(0xffffffffu, kv, src);
    }
    if (m != 0xffffffffu) break;  // the owner lies in this round
  }
  return r;
}

}  // namespace ua
