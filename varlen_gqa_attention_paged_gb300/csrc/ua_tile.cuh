// ua_tile.cuh -- the attention tile kernel of libua.so (included by ua_tile_d*.cu).
//
// One CTA owns (q-block, kv-head g, key partition z).  A q-block is BM consecutive
// rows of the packed (query token x head-in-group) row space of one sequence, so
// every GQA head that reads kv-head g shares one pass over the keys (vllm-rdna PR
// #34 "FA-RDNA2 D=128 prefill", "Change" 1: several heads of a group in one tile).
// The CTA walks the keys [ks, ke) of its partition; with one partition it writes the
// normalised output (the "2D" path), with several it writes fp32 max / sum /
// unnormalised output for the merge kernel (the split-KV path of the aiter PR #3962).
//
// Warp roles (160 threads):
//   warp 4      producer: gathers each tile of T keys through the block table into a
//               STAGES-deep shared-memory ring.  With block_size % 16 == 0 every
//               16-key page slice is one TMA tensor box per column block (completion
//               counted in bytes on an mbarrier); otherwise 16-byte cp.async copies.
//               Rows of 128 bytes or more land in the 128-byte swizzled layout (16-byte
//               chunk c of row r stored at chunk c ^ (r & 7)), which keeps the ldmatrix
//               reads below free of bank conflicts.
//   warps 0..3  consumers: QK^T and P.V on tensor cores (mma.sync m16n8k16, fp32
//               accumulate), score transform, online softmax in base 2 with quad
//               shuffles.  fp8 e4m3 codes are turned into f16 MMA operands in
//               registers: the head dimension is permuted so that every lane's operand
//               bytes are contiguous in shared memory (see kPermD).
//   WM = 1 (decode-shaped q-blocks, BM = 16): the four consumer warps share the 16
//          rows and each takes 16 keys of every tile; their states merge at the end.
//   WM = 4 (BM = 64): each consumer warp owns 16 rows and walks every key.
#pragma once

#include <atomic>
#include <climits>

#include <cuda.h>

#include "ua_device.cuh"
#include "ua_internal.h"

#include "ua.h"

namespace ua {

template <int KV>
struct KvTraits;
template <>
struct KvTraits<KV_F16> {
  static constexpr int kEsz = 2;
  static constexpr bool kF16Mma = true;
};
template <>
struct KvTraits<KV_BF16> {
  static constexpr int kEsz = 2;
  static constexpr bool kF16Mma = false;
};
template <>
struct KvTraits<KV_E4M3> {
  static constexpr int kEsz = 1;
  static constexpr bool kF16Mma = true;
};

// Byte offset of 16-byte chunk `c` of row `r` inside a 128-byte-swizzled column block.
__host__ __device__ constexpr uint32_t sw128(uint32_t r, uint32_t c) {
  return r * 128u + ((c ^ (r & 7u)) << 4);
}

template <int D, int KV, int WM>
struct TileCfg {
  static constexpr int kConsumerWarps = 4;
  static constexpr int kThreads = 32 * (kConsumerWarps + 1);
  static constexpr int kWN = kConsumerWarps / WM;  // warps sharing one 16-row m-tile
  static constexpr int kT = 64;                    // keys per pipeline stage (4 pages of 16)
  static constexpr int kEsz = KvTraits<KV>::kEsz;
  static constexpr int kRowBytes = D * kEsz;       // one K or V row in the cache
  // Rows of 128 bytes or more are stored as 128-byte swizzled column blocks; 64-byte
  // rows (fp8 with head_dim 64) are stored plainly (only the dequant pass reads them).
  static constexpr bool kSwz = kRowBytes >= 128;
  static constexpr int kCBW = kSwz ? 128 : kRowBytes;  // bytes of a row in one column block
  static constexpr int kCB = kRowBytes / kCBW;         // column blocks per row
  static constexpr int kCBBytes = kT * kCBW;           // one column block of a tile
  static constexpr int kStageBytes = 2 * kCB * kCBBytes;  // K then V
  // fp8 operands are dequantised in registers, with the head dimension permuted: the
  // QK^T sum runs over d in any order (Q and K permuted alike), and the P.V output
  // columns are put back in order when written.
  static constexpr bool kPermD = KV == KV_E4M3;
  static constexpr int kMergeBytes = (kWN > 1) ? kConsumerWarps * (2 * 16 + (D / 8) * 32 * 4) * 4 : 0;
  // decode-shaped CTAs of one cluster exchange their partitions' rows (max, sum, D
  // unnormalised outputs of 16 rows) through distributed shared memory
  static constexpr int kPartBytes = (WM == 1) ? 16 * (D + 2) * 4 : 0;
  // decode-shaped CTAs aim at two per SM (about 110 KB each); the 64-row variant at one
  static constexpr int kBudget = (WM == 1 ? 110 : 200) * 1024;
  static constexpr int kStagesFit = kBudget / kStageBytes;
  static constexpr int kStages = kStagesFit < 2 ? 2 : (kStagesFit > 4 ? 4 : kStagesFit);
  static constexpr int kPipeRaw = (kStages * kStageBytes > kMergeBytes + kPartBytes)
                                      ? kStages * kStageBytes
                                      : kMergeBytes + kPartBytes;
  static constexpr int kPipeBytes = (kPipeRaw + 1023) & ~1023;
  static constexpr int kSmemBytes = 1024 + kPipeBytes + 2 * kStages * 8;
  // two CTAs per SM when they fit, but not at d256, whose 16 x 256 fp32 accumulators alone
  // take 128 registers a thread
  static constexpr int kMinBlocks = (D <= 128 && 2 * kSmemBytes <= 227 * 1024) ? 2 : 1;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kRowBytes % kCBW == 0 && kCBW % 16 == 0, "rows are whole column blocks");
  static_assert(kSwz || KV == KV_E4M3, "16-bit rows are at least 128 bytes");

  // Byte offset of 16-byte chunk c of tile row r in a K or V stage.
  static __device__ __forceinline__ uint32_t raw_off(uint32_t r, uint32_t c) {
    if constexpr (kSwz) return (c / 8) * kCBBytes + sw128(r, c % 8);
    else return r * kCBW + c * 16;
  }
  // Byte offset of byte `x` of tile row r (x % 16 + the 16-byte chunk's offset).
  static __device__ __forceinline__ uint32_t raw_byte(uint32_t r, uint32_t x) {
    return raw_off(r, x / 16) + (x & 15u);
  }
};

// Writes row rr (0: fragment row gq, 1: gq + 8) of a warp's P.V accumulators times `mul`
// to `dst` (D values of type `dtype`).  Fragment column 2cq + e of n-tile nd is output
// column 8 nd + 2cq + e, or (2cq + e) D/8 + nd when the head dimension is permuted.
template <int D, bool PERM>
__device__ __forceinline__ void store_o_row(const float (&o)[D / 8][4], int rr, int cq, float mul,
                                            void* dst, int dtype) {
  if constexpr (!PERM) {
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      const int col = nd * 8 + 2 * cq;
      const float x0 = o[nd][2 * rr] * mul, x1 = o[nd][2 * rr + 1] * mul;
      if (dtype == UA_DT_F32) {
        *reinterpret_cast<float2*>(static_cast<float*>(dst) + col) = make_float2(x0, x1);
      } else {
        const uint32_t v = dtype == UA_DT_BF16 ? pack_bf16(x0, x1) : pack_f16(x0, x1);
        *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(dst) + col) = v;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int base = (2 * cq + e) * (D / 8);
#pragma unroll
      for (int nd = 0; nd < D / 8; nd += 4) {
        const float x0 = o[nd][2 * rr + e] * mul, x1 = o[nd + 1][2 * rr + e] * mul;
        const float x2 = o[nd + 2][2 * rr + e] * mul, x3 = o[nd + 3][2 * rr + e] * mul;
        if (dtype == UA_DT_F32) {
          *reinterpret_cast<float4*>(static_cast<float*>(dst) + base + nd) =
              make_float4(x0, x1, x2, x3);
        } else {
          const bool bf = dtype == UA_DT_BF16;
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(dst) + base + nd) =
              make_uint2(bf ? pack_bf16(x0, x1) : pack_f16(x0, x1),
                         bf ? pack_bf16(x2, x3) : pack_f16(x2, x3));
        }
      }
    }
  }
}

// Sequence owning q-block slot x: the last b with floor(cu[b] * G / BM) + b <= x
// (a monotone slot layout that leaves at most one idle slot per sequence).
__device__ __forceinline__ int find_seq(const int32_t* __restrict__ cu, int num_seqs, int x,
                                        int group, int bm) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int start =
        static_cast<int>((static_cast<long long>(__ldg(cu + mid)) * group) / bm) + mid;
    if (start <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}

__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}

// The mbarrier's pending count rises by one now and falls once this thread's earlier
// cp.async copies land (no net arrival).

__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// LSE merge of one output row over the np (1 <= np <= 16) split partitions of a
// thread-block cluster, by one warp (the merge of the split path):
//   M = max_{l_z > 0} m_z,  L = sum l_z 2^(m_z - M),  out = sum acc_z 2^(m_z - M) / L.
// Partition zz is the cluster's CTA rank0 + rank_step * zz; in its shared memory the row's
// max and sum sit at byte offsets m_off and l_off and its partial row (D floats) at
// row_off.  Every partition's max, sum and slice of the row are loaded before any is used
// (warp-uniform branches, no selects on loaded values), so the round trips through
// distributed shared memory overlap.  An empty partition weighs 0 (its partial row is 0).
// Writes the normalised row to dst in out_dtype.
template <int D>
__device__ __forceinline__ void cluster_merge_row(uint32_t m_off, uint32_t l_off,
                                                  uint32_t row_off, int np, uint32_t rank0,
                                                  uint32_t rank_step, int lane, uint8_t* dst,
                                                  int out_dtype) {
  constexpr int kPer = D / 32;                       // columns a lane merges
  constexpr int kBatch = kPer > 4 ? 64 / kPer : 16;  // partitions loaded at once
  float mz = -INFINITY, lz = 0.f;
  if (lane < np) {
    const uint32_t rank = rank0 + rank_step * lane;
    mz = ld_cluster_f32(cluster_map(m_off, rank));
    lz = ld_cluster_f32(cluster_map(l_off, rank));
  }
  float v[kBatch][kPer];
  auto load = [&](int z0) {
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (z0 + i < np) {  // uniform
        const uint32_t a =
            cluster_map(row_off + lane * kPer * 4, rank0 + rank_step * (z0 + i));
        if constexpr (kPer >= 4) {
#pragma unroll
          for (int e = 0; e < kPer; e += 4) {
            const float4 x = ld_cluster_f32x4(a + e * 4);
            v[i][e] = x.x;
            v[i][e + 1] = x.y;
            v[i][e + 2] = x.z;
            v[i][e + 3] = x.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < kPer; ++e) v[i][e] = ld_cluster_f32(a + e * 4);
        }
      }
    }
  };
  load(0);
  float M = lz > 0.f ? mz : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float wz = (lz > 0.f && M != -INFINITY) ? fast_exp2(mz - M) : 0.f;
  float L = lz * wz;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  for (int z0 = 0; z0 < np; z0 += kBatch) {
    if (z0 > 0) load(z0);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (z0 + i < np) {  // uniform
        const float wt = __shfl_sync(0xffffffffu, wz, z0 + i);
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[e] = fmaf(v[i][e], wt, acc[e]);
      }
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < kPer; e += 2) {
    const int col = lane * kPer + e;
    const float x0 = acc[e] * inv, x1 = acc[e + 1] * inv;
    if (out_dtype == UA_DT_F32) {
      *reinterpret_cast<float2*>(reinterpret_cast<float*>(dst) + col) = make_float2(x0, x1);
    } else {
      const uint32_t w = out_dtype == UA_DT_BF16 ? pack_bf16(x0, x1) : pack_f16(x0, x1);
      *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(dst) + col) = w;
    }
  }
}

template <int D, int KV, int WM, bool FEAT, bool TMA>
__global__ void __launch_bounds__(160, (TileCfg<D, KV, WM>::kMinBlocks))
    ua_attn_tile_kernel(const __grid_constant__ TileParams tp) {
  using C = TileCfg<D, KV, WM>;
  constexpr int T = C::kT;
  constexpr int S = C::kStages;
  constexpr bool kF16Mma = KvTraits<KV>::kF16Mma;
  constexpr int BM = 16 * WM;
  const AttnParams& p = tp.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* const smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* const pipe = smem;
  uint64_t* const full = reinterpret_cast<uint64_t*>(smem + C::kPipeBytes);
  uint64_t* const empty = full + S;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int z = blockIdx.z;
  const int G = p.group;

  // Programmatic dependent launch: this grid may be scheduled while the previous kernel
  // on the stream finishes.  Set-up that reads no input (the barriers, the tensor maps
  // fetched into the descriptor cache) runs before the wait on that kernel; everything
  // else after it.  The next kernel (the merge) is let in early in turn.
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kConsumerWarps);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  if constexpr (TMA) {
    if (warp == C::kConsumerWarps && lane == 0) {
      tma_prefetch_desc(&tp.tmap_k);
      tma_prefetch_desc(&tp.tmap_v);
    }
  }
  __syncthreads();
  grid_dependency_wait();
  grid_launch_dependents();

  // ---- which rows and keys this CTA owns.  Slot x is sequence x when every sequence
  // fits one q-block (decode batches: no search); otherwise a binary search over
  // cu_seqlens_q finds the sequence.
  const int b = p.slot_per_seq ? static_cast<int>(blockIdx.x)
                               : find_seq(p.cu_seqlens_q, p.num_seqs, blockIdx.x, G, BM);
  const int q0 = __ldg(p.cu_seqlens_q + b);
  const int q_len = __ldg(p.cu_seqlens_q + b + 1) - q0;
  const int kv_len = __ldg(p.seq_lens_k + b);
  const int rows_b = q_len * G;
  const int slot0 =
      p.slot_per_seq ? b : static_cast<int>((static_cast<long long>(q0) * G) / BM) + b;
  const int r0 = (static_cast<int>(blockIdx.x) - slot0) * BM;
  if (p.slot_per_seq && rows_b > BM && threadIdx.x == 0 && z == 0 && g == 0)
    atomicOr(p.status, DEV_BAD_SHAPE);  // q_len above max_seqlen_q: rows past BM unwritten
  if (r0 < 0 || r0 >= rows_b) return;  // idle slot: uniform for the CTA
  const int r1 = min(r0 + BM, rows_b);
  const int ctx = kv_len - q_len;
  const int pos_first = ctx + r0 / G;
  const int pos_last = ctx + (r1 - 1) / G;
  const int hi = max(0, min(pos_last + 1, kv_len));
  // the walk starts on a 16-key page boundary; keys before a row's window are masked
  const int lo = min(hi, p.window_left >= 0 ? max(0, pos_first - p.window_left) : 0) & ~15;
  int part = (hi - lo + p.n_part - 1) / p.n_part;
  part = (part + 15) & ~15;
  const int ks = min(lo + z * part, hi);
  const int ke = min(ks + part, hi);
  const int ntiles = (ke - ks + T - 1) / T;

  if (warp == C::kConsumerWarps) {
    // ======================================================== producer warp
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    const uint64_t policy = l2_policy_evict_first();
    const int bs = p.block_size;
    int issued = 0;
    if constexpr (TMA) {
      // lane j < T/16 owns page slice j (keys key0 + 16j .. +15) of every tile
      const int oob = p.num_blocks * bs;  // first row coordinate past the cache: zero fill
      auto page_row = [&](int t) -> int {
        const int key = ks + t * T + 16 * lane;
        if (lane >= T / 16 || key >= ke) return oob;
        const int col = key / bs;
        const int blk = col < p.max_blocks_per_seq ? __ldg(bt + col) : -1;
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(p.num_blocks)) {
          atomicOr(p.status, DEV_BAD_BLOCK);
          return oob;
        }
        return blk * bs + key % bs;
      };
      int row_next = ntiles > 0 ? page_row(0) : oob;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % S;
        const int row = row_next;
        if (t + 1 < ntiles) row_next = page_row(t + 1);  // block-table lookups one tile ahead
        if (t >= S &&
            !mbar_wait_bounded(&empty[s], ((t / S) & 1) ^ 1, p.status, DEV_TIMEOUT))
          break;
        uint8_t* kdst = pipe + s * C::kStageBytes;
        uint8_t* vdst = kdst + C::kCB * C::kCBBytes;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        __syncwarp();
        if (lane < T / 16) {
#pragma unroll
          for (int cb = 0; cb < C::kCB; ++cb) {
            const int x = cb * (C::kCBW / C::kEsz);
            tma_load_3d(kdst + cb * C::kCBBytes + lane * 16 * C::kCBW, &tp.tmap_k, x, g, row,
                        &full[s], policy);
            tma_load_3d(vdst + cb * C::kCBBytes + lane * 16 * C::kCBW, &tp.tmap_v, x, g, row,
                        &full[s], policy);
          }
        }
        issued = t + 1;
      }
    } else {
      // any block size: 16-byte cp.async per chunk, rows with no key zero-filled
      const size_t slot_pitch = static_cast<size_t>(p.hkv) * C::kRowBytes;
      const uint8_t* kg = static_cast<const uint8_t*>(p.k) + static_cast<size_t>(g) * C::kRowBytes;
      const uint8_t* vg = static_cast<const uint8_t*>(p.v) + static_cast<size_t>(g) * C::kRowBytes;
      constexpr int kChunks = C::kRowBytes / 16;  // per row
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % S;
        if (t >= S &&
            !mbar_wait_bounded(&empty[s], ((t / S) & 1) ^ 1, p.status, DEV_TIMEOUT))
          break;
        const int key0 = ks + t * T;
        uint8_t* kdst = pipe + s * C::kStageBytes;
        uint8_t* vdst = kdst + C::kCB * C::kCBBytes;
#pragma unroll 1
        for (int rr = 0; rr < T / 32; ++rr) {
          const int row = lane + 32 * rr;
          const int key = key0 + row;
          long long off = -1;
          if (key < ke && key < kv_len) {
            const int col = key / bs;
            const int blk = col < p.max_blocks_per_seq ? __ldg(bt + col) : -1;
            if (static_cast<unsigned>(blk) < static_cast<unsigned>(p.num_blocks))
              off = static_cast<long long>((static_cast<size_t>(blk) * bs + key % bs) * slot_pitch);
            else
              atomicOr(p.status, DEV_BAD_BLOCK);
          }
#pragma unroll 4
          for (int c = 0; c < kChunks; ++c) {
            const uint32_t so = C::raw_off(row, c);
            if (off >= 0) {
              cp_async_16(kdst + so, kg + off + 16 * c);
              cp_async_16(vdst + so, vg + off + 16 * c);
            } else {
              *reinterpret_cast<uint4*>(kdst + so) = make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(vdst + so) = make_uint4(0, 0, 0, 0);
            }
          }
        }
        cp_async_arrive(&full[s]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
        issued = t + 1;
      }
    }
    // Never leave copies in flight into this CTA's shared memory.
    for (int t = max(0, issued - S); t < issued; ++t)
      mbar_wait_bounded(&full[t % S], (t / S) & 1, p.status, DEV_TIMEOUT);
    if (WM == 1 && p.cluster_merge) {  // the consumers' two cluster barriers
      cluster_sync();
      cluster_sync_relaxed();
    }
    return;
  }

  // ========================================================== consumer warps
  const int mt = warp / C::kWN;  // m-tile of this warp
  const int kgp = warp % C::kWN;  // key slice of this warp within a tile (WM = 1)
  const int gq = lane >> 2, cq = lane & 3;

  float k_scale = 1.f, v_scale = 1.f;
  if constexpr (KV == KV_E4M3) {
    k_scale = __ldg(p.kv_scale);
    v_scale = __ldg(p.kv_scale + 1);
  }
  const float scale = p.scale * k_scale;
  const float scale_log2 = scale * kLog2e;

  // Rows gq and gq + 8 of this warp's m-tile.
  bool rv[2];
  int rt[2], rh[2], ri[2], rpos[2], rlo[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int r = r0 + mt * 16 + gq + 8 * rr;
    rv[rr] = r < r1 && q0 + r / G < p.total_q;  // never index past the q / out tensors
    const int i = rv[rr] ? r / G : 0;
    ri[rr] = i;
    rt[rr] = q0 + i;
    rh[rr] = g * G + (rv[rr] ? r % G : 0);
    rpos[rr] = ctx + i;
    rlo[rr] = p.window_left >= 0 ? max(0, rpos[rr] - p.window_left) : 0;
  }
  // Bounds over the valid rows of the m-tile, to skip fully masked 16-key chunks and
  // to apply the mask only on boundary chunks.
  const bool tile_any = (r0 + mt * 16) < r1;
  int pmin = INT_MAX, pmax = INT_MIN, lomin = INT_MAX, lomax = INT_MIN;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    if (rv[rr]) {
      pmin = min(pmin, rpos[rr]);
      pmax = max(pmax, rpos[rr]);
      lomin = min(lomin, rlo[rr]);
      lomax = max(lomax, rlo[rr]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, o));
    pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
    lomin = min(lomin, __shfl_xor_sync(0xffffffffu, lomin, o));
    lomax = max(lomax, __shfl_xor_sync(0xffffffffu, lomax, o));
  }

  // Q fragments (A operand, row-major 16 x D), in the MMA input type.
  uint32_t qf[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int rr = j & 1;
      // fp8: k-slice kk of lane cq is d = cq D/4 + 4 kk + {0..3} (the K bytes it reads)
      const int col = C::kPermD ? cq * (D / 4) + 4 * kk + 2 * (j >> 1)
                                : kk * 16 + 2 * cq + 8 * (j >> 1);
      uint32_t v = 0;
      if (rv[rr]) {
        const uint16_t* qrow = static_cast<const uint16_t*>(p.q) +
                               (static_cast<size_t>(rt[rr]) * p.hq + rh[rr]) * D;
        v = __ldg(reinterpret_cast<const unsigned int*>(qrow + col));
        if constexpr (KV == KV_E4M3) {
          if (p.q_dtype == UA_DT_BF16) v = pack_f16(bf16_lo(v), bf16_hi(v));
        }
      }
      qf[kk][j] = v;
    }
  }

  float slope[2] = {0.f, 0.f};
  if constexpr (FEAT) {
    if (p.alibi != nullptr) {
      slope[0] = rv[0] ? __ldg(p.alibi + rh[0]) : 0.f;
      slope[1] = rv[1] ? __ldg(p.alibi + rh[1]) : 0.f;
    }
  }
  const float inv_softcap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;

  // Online-softmax state (base 2).  The sink is the initial running max of partition 0
  // and adds e^{sink - m} once to the row sum (counted by lane cq == 0 of the quad).
  float m_run[2], l_run[2];
  float o_acc[D / 8][4];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const bool sink = p.sinks != nullptr && z == 0 && kgp == 0 && rv[rr];
    m_run[rr] = sink ? __ldg(p.sinks + rh[rr]) * kLog2e : -INFINITY;
    l_run[rr] = (sink && cq == 0) ? 1.f : 0.f;
  }
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd)
#pragma unroll
    for (int e = 0; e < 4; ++e) o_acc[nd][e] = 0.f;

  // Cache slots at or past kv_len in the sequence's last page hold no key and may hold
  // anything (NaN included): their P is 0, and their V values are zeroed before P.V so
  // that 0 * NaN never enters the accumulator.
  bool aborted = false;

  for (int t = 0; t < ntiles; ++t) {
    const int s = t % S;
    if (!mbar_wait_bounded(&full[s], (t / S) & 1, p.status, DEV_TIMEOUT)) {
      aborted = true;
      break;
    }
    const uint8_t* kst = pipe + s * C::kStageBytes;
    const uint8_t* vst = kst + C::kCB * C::kCBBytes;
    const int key_tile = ks + t * T;

#pragma unroll 1
    for (int ch = (WM == 1 ? kgp : 0); ch < T / 16; ch += (WM == 1 ? 4 : 1)) {
      const int kc0 = key_tile + 16 * ch;
      if (!tile_any || kc0 >= ke || kc0 > pmax || kc0 + 16 <= lomin) continue;

      // ---- S = Q K^T for 16 keys (two n8 chunks)
      float sc[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[n][e] = 0.f;
      if constexpr (C::kPermD) {
        // Lane (gq, cq) reads bytes [cq D/4, (cq + 1) D/4) of K rows gq and gq + 8: word
        // q of its 16-byte chunk u holds d = cq D/4 + 4 kk + {0..3} of k-slice kk = 4u + q,
        // i.e. the B operand pairs (2cq, 2cq+1) and (2cq+8, 2cq+9) of that slice.
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          const uint32_t trow = 16 * ch + gq + 8 * n;
#pragma unroll
          for (int u = 0; u < D / 64; ++u) {
            const uint4 raw =
                *reinterpret_cast<const uint4*>(kst + C::raw_byte(trow, cq * (D / 4) + 16 * u));
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
              mma_16816<true>(sc[n], qf[4 * u + q], e4m3x2_to_f16x2(static_cast<uint16_t>(w[q])),
                              e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] >> 16)));
          }
        }
      } else {
        const uint32_t kbase = smem_addr(kst);
        const uint32_t kr = 16 * ch + (lane & 7) + ((lane >> 4) << 3);
        const uint32_t half = (lane >> 3) & 1;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t c = (kk & 3) * 2 + half;  // 16-byte chunk within the column block
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + (kk >> 2) * C::kCBBytes + sw128(kr, c), b0, b1, b2, b3);
          mma_16816<kF16Mma>(sc[0], qf[kk], b0, b1);
          mma_16816<kF16Mma>(sc[1], qf[kk], b2, b3);
        }
      }

      // ---- score transform and mask (log2 domain)
      const bool need_mask = kc0 < lomax || kc0 + 15 > pmin || kc0 + 16 > ke;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int rr = e >> 1;
          const int j = kc0 + n * 8 + 2 * cq + (e & 1);
          float x;
          if constexpr (FEAT) {
            x = sc[n][e] * scale;
            if (p.softcap > 0.f) x = p.softcap * fast_tanh(x * inv_softcap);
            x += slope[rr] * static_cast<float>(j - ctx);
            if (p.qq_bias != nullptr && rv[rr] && j >= ctx && j <= rpos[rr] &&
                ri[rr] < p.max_seqlen_q)
              x += __ldg(p.qq_bias + static_cast<size_t>(ri[rr]) * p.qq_stride + (j - ctx));
            x *= kLog2e;
          } else {
            x = sc[n][e] * scale_log2;
          }
          if (need_mask) {
            const bool ok = rv[rr] && j >= rlo[rr] && j <= rpos[rr] && j < ke;
            x = ok ? x : -INFINITY;
          }
          sc[n][e] = x;
        }
      }

      // ---- online softmax (rows gq, gq + 8; a row's 16 scores sit in one quad).  A row's
      // running max moves only when a score passes it by more than 8 (log2 units), so P
      // stays below 2^8 and the accumulators are rescaled only on those chunks.
      float alpha[2];
      bool grow_any = false;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        float mx = fmaxf(fmaxf(sc[0][2 * rr], sc[0][2 * rr + 1]),
                         fmaxf(sc[1][2 * rr], sc[1][2 * rr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const bool grow = mx > m_run[rr] + 8.f;  // from -inf: the first finite score
        alpha[rr] = grow ? fast_exp2(m_run[rr] - mx) : 1.f;
        if (grow) m_run[rr] = mx;
        grow_any |= grow;
        const float m_use = (m_run[rr] == -INFINITY) ? 0.f : m_run[rr];
        float rs = 0.f;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          sc[n][2 * rr] = fast_exp2(sc[n][2 * rr] - m_use);
          sc[n][2 * rr + 1] = fast_exp2(sc[n][2 * rr + 1] - m_use);
          rs += sc[n][2 * rr] + sc[n][2 * rr + 1];
        }
        l_run[rr] = l_run[rr] * alpha[rr] + rs;
      }
      if (__any_sync(0xffffffffu, grow_any)) {
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
          o_acc[nd][0] *= alpha[0];
          o_acc[nd][1] *= alpha[0];
          o_acc[nd][2] *= alpha[1];
          o_acc[nd][3] *= alpha[1];
        }
      }

      // ---- O += P V  (P as the A operand straight from the S accumulators)
      uint32_t pa[4], pl[4];
      if constexpr (kF16Mma) {
        pa[0] = pack_f16(sc[0][0], sc[0][1]);
        pa[1] = pack_f16(sc[0][2], sc[0][3]);
        pa[2] = pack_f16(sc[1][0], sc[1][1]);
        pa[3] = pack_f16(sc[1][2], sc[1][3]);
      } else {
        // bf16 P carries 8 significant bits; a second bf16 term holds the remainder so
        // P V keeps ~16 bits (P = hi + lo).
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float x0 = sc[q >> 1][2 * (q & 1)], x1 = sc[q >> 1][2 * (q & 1) + 1];
          pa[q] = pack_bf16(x0, x1);
          pl[q] = pack_bf16(x0 - bf16_lo(pa[q]), x1 - bf16_hi(pa[q]));
        }
      }
      {
        const int k0 = kc0 + 2 * cq;
        const bool tail = kc0 + 16 > kv_len;
        // b0/b2 hold keys k0, k0+1 and b1/b3 keys k0+8, k0+9 of the chunk
        const uint32_t m01 = (k0 < kv_len ? 0xffffu : 0u) | (k0 + 1 < kv_len ? 0xffff0000u : 0u);
        const uint32_t m89 =
            (k0 + 8 < kv_len ? 0xffffu : 0u) | (k0 + 9 < kv_len ? 0xffff0000u : 0u);
        if constexpr (C::kPermD) {
          // Lane (gq, cq) reads bytes [gq D/8, (gq + 1) D/8) of V rows 2cq, 2cq+1, 2cq+8,
          // 2cq+9: byte nd of them is output column gq D/8 + nd (fragment column gq of
          // n-tile nd).  A byte permute pairs the two keys of each B operand half.
          constexpr int kW = D / 32;  // 32-bit words of a row per lane
          uint32_t vw[4][kW];
#pragma unroll
          for (int r4 = 0; r4 < 4; ++r4) {
            const uint32_t trow = 16 * ch + 2 * cq + (r4 & 1) + 8 * (r4 >> 1);
            if constexpr (kW % 4 == 0) {
#pragma unroll
              for (int x = 0; x < kW; x += 4) {
                const uint4 v4 =
                    *reinterpret_cast<const uint4*>(vst + C::raw_byte(trow, gq * (D / 8) + 4 * x));
                vw[r4][x] = v4.x;
                vw[r4][x + 1] = v4.y;
                vw[r4][x + 2] = v4.z;
                vw[r4][x + 3] = v4.w;
              }
            } else {
              const uint2 v2 = *reinterpret_cast<const uint2*>(vst + C::raw_byte(trow, gq * (D / 8)));
              vw[r4][0] = v2.x;
              vw[r4][1] = v2.y;
            }
          }
#pragma unroll
          for (int x = 0; x < kW; ++x) {
            const uint32_t p0[2] = {__byte_perm(vw[0][x], vw[1][x], 0x5140),
                                    __byte_perm(vw[0][x], vw[1][x], 0x7362)};
            const uint32_t p1[2] = {__byte_perm(vw[2][x], vw[3][x], 0x5140),
                                    __byte_perm(vw[2][x], vw[3][x], 0x7362)};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t b0 = e4m3x2_to_f16x2(static_cast<uint16_t>(p0[q >> 1] >> (16 * (q & 1))));
              uint32_t b1 = e4m3x2_to_f16x2(static_cast<uint16_t>(p1[q >> 1] >> (16 * (q & 1))));
              if (tail) {
                b0 &= m01;
                b1 &= m89;
              }
              mma_16816<true>(o_acc[4 * x + q], pa, b0, b1);
            }
          }
        } else {
          const uint32_t vbase = smem_addr(vst);
          const uint32_t vr = 16 * ch + (lane & 7) + (((lane >> 3) & 1) << 3);
          const uint32_t dh = lane >> 4;
#pragma unroll
          for (int nd = 0; nd < D / 8; nd += 2) {
            const uint32_t c = (nd & 7) + dh;  // 16-byte chunk within the column block
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(vbase + (nd >> 3) * C::kCBBytes + sw128(vr, c), b0, b1, b2, b3);
            if (tail) {
              b0 &= m01;
              b2 &= m01;
              b1 &= m89;
              b3 &= m89;
            }
            mma_16816<kF16Mma>(o_acc[nd], pa, b0, b1);
            mma_16816<kF16Mma>(o_acc[nd + 1], pa, b2, b3);
            if constexpr (!kF16Mma) {
              mma_16816<kF16Mma>(o_acc[nd], pl, b0, b1);
              mma_16816<kF16Mma>(o_acc[nd + 1], pl, b2, b3);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // Row sums: combine the quad's partial sums.
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 1);
    l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 2);
  }

  if (aborted) s_abort = 1;
  named_bar_sync(1, 32 * C::kConsumerWarps);
  // Split partitions of a decode-shaped q-block that form one cluster merge through
  // distributed shared memory (every CTA reaches both cluster barriers, an aborted one
  // too); otherwise an aborted CTA writes nothing.
  const bool cmerge = WM == 1 && p.cluster_merge != 0;
  if (s_abort && !cmerge) return;
  const bool ok = s_abort == 0;

  const size_t n_part = static_cast<size_t>(p.n_part);
  float* const partial = reinterpret_cast<float*>(pipe + C::kMergeBytes);  // [16][D], m[16], l[16]
  // Rows rr of the warp's fragments: the normalised output (one partition), the
  // partition's max / sum / unnormalised output in the split scratch, or (cluster merge)
  // in this CTA's shared memory.
  auto write_rows = [&]() {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      if (!rv[rr]) continue;
      const size_t row = static_cast<size_t>(rt[rr]) * p.hq + rh[rr];
      if (n_part == 1) {
        const float inv = l_run[rr] > 0.f ? v_scale / l_run[rr] : 0.f;
        const size_t esz = p.out_dtype == UA_DT_F32 ? 4 : 2;
        store_o_row<D, C::kPermD>(o_acc, rr, cq, inv, static_cast<uint8_t*>(p.out) + row * D * esz,
                                  p.out_dtype);
      } else if (cmerge) {
        const int pr = gq + 8 * rr;  // row within the q-block
        if (cq == 0) {
          partial[16 * D + pr] = m_run[rr];
          partial[16 * D + 16 + pr] = l_run[rr];
        }
        store_o_row<D, C::kPermD>(o_acc, rr, cq, v_scale, partial + pr * D, UA_DT_F32);
      } else {
        const size_t w = row * n_part + z;
        if (cq == 0) {
          p.ws_m[w] = m_run[rr];
          p.ws_l[w] = l_run[rr];
        }
        store_o_row<D, C::kPermD>(o_acc, rr, cq, v_scale, p.ws_acc + w * D, UA_DT_F32);
      }
    }
  };
  if constexpr (C::kWN == 1) {
    // Each warp owns its 16 rows: write straight from registers.
    write_rows();
  } else {
    // Four warps hold the same 16 rows over different keys (the pipeline buffers are free:
    // every copy landed and every consumer is done).  Each warp rescales its state to the
    // rows' max (exchanged through shared memory); warp 0 adds the others' partial sums,
    // read in the MMA fragment layout (conflict-free), and writes the rows.
    float* sm_m = reinterpret_cast<float*>(pipe);                      // [4][16]
    float* sm_l = sm_m + C::kConsumerWarps * 16;                       // [4][16]
    float4* sm_o = reinterpret_cast<float4*>(sm_l + C::kConsumerWarps * 16);  // [4][D/8][32]
    if (cq == 0) {
      sm_m[warp * 16 + gq] = m_run[0];
      sm_m[warp * 16 + gq + 8] = m_run[1];
    }
    named_bar_sync(1, 32 * C::kConsumerWarps);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = gq + 8 * rr;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::kConsumerWarps; ++w) M = fmaxf(M, sm_m[w * 16 + row]);
      const float wt = M == -INFINITY ? 0.f : fast_exp2(m_run[rr] - M);
      m_run[rr] = M;
      l_run[rr] *= wt;
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        o_acc[nd][2 * rr] *= wt;
        o_acc[nd][2 * rr + 1] *= wt;
      }
    }
    if (warp != 0) {
      if (cq == 0) {
        sm_l[warp * 16 + gq] = l_run[0];
        sm_l[warp * 16 + gq + 8] = l_run[1];
      }
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd)
        sm_o[(warp * (D / 8) + nd) * 32 + lane] =
            make_float4(o_acc[nd][0], o_acc[nd][1], o_acc[nd][2], o_acc[nd][3]);
    }
    named_bar_sync(1, 32 * C::kConsumerWarps);
    if (warp == 0) {
#pragma unroll
      for (int w = 1; w < C::kConsumerWarps; ++w) {
        l_run[0] += sm_l[w * 16 + gq];
        l_run[1] += sm_l[w * 16 + gq + 8];
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
          const float4 o4 = sm_o[(w * (D / 8) + nd) * 32 + lane];
          o_acc[nd][0] += o4.x;
          o_acc[nd][1] += o4.y;
          o_acc[nd][2] += o4.z;
          o_acc[nd][3] += o4.w;
        }
      }
      if (ok) write_rows();
    }
  }
  if (!cmerge) return;

  // Cluster merge: the cluster is the n_part partitions (grid z) of cluster_y kv-heads of
  // this q-block slot; partition zz of this kv-head is the cluster's CTA
  // cluster_ctaid.y + cluster_y * zz.  Row r of the q-block is merged by partition
  // r mod n_part, one warp a row.
  cluster_sync();
  {
    const int np = p.n_part;
    const uint32_t cy = cluster_nctaid_y(), yc = cluster_ctaid_y();
    const uint32_t part_s = smem_addr(partial);
    const size_t esz = p.out_dtype == UA_DT_F32 ? 4 : 2;
    for (int k = warp;; k += C::kConsumerWarps) {
      const int r = z + np * k;  // row within the q-block
      if (r >= r1 - r0) break;
      const int tok = q0 + (r0 + r) / G;
      if (tok >= p.total_q) break;
      const size_t orow = static_cast<size_t>(tok) * p.hq + g * G + (r0 + r) % G;
      cluster_merge_row<D>(part_s + (16 * D + r) * 4, part_s + (16 * D + 16 + r) * 4,
                           part_s + r * D * 4, np, yc, cy, lane,
                           static_cast<uint8_t*>(p.out) + orow * D * esz, p.out_dtype);
    }
  }
  // no CTA leaves while the cluster still reads its shared memory (those reads have
  // returned: a relaxed arrival, which need not wait for the output stores)
  cluster_sync_relaxed();
}

template <int D, int KV, int WM, bool FEAT, bool TMA>
cudaError_t launch_tile_t(const TileParams& tp, dim3 grid, int cluster_y, int cluster_z,
                          cudaStream_t stream) {
  using C = TileCfg<D, KV, WM>;
  auto kern = ua_attn_tile_kernel<D, KV, WM, FEAT, TMA>;
  static std::atomic<unsigned long long> configured{0};  // one bit per device
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    // clusters of up to 16 CTAs (the partitions of a decode slot)
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
    configured.fetch_or(bit);
  }
  return launch_pdl_cluster(kern, grid, dim3(C::kThreads), C::kSmemBytes, stream, cluster_y,
                            cluster_z, tp);
}

template <int D>
cudaError_t launch_tile_dispatch(const TileParams& tp, dim3 grid, int wm, int kv, bool feat,
                                 bool tma, int cluster_y, int cluster_z, cudaStream_t s) {
#define UA_TILE_CASE(KVV, WMV)                                                        \
  if (kv == KVV && wm == WMV) {                                                       \
    if (tma)                                                                          \
      return feat ? launch_tile_t<D, KVV, WMV, true, true>(tp, grid, cluster_y, cluster_z, s)    \
                  : launch_tile_t<D, KVV, WMV, false, true>(tp, grid, cluster_y, cluster_z, s);  \
    return feat ? launch_tile_t<D, KVV, WMV, true, false>(tp, grid, cluster_y, cluster_z, s)     \
                : launch_tile_t<D, KVV, WMV, false, false>(tp, grid, cluster_y, cluster_z, s);   \
  }
  UA_TILE_CASE(KV_F16, 1)
  UA_TILE_CASE(KV_F16, 4)
  UA_TILE_CASE(KV_BF16, 1)
  UA_TILE_CASE(KV_BF16, 4)
  UA_TILE_CASE(KV_E4M3, 1)
  UA_TILE_CASE(KV_E4M3, 4)
#undef UA_TILE_CASE
  return cudaErrorInvalidValue;
}

template <int D>
int tile_ctas_per_sm_d(int kv, int wm) {
  if (kv == KV_E4M3)
    return wm == 1 ? TileCfg<D, KV_E4M3, 1>::kMinBlocks : TileCfg<D, KV_E4M3, 4>::kMinBlocks;
  return wm == 1 ? TileCfg<D, KV_BF16, 1>::kMinBlocks : TileCfg<D, KV_BF16, 4>::kMinBlocks;
}

}  // namespace ua
