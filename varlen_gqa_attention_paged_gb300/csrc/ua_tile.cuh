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
//   warp 4      producer: for each tile of T keys it looks every key up in the block
//               table and issues one bulk async copy (TMA engine) per K row and per V
//               row into a STAGES-deep shared-memory ring, completing on an mbarrier.
//   warps 0..3  consumers: QK^T and P.V on tensor cores (mma.sync m16n8k16, fp32
//               accumulate), score transform, online softmax in base 2 with quad
//               shuffles, fp8 e4m3 -> f16 dequant of the tile in shared memory.
//   WM = 1 (decode-shaped q-blocks, BM = 16): the four consumer warps share the 16
//          rows and each takes 16 keys of every tile; their states merge at the end.
//   WM = 4 (BM = 64): each consumer warp owns 16 rows and walks every key.
#pragma once

#include <atomic>
#include <climits>

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

template <int D, int KV, int WM>
struct TileCfg {
  static constexpr int kConsumerWarps = 4;
  static constexpr int kThreads = 32 * (kConsumerWarps + 1);
  static constexpr int kWN = kConsumerWarps / WM;  // warps sharing one 16-row m-tile
  static constexpr int kT = 64;                    // keys per pipeline stage
  static constexpr int kEsz = KvTraits<KV>::kEsz;
  static constexpr int kRowBytes = D * kEsz;       // one K or V row in the cache
  static constexpr int kRawStride = kRowBytes + 16;     // padded: ldmatrix rows hit 8 bank groups
  static constexpr int kF16Stride = D * 2 + 16;
  static constexpr int kStageBytes = 2 * kT * kRawStride;  // K rows then V rows
  static constexpr int kConvBytes = (KV == KV_E4M3) ? kConsumerWarps * 2 * 16 * kF16Stride : 0;
  static constexpr int kMergeBytes = (kWN > 1) ? kConsumerWarps * 16 * (D + 2) * 4 : 0;
  static constexpr int kStages = (4 * kStageBytes + kConvBytes <= 200 * 1024) ? 4 : 3;
  static constexpr int kPipeBytes =
      (kStages * kStageBytes > kMergeBytes) ? kStages * kStageBytes : kMergeBytes;
  static constexpr int kSmemBytes = kPipeBytes + kConvBytes + 2 * kStages * 8;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kRowBytes % 16 == 0, "bulk copies move 16-byte multiples");
};

// Sequence owning q-block slot x: the last b with floor(cu[b] * G / BM) + b <= x
// (a monotone slot layout that leaves at most one idle slot per sequence).
__device__ __forceinline__ int find_seq(const int32_t* __restrict__ cu, int num_seqs, int x,
                                        int group, int bm) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int start = static_cast<int>((static_cast<long long>(__ldg(cu + mid)) * group) / bm) + mid;
    if (start <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <int D, int KV, int WM, bool FEAT>
__global__ void __launch_bounds__(160, 1) ua_attn_tile_kernel(const __grid_constant__ AttnParams p) {
  using C = TileCfg<D, KV, WM>;
  constexpr int T = C::kT;
  constexpr int S = C::kStages;
  constexpr bool kF16Mma = KvTraits<KV>::kF16Mma;
  constexpr int BM = 16 * WM;

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* const pipe = smem;
  uint8_t* const conv = smem + C::kPipeBytes;
  uint64_t* const full = reinterpret_cast<uint64_t*>(conv + C::kConvBytes);
  uint64_t* const empty = full + S;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int z = blockIdx.z;
  const int G = p.group;

  // ---- which rows and keys this CTA owns
  const int b = find_seq(p.cu_seqlens_q, p.num_seqs, blockIdx.x, G, BM);
  const int q0 = __ldg(p.cu_seqlens_q + b);
  const int q_len = __ldg(p.cu_seqlens_q + b + 1) - q0;
  const int rows_b = q_len * G;
  const int slot0 = static_cast<int>((static_cast<long long>(q0) * G) / BM) + b;
  const int r0 = (static_cast<int>(blockIdx.x) - slot0) * BM;
  if (r0 < 0 || r0 >= rows_b) return;  // idle slot: uniform for the CTA
  const int r1 = min(r0 + BM, rows_b);
  const int kv_len = __ldg(p.seq_lens_k + b);
  const int ctx = kv_len - q_len;
  const int pos_first = ctx + r0 / G;
  const int pos_last = ctx + (r1 - 1) / G;
  const int hi = max(0, min(pos_last + 1, kv_len));
  const int lo = min(hi, p.window_left >= 0 ? max(0, pos_first - p.window_left) : 0);
  int part = (hi - lo + p.n_part - 1) / p.n_part;
  part = (part + 15) & ~15;
  const int ks = min(lo + z * part, hi);
  const int ke = min(ks + part, hi);
  const int ntiles = (ke - ks + T - 1) / T;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kConsumerWarps);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == C::kConsumerWarps) {
    // ======================================================== producer warp
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    const size_t slot_pitch = static_cast<size_t>(p.hkv) * C::kRowBytes;
    const uint8_t* kg = static_cast<const uint8_t*>(p.k) + static_cast<size_t>(g) * C::kRowBytes;
    const uint8_t* vg = static_cast<const uint8_t*>(p.v) + static_cast<size_t>(g) * C::kRowBytes;
    const uint64_t policy = l2_policy_evict_first();
    int issued = 0;
    for (int t = 0; t < ntiles; ++t) {
      const int s = t % S;
      if (t >= S && !mbar_wait_bounded(&empty[s], ((t / S) & 1) ^ 1, p.status, DEV_TIMEOUT)) break;
      const int key0 = ks + t * T;
      const int nvalid = min(T, ke - key0);
      uint8_t* kdst = pipe + s * C::kStageBytes;
      uint8_t* vdst = kdst + T * C::kRawStride;
      size_t off[T / 32];
      bool ok[T / 32];
      int bytes = 0;
#pragma unroll
      for (int rr = 0; rr < T / 32; ++rr) {
        const int row = lane + 32 * rr;
        ok[rr] = false;
        off[rr] = 0;
        if (row < nvalid) {
          const int key = key0 + row;
          const int col = key / p.block_size;
          const int blk = col < p.max_blocks_per_seq ? __ldg(bt + col) : -1;
          if (static_cast<unsigned>(blk) < static_cast<unsigned>(p.num_blocks)) {
            ok[rr] = true;
            off[rr] = (static_cast<size_t>(blk) * p.block_size + key % p.block_size) * slot_pitch;
            bytes += 2 * C::kRowBytes;
          } else {
            atomicOr(p.status, DEV_BAD_BLOCK);
          }
        }
        if (!ok[rr]) {  // rows with no key behind them read as zero
          uint4* kz = reinterpret_cast<uint4*>(kdst + row * C::kRawStride);
          uint4* vz = reinterpret_cast<uint4*>(vdst + row * C::kRawStride);
#pragma unroll
          for (int c = 0; c < C::kRowBytes / 16; ++c) {
            kz[c] = make_uint4(0, 0, 0, 0);
            vz[c] = make_uint4(0, 0, 0, 0);
          }
        }
      }
      bytes = __reduce_add_sync(0xffffffffu, bytes);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(bytes));
      __syncwarp();
#pragma unroll
      for (int rr = 0; rr < T / 32; ++rr) {
        if (ok[rr]) {
          const int row = lane + 32 * rr;
          bulk_copy_g2s(kdst + row * C::kRawStride, kg + off[rr], C::kRowBytes, &full[s], policy);
          bulk_copy_g2s(vdst + row * C::kRawStride, vg + off[rr], C::kRowBytes, &full[s], policy);
        }
      }
      issued = t + 1;
    }
    // Never leave copies in flight into this CTA's shared memory.
    for (int t = max(0, issued - S); t < issued; ++t)
      mbar_wait_bounded(&full[t % S], (t / S) & 1, p.status, DEV_TIMEOUT);
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
      const int col = kk * 16 + 2 * cq + 8 * (j >> 1);
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

  uint8_t* const conv_k = conv + warp * 2 * 16 * C::kF16Stride;
  uint8_t* const conv_v = conv_k + 16 * C::kF16Stride;
  bool aborted = false;

  for (int t = 0; t < ntiles; ++t) {
    const int s = t % S;
    if (!mbar_wait_bounded(&full[s], (t / S) & 1, p.status, DEV_TIMEOUT)) {
      aborted = true;
      break;
    }
    const uint8_t* kst = pipe + s * C::kStageBytes;
    const uint8_t* vst = kst + T * C::kRawStride;
    const int key_tile = ks + t * T;

#pragma unroll 1
    for (int ch = (WM == 1 ? kgp : 0); ch < 4; ch += (WM == 1 ? 4 : 1)) {
      const int kc0 = key_tile + 16 * ch;
      if (!tile_any || kc0 >= ke || kc0 > pmax || kc0 + 16 <= lomin) continue;

      uint32_t kbase, vbase;
      int stride;
      if constexpr (KV == KV_E4M3) {
        // Dequantise the chunk's 16 K rows and 16 V rows to f16 (exact); the scales
        // are applied to the scores and to the output instead.
        __syncwarp();
#pragma unroll
        for (int it = 0; it < (2 * 16 * D / 16) / 32; ++it) {
          const int idx = it * 32 + lane;                // one 16-code group per lane
          const int which = idx / (16 * D / 16);         // 0: K, 1: V
          const int rem = idx % (16 * D / 16);
          const int row = rem / (D / 16), grp = rem % (D / 16);
          const uint8_t* src = (which ? vst : kst) + (16 * ch + row) * C::kRawStride + grp * 16;
          const uint4 raw = *reinterpret_cast<const uint4*>(src);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t h[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            h[2 * q] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] & 0xffffu));
            h[2 * q + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] >> 16));
          }
          uint8_t* dst = (which ? conv_v : conv_k) + row * C::kF16Stride + grp * 32;
          reinterpret_cast<uint4*>(dst)[0] = make_uint4(h[0], h[1], h[2], h[3]);
          reinterpret_cast<uint4*>(dst)[1] = make_uint4(h[4], h[5], h[6], h[7]);
        }
        __syncwarp();
        kbase = smem_addr(conv_k);
        vbase = smem_addr(conv_v);
        stride = C::kF16Stride;
      } else {
        kbase = smem_addr(kst + 16 * ch * C::kRawStride);
        vbase = smem_addr(vst + 16 * ch * C::kRawStride);
        stride = C::kRawStride;
      }

      // ---- S = Q K^T for 16 keys (two n8 chunks)
      float sc[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[n][e] = 0.f;
      {
        const uint32_t lane_addr =
            kbase + ((lane & 7) + ((lane >> 4) << 3)) * stride + (((lane >> 3) & 1) << 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(lane_addr + kk * 32, b0, b1, b2, b3);
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
            if (p.softcap > 0.f) x = p.softcap * tanhf(x * inv_softcap);
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

      // ---- online softmax (rows gq, gq + 8; a row's 16 scores sit in one quad)
      float alpha[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        float mx = fmaxf(fmaxf(sc[0][2 * rr], sc[0][2 * rr + 1]),
                         fmaxf(sc[1][2 * rr], sc[1][2 * rr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run[rr], mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        alpha[rr] = fast_exp2(m_run[rr] - m_use);
        m_run[rr] = m_new;
        float rs = 0.f;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          sc[n][2 * rr] = fast_exp2(sc[n][2 * rr] - m_use);
          sc[n][2 * rr + 1] = fast_exp2(sc[n][2 * rr + 1] - m_use);
          rs += sc[n][2 * rr] + sc[n][2 * rr + 1];
        }
        l_run[rr] = l_run[rr] * alpha[rr] + rs;
      }
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        o_acc[nd][0] *= alpha[0];
        o_acc[nd][1] *= alpha[0];
        o_acc[nd][2] *= alpha[1];
        o_acc[nd][3] *= alpha[1];
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
        const uint32_t lane_addr =
            vbase + ((lane & 7) + (((lane >> 3) & 1) << 3)) * stride + ((lane >> 4) << 4);
#pragma unroll
        for (int nd = 0; nd < D / 8; nd += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(lane_addr + nd * 16, b0, b1, b2, b3);
          mma_16816<kF16Mma>(o_acc[nd], pa, b0, b1);
          mma_16816<kF16Mma>(o_acc[nd + 1], pa, b2, b3);
          if constexpr (!kF16Mma) {
            mma_16816<kF16Mma>(o_acc[nd], pl, b0, b1);
            mma_16816<kF16Mma>(o_acc[nd + 1], pl, b2, b3);
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
  if (s_abort) return;

  const size_t n_part = static_cast<size_t>(p.n_part);
  if constexpr (C::kWN == 1) {
    // Each warp owns its 16 rows: write straight from registers.
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      if (!rv[rr]) continue;
      const size_t row = static_cast<size_t>(rt[rr]) * p.hq + rh[rr];
      if (n_part == 1) {
        const float inv = l_run[rr] > 0.f ? v_scale / l_run[rr] : 0.f;
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
          const int col = nd * 8 + 2 * cq;
          const float x0 = o_acc[nd][2 * rr] * inv, x1 = o_acc[nd][2 * rr + 1] * inv;
          if (p.out_dtype == UA_DT_F32) {
            *reinterpret_cast<float2*>(static_cast<float*>(p.out) + row * D + col) =
                make_float2(x0, x1);
          } else {
            const uint32_t v = p.out_dtype == UA_DT_BF16 ? pack_bf16(x0, x1) : pack_f16(x0, x1);
            *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + row * D + col) = v;
          }
        }
      } else {
        const size_t w = row * n_part + z;
        if (cq == 0) {
          p.ws_m[w] = m_run[rr];
          p.ws_l[w] = l_run[rr];
        }
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
          const int col = nd * 8 + 2 * cq;
          *reinterpret_cast<float2*>(p.ws_acc + w * D + col) =
              make_float2(o_acc[nd][2 * rr] * v_scale, o_acc[nd][2 * rr + 1] * v_scale);
        }
      }
    }
  } else {
    // Four warps hold the same 16 rows over different keys: merge through shared memory
    // (the pipeline buffers are free: every copy landed and every consumer is done).
    float* sm_m = reinterpret_cast<float*>(pipe);
    float* sm_l = sm_m + C::kConsumerWarps * 16;
    float* sm_o = sm_l + C::kConsumerWarps * 16;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = gq + 8 * rr;
      if (cq == 0) {
        sm_m[warp * 16 + row] = m_run[rr];
        sm_l[warp * 16 + row] = l_run[rr];
      }
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        const int col = nd * 8 + 2 * cq;
        *reinterpret_cast<float2*>(sm_o + (warp * 16 + row) * D + col) =
            make_float2(o_acc[nd][2 * rr], o_acc[nd][2 * rr + 1]);
      }
    }
    named_bar_sync(1, 32 * C::kConsumerWarps);
    const int tid = threadIdx.x;  // 0..127
    for (int idx = tid; idx < 16 * (D / 4); idx += 32 * C::kConsumerWarps) {
      const int row = idx / (D / 4);
      const int col = (idx % (D / 4)) * 4;
      const int r = r0 + row;
      if (r >= r1 || q0 + r / G >= p.total_q) continue;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::kConsumerWarps; ++w) M = fmaxf(M, sm_m[w * 16 + row]);
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < C::kConsumerWarps; ++w) {
          const float wt = fast_exp2(sm_m[w * 16 + row] - M);
          L += sm_l[w * 16 + row] * wt;
          const float4 o4 = *reinterpret_cast<const float4*>(sm_o + (w * 16 + row) * D + col);
          acc.x += o4.x * wt;
          acc.y += o4.y * wt;
          acc.z += o4.z * wt;
          acc.w += o4.w * wt;
        }
      }
      const int i = r / G;
      const size_t orow = static_cast<size_t>(q0 + i) * p.hq + g * G + r % G;
      if (n_part == 1) {
        const float inv = L > 0.f ? v_scale / L : 0.f;
        const float x0 = acc.x * inv, x1 = acc.y * inv, x2 = acc.z * inv, x3 = acc.w * inv;
        if (p.out_dtype == UA_DT_F32) {
          *reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * D + col) =
              make_float4(x0, x1, x2, x3);
        } else if (p.out_dtype == UA_DT_BF16) {
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + orow * D + col) =
              make_uint2(pack_bf16(x0, x1), pack_bf16(x2, x3));
        } else {
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + orow * D + col) =
              make_uint2(pack_f16(x0, x1), pack_f16(x2, x3));
        }
      } else {
        const size_t w = orow * n_part + z;
        if (col == 0) {
          p.ws_m[w] = M;
          p.ws_l[w] = L;
        }
        *reinterpret_cast<float4*>(p.ws_acc + w * D + col) =
            make_float4(acc.x * v_scale, acc.y * v_scale, acc.z * v_scale, acc.w * v_scale);
      }
    }
  }
}

template <int D, int KV, int WM, bool FEAT>
cudaError_t launch_tile_t(const AttnParams& p, dim3 grid, cudaStream_t stream) {
  using C = TileCfg<D, KV, WM>;
  auto kern = ua_attn_tile_kernel<D, KV, WM, FEAT>;
  static std::atomic<unsigned long long> configured{0};  // one bit per device
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    configured.fetch_or(bit);
  }
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_tile_dispatch(const AttnParams& p, dim3 grid, int wm, int kv, bool feat,
                                 cudaStream_t s) {
#define UA_TILE_CASE(KVV, WMV)                                                  \
  if (kv == KVV && wm == WMV)                                                   \
    return feat ? launch_tile_t<D, KVV, WMV, true>(p, grid, s)                  \
                : launch_tile_t<D, KVV, WMV, false>(p, grid, s);
  UA_TILE_CASE(KV_F16, 1)
  UA_TILE_CASE(KV_F16, 4)
  UA_TILE_CASE(KV_BF16, 1)
  UA_TILE_CASE(KV_BF16, 4)
  UA_TILE_CASE(KV_E4M3, 1)
  UA_TILE_CASE(KV_E4M3, 4)
#undef UA_TILE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace ua
