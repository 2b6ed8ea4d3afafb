// ua_decode.cuh -- the key-major decode tile kernel of libua.so (included by
// ua_decode_d*.cu): decode batches with at most 8 rows (query token x head) per kv-head,
// fp16 / bf16 / fp8-e4m3 caches paged in blocks of a multiple of 16, head_dim <= 128.
//
// The tile kernel (ua_tile.cuh) puts a q-block's rows on the MMA's M side; a decode
// q-block has only G rows (often 4), so most of that 16-row tile's softmax and P.V work
// is padding.  Here the operands turn around, with 16 keys on M and the rows on N (8):
//   S^T (16 keys x 8 rows)  = K (16 keys x 16 d) . Q^T (16 d x 8 rows),      D/16 MMAs
//   O^T (16 d x 8 rows)    += V^T (16 d x 16 keys) . P^T (16 keys x 8 rows), D/16 MMAs
// per 16-key chunk (mma.sync m16n8k16, fp32 accumulate).  P^T reaches the B operand of the
// second product through an in-register 8x8 transpose (movmatrix) of the S^T accumulator.
// A thread holds half the accumulators of the row-major tile, so three CTAs (twelve
// consumer warps) fit an SM.  Everything else follows the tile kernel: one producer warp
// streams 64-key stages of one-head TMA page boxes through an mbarrier ring; the consumers
// take 16 keys of every stage each (the FA-RDNA2 "Change" 1 packing of a kv-head's GQA
// heads into one tile; the aiter split-K partitioning); fp8 codes become f16 operands in
// registers with a permuted head dimension.  The q-block's rows leave a CTA as one
// partial per row in shared memory: written out (one partition), merged with the other
// partitions of the cluster through distributed shared memory, or handed to the merge
// kernel through the global scratch.
#pragma once

#include "ua_tile.cuh"

namespace ua {

// Bring the line holding `ptr` into L2 (a hint: no value is read, and L2 is coherent, so a
// write by an earlier kernel is never missed by a later load).
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// W consumer warps (4, or 8 for grids of at most one CTA per SM), each taking 16 keys of
// every stage.  HP kv-heads per CTA (1, or 2 for fp8 caches with at most 4 rows per kv-head:
// the two heads' q-blocks share the MMA's 8 columns, and one page box carries both heads).
template <int D, int KV, int W = 4, int HP = 1>
struct DecCfg {
  static constexpr int kConsumerWarps = W;
  static constexpr int kThreads = 32 * (kConsumerWarps + 1);
  static constexpr int kRows = 8;                  // rows of a q-block (the MMA's N)
  static constexpr int kHP = HP;
  static constexpr int kRH = kRows / HP;           // rows of one kv-head (columns kRH h ..)
  static constexpr int kT = 16 * W;                // keys per pipeline stage (W pages of 16)
  static constexpr int kKPL = kT / 32;             // keys whose scales one producer lane stages
  static constexpr int kEsz = KvTraits<KV>::kEsz;
  static constexpr int kRowBytes = D * kEsz;       // one K or V row in the cache
  static constexpr bool kSwz = kRowBytes >= 128;   // 128-byte swizzled column blocks
  static constexpr int kCBW = kSwz ? 128 : kRowBytes;
  static constexpr int kCB = kRowBytes / kCBW;
  static constexpr int kCBBytes = kT * HP * kCBW;  // one column block of a stage's keys x heads
  static constexpr int kStageBytes = 2 * kCB * kCBBytes;  // K then V
  static constexpr bool kPermD = KV == KV_E4M3;     // fp8: permuted head dimension
  static constexpr int kMT = D / 16;                // O^T m-tiles of 16 d
  // end of a CTA: the warps' maxima and sums [4][8] each, then their O^T fragments
  // [4][kMT][32] float4; then the CTA's partial rows [8][D], maxima [8] and sums [8]
  static constexpr int kMergeBytes = kConsumerWarps * (2 * kRows + kMT * 32 * 4) * 4;
  static constexpr int kPartBytes = kRows * (D + 2) * 4;
  // four consumer warps: three CTAs per SM, at most ~72 KB of shared memory each; two
  // kv-heads a CTA: two CTAs per SM with three 32 KB stages (the fp8 decode is bound by the
  // SM's issue rate where three CTAs share an SM: measured 18.7 against 20.0 us for the
  // sliding-window decode); eight consumer warps: one CTA per SM
  static constexpr int kBudget = HP == 2 ? 100 * 1024 : W == 4 ? 72 * 1024 : 200 * 1024;
  static constexpr int kStagesFit = kBudget / kStageBytes;
  static constexpr int kStages = kStagesFit < 2 ? 2 : (kStagesFit > 6 ? 6 : kStagesFit);
  static constexpr int kPipeRaw = (kStages * kStageBytes > kMergeBytes + kPartBytes)
                                      ? kStages * kStageBytes
                                      : kMergeBytes + kPartBytes;
  static constexpr int kPipeBytes = (kPipeRaw + 1023) & ~1023;
  // fp8 per-token scales of a stage's keys, K then V, behind the barriers
  static constexpr int kScaleBytes = kPermD ? kStages * 2 * kT * 4 : 0;
  static constexpr int kSmemBytes = 1024 + kPipeBytes + 2 * kStages * 8 + kScaleBytes;
  static constexpr int kMinBlocks = W != 4    ? 1
                                   : HP == 2  ? 2
                                   : (3 * (kSmemBytes + 1024) <= 228 * 1024) ? 3
                                                                             : 2;
  static_assert(W == 4 || W == 8, "four or eight consumer warps");
  static_assert(D <= 128, "the key-major decode tile covers head_dim <= 128");
  static_assert(kRowBytes % kCBW == 0 && kCBW % 16 == 0, "rows are whole column blocks");
  static_assert(HP == 1 || (HP == 2 && KV == KV_E4M3 && W == 4),
                "two kv-heads a CTA: fp8 caches, four consumer warps");

  // Line of head h's row of stage key r in a column block: a page box of HP heads lands
  // head by head (16 lines each), so a line's swizzle phase is r mod 8 for every head.
  static __device__ __forceinline__ uint32_t line(uint32_t r, uint32_t h) {
    return HP == 1 ? r : ((r / 16) * HP + h) * 16 + (r % 16);
  }
  // Byte offset of byte x of head h's row of stage key r in a K or V stage.
  static __device__ __forceinline__ uint32_t raw_byte(uint32_t r, uint32_t x, uint32_t h = 0) {
    const uint32_t l = line(r, h);
    if constexpr (kSwz) return (x / 128) * kCBBytes + sw128(l, (x % 128) / 16) + (x & 15u);
    else return l * kCBW + x;
  }
  // Output column of O^T fragment row i (0..15) of m-tile m: the natural order, or (fp8)
  // the permuted order that makes each lane's V bytes one contiguous run.
  static __device__ __forceinline__ int out_col(int m, int i) {
    if constexpr (kPermD) return (i & 7) * (D / 8) + 2 * m + (i >> 3);
    else return 16 * m + i;
  }
};

// QT: e4m3 terms of Q for fp8 caches (2 for a bf16 q, 3 for an f16 q); unused otherwise.
// W: consumer warps of a CTA.  HP: kv-heads of a CTA (grid y = H_kv / HP).
template <int D, int KV, bool FEAT, int QT, int W, int HP = 1>
__global__ void __launch_bounds__(DecCfg<D, KV, W, HP>::kThreads,
                                  (DecCfg<D, KV, W, HP>::kMinBlocks))
    ua_decode_kernel(const __grid_constant__ TileParams tp) {
  using C = DecCfg<D, KV, W, HP>;
  constexpr int T = C::kT;
  constexpr int S = C::kStages;
  constexpr int NR = C::kRows;
  constexpr int RH = C::kRH;
  constexpr bool kF16Mma = KvTraits<KV>::kF16Mma;
  const AttnParams& p = tp.p;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* const smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* const pipe = smem;
  uint64_t* const full = reinterpret_cast<uint64_t*>(smem + C::kPipeBytes);
  uint64_t* const empty = full + S;
  float* const sks = reinterpret_cast<float*>(empty + S);  // [S][T] K scales (per-token fp8)
  float* const svs = sks + S * T;                           // [S][T] V scales
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.y * HP;  // first kv-head of the CTA
  const int z = blockIdx.z;
  const int G = p.group;
  // fp8 per-token scales (aiter PR #3962 test matrix): key j's K and V rows carry their own
  // scale, element (block, slot, g) of two separately strided arrays (one kv-head a CTA)
  const bool tok = KV == KV_E4M3 && HP == 1 && p.k_scale_tok != nullptr;

  // Set-up that reads no input runs before the wait on the previous grid (programmatic
  // dependent launch), so it overlaps that grid's tail: the barriers, and the cache
  // tensor maps fetched into the descriptor cache.
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // lane 0's arrival with the page bytes (per-token scales: their copies too)
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kConsumerWarps);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == C::kConsumerWarps) {
    if (lane == 0) {
      tma_prefetch_desc(&tp.tmap_k);
      tma_prefetch_desc(&tp.tmap_v);
      prefetch_l2(p.cu_seqlens_q + blockIdx.x);
      prefetch_l2(p.seq_lens_k + blockIdx.x);
    }
    // the sequence's block-table row (slot x is sequence x), one 128-byte line a lane, up to
    // 256 lines (8192 pages)
    const int32_t* btr = p.block_table + static_cast<size_t>(blockIdx.x) * p.max_blocks_per_seq;
    const int bt_end = min(p.max_blocks_per_seq, 256 * 32);
    for (int i = 32 * lane; i < bt_end; i += 32 * 32) prefetch_l2(btr + i);
  }
  __syncthreads();
  grid_dependency_wait();
  grid_launch_dependents();

  // Slot x is sequence x (decode plans); its rows q_len x G of each kv-head, at most RH
  // (8 / HP).  Column c of the q-block is row c mod RH of kv-head g + c / RH.
  const int b = static_cast<int>(blockIdx.x);
  const int q0 = __ldg(p.cu_seqlens_q + b);
  const int q_len = __ldg(p.cu_seqlens_q + b + 1) - q0;
  const int kv_len = __ldg(p.seq_lens_k + b);
  const int rows_b = q_len * G;
  if (rows_b > RH && threadIdx.x == 0 && z == 0 && g == 0)
    atomicOr(p.status, DEV_BAD_SHAPE);  // q_len above max_seqlen_q: rows past RH unwritten
  if (rows_b <= 0) return;              // idle slot: uniform for the slot's cluster
  const int nr = min(rows_b, RH);
  const int ctx = kv_len - q_len;
  const int pos_first = ctx;
  const int pos_last = ctx + (nr - 1) / G;
  const int hi = max(0, min(pos_last + 1, kv_len));
  // the walk starts on a 16-key page boundary; keys before a row's window are masked
  const int lo = min(hi, p.window_left >= 0 ? max(0, pos_first - p.window_left) : 0) & ~15;
  int part = (hi - lo + p.n_part - 1) / p.n_part;
  part = (part + 15) & ~15;
  const int ks = min(lo + z * part, hi);
  const int ke = min(ks + part, hi);
  const int ntiles = (ke - ks + T - 1) / T;
  const bool cmerge = p.cluster_merge != 0;

  if (warp == C::kConsumerWarps) {
    // ======================================================== producer warp
    // lane j < W owns page slice j (keys key0 + 16j .. +15) of every tile: one TMA box of
    // 16 cache rows per column block, K and V; rows with no key read the zero-filled row
    // coordinate past the cache.
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    const uint64_t policy = l2_policy_evict_first();
    const int bs = p.block_size;
    const int oob = p.num_blocks * bs;
    // this lane's cache row of tile t
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
    // one stage's page boxes, K and V, on stage s's full barrier
    auto issue = [&](int s, int row) {
      uint8_t* kdst = pipe + s * C::kStageBytes;
      uint8_t* vdst = kdst + C::kCB * C::kCBBytes;
      if (lane < T / 16) {
#pragma unroll
        for (int cb = 0; cb < C::kCB; ++cb) {
          const int x = cb * (C::kCBW / C::kEsz);
          uint8_t* const kd = kdst + cb * C::kCBBytes + lane * 16 * HP * C::kCBW;
          uint8_t* const vd = vdst + cb * C::kCBBytes + lane * 16 * HP * C::kCBW;
          if constexpr (HP == 1) {  // view [row][head][d]: box {cols, 1 head, 16 rows}
            tma_load_3d(kd, &tp.tmap_k, x, g, row, &full[s], policy);
            tma_load_3d(vd, &tp.tmap_v, x, g, row, &full[s], policy);
          } else {  // view [head][row][d]: box {cols, 16 rows, HP heads}, head by head
            tma_load_3d(kd, &tp.tmap_k, x, row, g, &full[s], policy);
            tma_load_3d(vd, &tp.tmap_v, x, row, g, &full[s], policy);
          }
        }
      }
    };
    int issued = 0;
    // Per-token scales of this lane's kKPL keys kKPL lane .. of each stage (one page, whose
    // cache row a page lane holds): 4-byte cp.async copies into the stage's scale slots (0
    // past the walk or for a bad block), tracked by the stage's full barrier, so the
    // producer never waits for them.  (With the scales loaded into registers a tile ahead
    // the producer stalled on them: 24.1 against 20.2 us for the sliding-window decode with
    // no scale loads at all.)
    constexpr int KPL = C::kKPL;
    int row_next = ntiles > 0 ? page_row(0) : oob;
    for (int t = 0; t < ntiles; ++t) {
      const int s = t % S;
      const int row = row_next;
      if (t + 1 < ntiles) row_next = page_row(t + 1);  // block-table lookups one tile ahead
      if (t >= S && !mbar_wait_bounded(&empty[s], ((t / S) & 1) ^ 1, p.status, DEV_TIMEOUT))
        break;
      if (tok) {
        const int rowp = __shfl_sync(0xffffffffu, row, (KPL * lane) / 16);
        const int blk = rowp / bs;
#pragma unroll
        for (int e = 0; e < KPL; ++e) {
          const int kt = KPL * lane + e;  // key within the stage
          float* const ksd = sks + s * T + kt;
          float* const vsd = svs + s * T + kt;
          if (ks + t * T + kt < ke && rowp != oob) {
            const long long slot = rowp % bs + kt % 16;
            cp_async_4(ksd, p.k_scale_tok + blk * p.k_scale_stride[0] +
                                slot * p.k_scale_stride[1] + g * p.k_scale_stride[2]);
            cp_async_4(vsd, p.v_scale_tok + blk * p.v_scale_stride[0] +
                                slot * p.v_scale_stride[1] + g * p.v_scale_stride[2]);
          } else {
            *ksd = 0.f;
            *vsd = 0.f;
          }
        }
        // (each lane's copies raise the barrier's pending count now, before lane 0's
        // arrival below can complete the phase)
        cp_async_arrive(&full[s]);
        __syncwarp();
      }
      if (lane == 0) mbar_arrive_expect_tx(&full[s], C::kStageBytes);
      __syncwarp();
      issue(s, row);
      issued = t + 1;
    }
    // Never leave copies in flight into this CTA's shared memory.
    for (int t = max(0, issued - S); t < issued; ++t)
      mbar_wait_bounded(&full[t % S], (t / S) & 1, p.status, DEV_TIMEOUT);
    if (cmerge) {  // the consumers' two cluster barriers
      cluster_sync();
      cluster_sync_relaxed();
    }
    return;
  }

  // ========================================================== consumer warps
  const int gq = lane >> 2, cq = lane & 3;

  float k_scale = 1.f, v_scale = 1.f;  // per tensor (per-token scales: 1, applied per key)
  if constexpr (KV == KV_E4M3) {
    if (!tok) {
      k_scale = __ldg(p.kv_scale);
      v_scale = __ldg(p.kv_scale + 1);
    }
  }
  const float scale = p.scale * k_scale;

  // The accumulator rows of this lane: 2cq and 2cq + 1 (N columns of the S^T / O^T tiles),
  // rows r of kv-head g + c / RH.
  bool rv[2];
  int rh[2], ri[2], rpos[2], rlo[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int c = 2 * cq + e, r = c % RH;
    rv[e] = r < nr && q0 + r / G < p.total_q;  // never index past the q / out tensors
    const int i = rv[e] ? r / G : 0;
    ri[e] = i;
    rh[e] = (g + c / RH) * G + (rv[e] ? r % G : 0);
    rpos[e] = ctx + i;
    rlo[e] = p.window_left >= 0 ? max(0, rpos[e] - p.window_left) : 0;
  }
  // Bounds over the q-block's rows (every lane sees all of them), to skip fully masked
  // 16-key chunks and to mask only boundary chunks.
  const int pmin = ctx, pmax = pos_last;
  const int lomin = p.window_left >= 0 ? max(0, pmin - p.window_left) : 0;
  const int lomax = p.window_left >= 0 ? max(0, pmax - p.window_left) : 0;

  // Q^T fragments (B operand, 16 d x 8 rows): column gq of the tile is row gq of the
  // q-block; lane cq holds d 2cq, 2cq + 1 (register 0) and 2cq + 8, 2cq + 9 (register 1)
  // of each 16-d slice, in the MMA input type (16-bit caches).
  //
  // fp8 caches: the QK product runs on the e4m3 tensor-core MMA straight from the cached
  // codes, so Q^T becomes e4m3 too, without losing precision: row gq is scaled by a power
  // of two 2^c that puts its largest magnitude in [128, 256), and written as the sum of QT
  // e4m3 terms (a 16-bit value's significand is the sum of its first two (bf16: 8 bits) or
  // three (f16: 11 bits) 4-bit pieces, each a normal e4m3 value in that range; pieces below
  // e4m3's smallest subnormal, 2^-9, are lost: under 2^-17 of the row's largest value).
  // Lane cq holds d = cq D/4 + 8t + {0..3} (b0) and + {4..7} (b1) of k-step t, the bytes of
  // the K rows it reads; the score then takes the factor 2^-c back.
  constexpr int kQT = C::kPermD ? QT : 1;
  uint32_t qt[C::kPermD ? 1 : D / 16][2];
  uint32_t q8[kQT][C::kPermD ? D / 32 : 1][2];
  float row_scale[2] = {1.f, 1.f};  // 2^-c of rows 2cq and 2cq + 1 (fp8)
  {
    const int rq = gq % RH;  // column gq: row rq of kv-head g + gq / RH
    const bool qv = rq < nr && q0 + rq / G < p.total_q;
    const uint16_t* qrow = static_cast<const uint16_t*>(p.q) +
                           (static_cast<size_t>(q0 + (qv ? rq / G : 0)) * p.hq +
                            (g + gq / RH) * G + (qv ? rq % G : 0)) *
                               D;
    if constexpr (!C::kPermD) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int col = kk * 16 + 2 * cq + 8 * h;
          qt[kk][h] = qv ? __ldg(reinterpret_cast<const unsigned int*>(qrow + col)) : 0u;
        }
      }
    } else {
      constexpr int kN = D / 4;  // values of row gq this lane holds
      float x[kN];
#pragma unroll
      for (int i = 0; i < kN; i += 8) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (qv) w = __ldg(reinterpret_cast<const uint4*>(qrow + cq * kN + i));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (p.q_dtype == UA_DT_BF16) {
            x[i + 2 * k] = bf16_lo(ww[k]);
            x[i + 2 * k + 1] = bf16_hi(ww[k]);
          } else {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[k]));
            x[i + 2 * k] = f.x;
            x[i + 2 * k + 1] = f.y;
          }
        }
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < kN; ++i) amax = fmaxf(amax, fabsf(x[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      // amax in [2^(E-127), 2^(E-126)) with E its biased exponent: c = 134 - E puts it in
      // [128, 256); c stays inside the normal range of fp32 powers of two
      const int ebits = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
      const int c = min(126, max(-126, 134 - ebits));
      const float up = __uint_as_float(static_cast<uint32_t>(127 + c) << 23);
      const float down = __uint_as_float(static_cast<uint32_t>(127 - c) << 23);
#pragma unroll
      for (int i = 0; i < kN; ++i) x[i] *= up;
#pragma unroll
      for (int term = 0; term < kQT; ++term) {
#pragma unroll
        for (int t = 0; t < D / 32; ++t) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int d0 = 8 * t + 4 * h;
            const uint32_t c01 = f32x2_to_e4m3x2(x[d0], x[d0 + 1]);
            const uint32_t c23 = f32x2_to_e4m3x2(x[d0 + 2], x[d0 + 3]);
            q8[term][t][h] = c01 | (c23 << 16);
            uint32_t f01, f23;  // the terms' exact values back, for the next residual
            e4m3x4_to_f16x4(q8[term][t][h], f01, f23);
            const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&f01));
            const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&f23));
            x[d0] -= v01.x;
            x[d0 + 1] -= v01.y;
            x[d0 + 2] -= v23.x;
            x[d0 + 3] -= v23.y;
          }
        }
      }
      // rows 2cq and 2cq + 1 of the accumulator are rows gq = 2cq, 2cq + 1 of lanes 8cq, 8cq + 4
      row_scale[0] = __shfl_sync(0xffffffffu, down, 8 * cq);
      row_scale[1] = __shfl_sync(0xffffffffu, down, 8 * cq + 4);
    }
  }

  // score scale of rows 2cq and 2cq + 1 (with the fp8 rows' 2^-c), and in log2 units
  const float srow[2] = {scale * row_scale[0], scale * row_scale[1]};
  const float srow2[2] = {srow[0] * kLog2e, srow[1] * kLog2e};

  float slope[2] = {0.f, 0.f};
  if constexpr (FEAT) {
    if (p.alibi != nullptr) {
      slope[0] = rv[0] ? __ldg(p.alibi + rh[0]) : 0.f;
      slope[1] = rv[1] ? __ldg(p.alibi + rh[1]) : 0.f;
    }
  }
  const float inv_softcap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;

  // Online-softmax state (base 2) of rows 2cq, 2cq + 1.  l_run sums this lane's keys
  // (row gq of the S^T tile and gq + 8); the lanes of a row add up at the end.  The sink
  // is the initial running max of partition 0 and adds e^{sink - m} once to the row sum
  // (counted by the gq == 0 lane of warp 0).
  const int kgp = warp;
  float m_run[2], l_run[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const bool sink = p.sinks != nullptr && z == 0 && kgp == 0 && rv[e];
    m_run[e] = sink ? __ldg(p.sinks + rh[e]) * kLog2e : -INFINITY;
    l_run[e] = (sink && gq == 0) ? 1.f : 0.f;
  }
  float ot[C::kMT][4];
#pragma unroll
  for (int m = 0; m < C::kMT; ++m)
#pragma unroll
    for (int e = 0; e < 4; ++e) ot[m][e] = 0.f;

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
    const int ch = kgp;  // this warp's 16 keys of the 64-key stage
    const int kc0 = ks + t * T + 16 * ch;
    if (kc0 < ke && kc0 <= pmax && kc0 + 16 > lomin) {
      // ---- S^T = K Q^T for 16 keys: element e of the accumulator is key kc0 + gq + 8(e>>1),
      // row 2cq + (e & 1)
      float st[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (C::kPermD) {
        // Lane (gq, cq) reads bytes [cq D/4, (cq + 1) D/4) of K rows gq and gq + 8: words
        // 2tt and 2tt + 1 of its 16-byte chunk u are the A registers (rows gq | gq + 8) of
        // k-step t = 2u + tt.  One accumulator per Q term keeps the MMA chains short.
        float sx[kQT][4];
#pragma unroll
        for (int term = 0; term < kQT; ++term)
#pragma unroll
          for (int e = 0; e < 4; ++e) sx[term][e] = 0.f;
        if constexpr (HP == 1) {
#pragma unroll
          for (int u = 0; u < D / 64; ++u) {
            const uint4 k0 = *reinterpret_cast<const uint4*>(
                kst + C::raw_byte(16 * ch + gq, cq * (D / 4) + 16 * u));
            const uint4 k8 = *reinterpret_cast<const uint4*>(
                kst + C::raw_byte(16 * ch + gq + 8, cq * (D / 4) + 16 * u));
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
              const uint32_t a[4] = {tt ? k0.z : k0.x, tt ? k8.z : k8.x, tt ? k0.w : k0.y,
                                     tt ? k8.w : k8.y};
#pragma unroll
              for (int term = 0; term < kQT; ++term)
                mma_16832_e4m3(sx[term], a, q8[term][2 * u + tt][0], q8[term][2 * u + tt][1]);
            }
          }
        } else {
          // Two kv-heads: k-step j of chunk u pairs word j of head g's rows (k 0..15 of the
          // MMA) with word j of head g + 1's rows (k 16..31).  The B operand is block
          // diagonal: a lane's Q word (its column's head) goes to b0 for a column of head g
          // and to b1 for head g + 1, the other half zero, so each column sums over its own
          // head's keys only.
          const uint32_t bm0 = gq < RH ? 0xffffffffu : 0u, bm1 = ~bm0;
#pragma unroll
          for (int u = 0; u < D / 64; ++u) {
            const uint4 x0 = *reinterpret_cast<const uint4*>(
                kst + C::raw_byte(16 * ch + gq, cq * (D / 4) + 16 * u, 0));
            const uint4 x8 = *reinterpret_cast<const uint4*>(
                kst + C::raw_byte(16 * ch + gq + 8, cq * (D / 4) + 16 * u, 0));
            const uint4 y0 = *reinterpret_cast<const uint4*>(
                kst + C::raw_byte(16 * ch + gq, cq * (D / 4) + 16 * u, 1));
            const uint4 y8 = *reinterpret_cast<const uint4*>(
                kst + C::raw_byte(16 * ch + gq + 8, cq * (D / 4) + 16 * u, 1));
            const uint32_t w0[4] = {x0.x, x0.y, x0.z, x0.w}, w8[4] = {x8.x, x8.y, x8.z, x8.w};
            const uint32_t v0[4] = {y0.x, y0.y, y0.z, y0.w}, v8[4] = {y8.x, y8.y, y8.z, y8.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t a[4] = {w0[j], w8[j], v0[j], v8[j]};
#pragma unroll
              for (int term = 0; term < kQT; ++term) {
                const uint32_t qw = q8[term][2 * u + j / 2][j & 1];
                mma_16832_e4m3(sx[term], a, qw & bm0, qw & bm1);
              }
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          st[e] = sx[0][e];
#pragma unroll
          for (int term = 1; term < kQT; ++term) st[e] += sx[term][e];
        }
      } else {
        // A fragments of the swizzled K rows: matrices (keys 0-7 | 8-15) x (d 0-7 | 8-15)
        const uint32_t kbase = smem_addr(kst);
        const uint32_t kr = 16 * ch + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t c = (kk & 3) * 2 + (lane >> 4);  // 16-byte chunk in the column block
          uint32_t a[4];
          ldsm_x4(kbase + (kk >> 2) * C::kCBBytes + sw128(kr, c), a[0], a[1], a[2], a[3]);
          mma_16816<kF16Mma>(st, a, qt[kk][0], qt[kk][1]);
        }
      }

      if constexpr (KV == KV_E4M3) {
        if (tok) {  // keys gq and gq + 8: their own K scales
          const float s0 = sks[s * T + 16 * ch + gq], s8 = sks[s * T + 16 * ch + gq + 8];
          st[0] *= s0;
          st[1] *= s0;
          st[2] *= s8;
          st[3] *= s8;
        }
      }

      // ---- score transform and mask (log2 domain)
      const bool need_mask = kc0 < lomax || kc0 + 15 > pmin || kc0 + 16 > ke;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rr = e & 1;
        const int j = kc0 + gq + 8 * (e >> 1);
        float x;
        if constexpr (FEAT) {
          x = st[e] * srow[rr];
          if (p.softcap > 0.f) x = p.softcap * fast_tanh(x * inv_softcap);
          x += slope[rr] * static_cast<float>(j - ctx);
          if (p.qq_bias != nullptr && rv[rr] && j >= ctx && j <= rpos[rr] &&
              ri[rr] < p.max_seqlen_q)
            x += __ldg(p.qq_bias + static_cast<size_t>(ri[rr]) * p.qq_stride + (j - ctx));
          x *= kLog2e;
        } else {
          x = st[e] * srow2[rr];
        }
        if (need_mask) {
          const bool ok = rv[rr] && j >= rlo[rr] && j <= rpos[rr] && j < ke;
          x = ok ? x : -INFINITY;
        }
        st[e] = x;
      }

      // ---- online softmax: row 2cq + e's 16 scores sit in lanes cq, cq + 4, ..., cq + 28
      // (registers e and e + 2).  A row's running max moves only when a score passes it
      // by more than 8 (log2 units), so P stays below 2^8 and the accumulators are
      // rescaled only on those chunks.
      float alpha[2];
      bool grow_any = false;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = fmaxf(st[e], st[e + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const bool grow = mx > m_run[e] + 8.f;  // from -inf: the first finite score
        alpha[e] = grow ? fast_exp2(m_run[e] - mx) : 1.f;
        if (grow) m_run[e] = mx;
        grow_any |= grow;
        const float m_use = (m_run[e] == -INFINITY) ? 0.f : m_run[e];
        st[e] = fast_exp2(st[e] - m_use);
        st[e + 2] = fast_exp2(st[e + 2] - m_use);
        l_run[e] = l_run[e] * alpha[e] + (st[e] + st[e + 2]);
      }
      if (__any_sync(0xffffffffu, grow_any)) {
#pragma unroll
        for (int m = 0; m < C::kMT; ++m) {
          ot[m][0] *= alpha[0];
          ot[m][1] *= alpha[1];
          ot[m][2] *= alpha[0];
          ot[m][3] *= alpha[1];
        }
      }

      // ---- P^T as the B operand: the S^T accumulator halves (keys gq and gq + 8, rows
      // 2cq, 2cq + 1) transposed in registers give keys 2cq, 2cq + 1 (register 0) and
      // 2cq + 8, 2cq + 9 (register 1) of row gq.
      uint32_t pb[2], pbl[2];
      if constexpr (kF16Mma) {
        if constexpr (KV == KV_E4M3) {
          if (tok) {  // P of keys gq and gq + 8 times their V scales (the row sum took P)
            const float s0 = svs[s * T + 16 * ch + gq], s8 = svs[s * T + 16 * ch + gq + 8];
            st[0] *= s0;
            st[1] *= s0;
            st[2] *= s8;
            st[3] *= s8;
          }
        }
        pb[0] = movmatrix_trans(pack_f16(st[0], st[1]));
        pb[1] = movmatrix_trans(pack_f16(st[2], st[3]));
      } else {
        // bf16 P carries 8 significant bits; a second bf16 term holds the remainder so
        // P V keeps ~16 bits (P = hi + lo).
        const uint32_t h0 = pack_bf16(st[0], st[1]), h1 = pack_bf16(st[2], st[3]);
        pb[0] = movmatrix_trans(h0);
        pb[1] = movmatrix_trans(h1);
        pbl[0] = movmatrix_trans(pack_bf16(st[0] - bf16_lo(h0), st[1] - bf16_hi(h0)));
        pbl[1] = movmatrix_trans(pack_bf16(st[2] - bf16_lo(h1), st[3] - bf16_hi(h1)));
      }

      // ---- O^T += V^T P^T: A registers 0/1 hold keys 2cq, 2cq + 1 and 2/3 keys 2cq + 8,
      // 2cq + 9 of the chunk
      const int k0 = kc0 + 2 * cq;
      const bool tail = kc0 + 16 > kv_len;
      const uint32_t m01 = (k0 < kv_len ? 0xffffu : 0u) | (k0 + 1 < kv_len ? 0xffff0000u : 0u);
      const uint32_t m89 = (k0 + 8 < kv_len ? 0xffffu : 0u) | (k0 + 9 < kv_len ? 0xffff0000u : 0u);
      if constexpr (C::kPermD) {
        // Lane (gq, cq) reads bytes [gq D/8, (gq + 1) D/8) of V rows 2cq, 2cq+1, 2cq+8,
        // 2cq+9; bytes 2m and 2m + 1 of that run are fragment rows gq and gq + 8 of
        // m-tile m (output columns gq D/8 + 2m and + 1).  A byte permute pairs the two
        // keys of each operand half.  Two kv-heads: one pass per head, with P^T's columns
        // of the other head zeroed, so both heads accumulate into their own columns of O^T.
        constexpr int kW = D / 32;  // 32-bit words of a row per lane
#pragma unroll
        for (int hh = 0; hh < HP; ++hh) {
          const uint32_t bm = HP == 1 || (gq / RH) == hh ? 0xffffffffu : 0u;
          const uint32_t pv0 = pb[0] & bm, pv1 = pb[1] & bm;
          uint32_t vw[4][kW];
#pragma unroll
          for (int r4 = 0; r4 < 4; ++r4) {
            const uint32_t trow = 16 * ch + 2 * cq + (r4 & 1) + 8 * (r4 >> 1);
            if constexpr (kW % 4 == 0) {
#pragma unroll
              for (int x = 0; x < kW; x += 4) {
                const uint4 v4 = *reinterpret_cast<const uint4*>(
                    vst + C::raw_byte(trow, gq * (D / 8) + 4 * x, hh));
                vw[r4][x] = v4.x;
                vw[r4][x + 1] = v4.y;
                vw[r4][x + 2] = v4.z;
                vw[r4][x + 3] = v4.w;
              }
            } else {
              const uint2 v2 =
                  *reinterpret_cast<const uint2*>(vst + C::raw_byte(trow, gq * (D / 8), hh));
              vw[r4][0] = v2.x;
              vw[r4][1] = v2.y;
            }
          }
#pragma unroll
          for (int x = 0; x < kW; ++x) {
            // bytes 4x, 4x + 1 (m-tile 2x) then 4x + 2, 4x + 3 (m-tile 2x + 1) of the rows
            const uint32_t lo0 = __byte_perm(vw[0][x], vw[1][x], 0x5140);
            const uint32_t hi0 = __byte_perm(vw[0][x], vw[1][x], 0x7362);
            const uint32_t lo8 = __byte_perm(vw[2][x], vw[3][x], 0x5140);
            const uint32_t hi8 = __byte_perm(vw[2][x], vw[3][x], 0x7362);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t w0 = h ? hi0 : lo0, w8 = h ? hi8 : lo8;
              uint32_t a[4];
              e4m3x4_to_f16x4(w0, a[0], a[1]);
              e4m3x4_to_f16x4(w8, a[2], a[3]);
              if (tail) {
                a[0] &= m01;
                a[1] &= m01;
                a[2] &= m89;
                a[3] &= m89;
              }
              mma_16816<true>(ot[2 * x + h], a, pv0, pv1);
            }
          }
        }
      } else {
        // A fragments of V^T from the swizzled V rows (transposing loads): matrices
        // (d 0-7 | 8-15 of the m-tile) x (keys 0-7 | 8-15)
        const uint32_t vbase = smem_addr(vst);
        const uint32_t vr = 16 * ch + (lane & 7) + ((lane >> 4) << 3);
        const uint32_t dh = (lane >> 3) & 1;
#pragma unroll
        for (int m = 0; m < C::kMT; ++m) {
          const uint32_t dc = 2 * m + dh;  // 16-byte chunk of the row
          uint32_t a[4];
          ldsm_x4_trans(vbase + (dc >> 3) * C::kCBBytes + sw128(vr, dc & 7), a[0], a[1], a[2],
                        a[3]);
          if (tail) {
            a[0] &= m01;
            a[1] &= m01;
            a[2] &= m89;
            a[3] &= m89;
          }
          mma_16816<kF16Mma>(ot[m], a, pb[0], pb[1]);
          if constexpr (!kF16Mma) mma_16816<kF16Mma>(ot[m], a, pbl[0], pbl[1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // Row sums: add up the lanes of a row (gq = 0..7).
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 4);
    l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 8);
    l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 16);
  }

  if (aborted) s_abort = 1;
  named_bar_sync(1, 32 * C::kConsumerWarps);
  // Split partitions of one cluster merge through distributed shared memory (every CTA
  // reaches both cluster barriers, an aborted one too); otherwise an aborted CTA writes
  // nothing.
  if (s_abort && !cmerge) return;
  const bool ok = s_abort == 0;

  // ---- the warps' states of the same rows: rescale to the rows' max (exchanged through
  // shared memory), then every warp leaves its O^T fragments there and warp w adds up
  // m-tiles w, w + W, ... of all warps (read in the MMA fragment layout) into the CTA's
  // partial rows.
  constexpr int W4 = C::kConsumerWarps;
  float* const sm_m = reinterpret_cast<float*>(pipe);                   // [W][8]
  float* const sm_l = sm_m + W4 * NR;                                   // [W][8]
  float4* const sm_o = reinterpret_cast<float4*>(sm_l + W4 * NR);       // [W][kMT][32]
  float* const partial = reinterpret_cast<float*>(pipe + C::kMergeBytes);  // [8][D], m[8], l[8]
  if (gq == 0) {
    sm_m[warp * NR + 2 * cq] = m_run[0];
    sm_m[warp * NR + 2 * cq + 1] = m_run[1];
  }
  named_bar_sync(1, 32 * W4);
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W4; ++w) M = fmaxf(M, sm_m[w * NR + 2 * cq + e]);
    const float wt = M == -INFINITY ? 0.f : fast_exp2(m_run[e] - M);
    m_run[e] = M;
    l_run[e] *= wt;
#pragma unroll
    for (int m = 0; m < C::kMT; ++m) {
      ot[m][e] *= wt;
      ot[m][e + 2] *= wt;
    }
  }
  if (gq == 0) {
    sm_l[warp * NR + 2 * cq] = l_run[0];
    sm_l[warp * NR + 2 * cq + 1] = l_run[1];
  }
#pragma unroll
  for (int m = 0; m < C::kMT; ++m)
    sm_o[(warp * C::kMT + m) * 32 + lane] = make_float4(ot[m][0], ot[m][1], ot[m][2], ot[m][3]);
  named_bar_sync(1, 32 * W4);
  // partial rows (v_scale applied): O^T element (m-tile m, fragment row gq + 8h, column
  // 2cq + e) is output column out_col(m, gq + 8h) of row 2cq + e
  for (int m = warp; m < C::kMT; m += W4) {
    float4 o4 = sm_o[m * 32 + lane];
#pragma unroll
    for (int w = 1; w < W4; ++w) {
      const float4 x = sm_o[(w * C::kMT + m) * 32 + lane];
      o4.x += x.x;
      o4.y += x.y;
      o4.z += x.z;
      o4.w += x.w;
    }
    const float o[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
    for (int e4 = 0; e4 < 4; ++e4)
      partial[(2 * cq + (e4 & 1)) * D + C::out_col(m, gq + 8 * (e4 >> 1))] = o[e4] * v_scale;
  }
  if (warp == 0 && gq == 0) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < W4; ++w) L += sm_l[w * NR + 2 * cq + e];
      partial[NR * D + 2 * cq + e] = m_run[e];
      partial[NR * D + NR + 2 * cq + e] = L;
    }
  }
  named_bar_sync(1, 32 * W4);

  const size_t n_part = static_cast<size_t>(p.n_part);
  const size_t esz = p.out_dtype == UA_DT_F32 ? 4 : 2;
  // q-block column c holds row c mod RH of kv-head g + c / RH: a row when that is below
  // nr and its token lies inside the batch
  auto col_valid = [&](int c) -> bool {
    const int r = c % RH;
    return r < nr && q0 + r / G < p.total_q;
  };
  auto out_row = [&](int c) -> size_t {
    const int r = c % RH;
    return static_cast<size_t>(q0 + r / G) * p.hq + (g + c / RH) * G + r % G;
  };
  const int ncols = HP == 1 ? nr : NR;  // columns up to the last that may hold a row
  if (n_part == 1 || !cmerge) {
    if (!ok) return;
    // one partition: normalised rows; several: the partition's max / sum / output rows
    // in the global scratch for the merge kernel
    for (int idx = threadIdx.x; idx < ncols * D; idx += 32 * C::kConsumerWarps) {
      const int r = idx / D, c = idx % D;
      if (!col_valid(r)) continue;
      const size_t row = out_row(r);
      const float v = partial[r * D + c];
      if (n_part == 1) {
        const float l = partial[NR * D + NR + r];
        const float x = l > 0.f ? v / l : 0.f;
        if (p.out_dtype == UA_DT_F32) static_cast<float*>(p.out)[row * D + c] = x;
        else if (p.out_dtype == UA_DT_BF16)
          static_cast<__nv_bfloat16*>(p.out)[row * D + c] = __float2bfloat16_rn(x);
        else static_cast<__half*>(p.out)[row * D + c] = __float2half_rn(x);
      } else {
        const size_t w = row * n_part + z;
        p.ws_acc[w * D + c] = v;
        if (c == 0) {
          p.ws_m[w] = partial[NR * D + r];
          p.ws_l[w] = partial[NR * D + NR + r];
        }
      }
    }
    return;
  }

  // Cluster merge: the cluster is the n_part partitions (grid z) of cluster_y CTAs (kv-heads,
  // or pairs of them) of this slot; partition zz of this CTA's heads is the cluster's CTA
  // cluster_ctaid.y + cluster_y * zz.  Column r is merged by partition r mod n_part, one
  // warp a row.
  cluster_sync();
  {
    const int np = p.n_part;
    const uint32_t cy = cluster_nctaid_y(), yc = cluster_ctaid_y();
    const uint32_t part_s = smem_addr(partial);
    for (int k = warp;; k += C::kConsumerWarps) {
      const int r = z + np * k;
      if (r >= ncols) break;
      if (!col_valid(r)) continue;
      cluster_merge_row<D>(part_s + (NR * D + r) * 4, part_s + (NR * D + NR + r) * 4,
                           part_s + r * D * 4, np, yc, cy, lane,
                           static_cast<uint8_t*>(p.out) + out_row(r) * D * esz, p.out_dtype);
    }
  }
  // no CTA leaves while the cluster still reads its shared memory (those reads have
  // returned: a relaxed arrival, which need not wait for the output stores)
  cluster_sync_relaxed();
}

template <int D, int KV, bool FEAT, int QT, int W, int HP = 1>
cudaError_t launch_decode_t(const TileParams& tp, dim3 grid, int cluster_y, int cluster_z,
                            cudaStream_t stream) {
  using C = DecCfg<D, KV, W, HP>;
  auto kern = ua_decode_kernel<D, KV, FEAT, QT, W, HP>;
  static std::atomic<unsigned long long> configured{0};  // one bit per device
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
    configured.fetch_or(bit);
  }
  return launch_pdl_cluster(kern, grid, dim3(C::kThreads), C::kSmemBytes, stream, cluster_y,
                            cluster_z, tp);
}

template <int D, int W>
cudaError_t launch_decode_width(const TileParams& tp, dim3 grid, int kv, bool feat,
                                int cluster_y, int cluster_z, cudaStream_t s) {
#define UA_DEC_CASE(KVV, QT)                                                                 \
  return feat ? launch_decode_t<D, KVV, true, QT, W>(tp, grid, cluster_y, cluster_z, s)      \
              : launch_decode_t<D, KVV, false, QT, W>(tp, grid, cluster_y, cluster_z, s);
  if (kv == KV_F16) UA_DEC_CASE(KV_F16, 1)
  if (kv == KV_BF16) UA_DEC_CASE(KV_BF16, 1)
  if (kv == KV_E4M3) {
    if (tp.p.q_dtype == UA_DT_BF16) UA_DEC_CASE(KV_E4M3, 2)
    UA_DEC_CASE(KV_E4M3, 3)
  }
#undef UA_DEC_CASE
  return cudaErrorInvalidValue;
}

// Two kv-heads a CTA (fp8 caches, four consumer warps; tensor maps over the head-outer
// view with boxes of two heads).
template <int D>
cudaError_t launch_decode_pair(const TileParams& tp, dim3 grid, bool feat, int cluster_y,
                               int cluster_z, cudaStream_t s) {
  if (tp.p.q_dtype == UA_DT_BF16)
    return feat ? launch_decode_t<D, KV_E4M3, true, 2, 4, 2>(tp, grid, cluster_y, cluster_z, s)
                : launch_decode_t<D, KV_E4M3, false, 2, 4, 2>(tp, grid, cluster_y, cluster_z, s);
  return feat ? launch_decode_t<D, KV_E4M3, true, 3, 4, 2>(tp, grid, cluster_y, cluster_z, s)
              : launch_decode_t<D, KV_E4M3, false, 3, 4, 2>(tp, grid, cluster_y, cluster_z, s);
}

// Clusters of cluster_y x cluster_z CTAs of the decode kernel that can be resident at
// once (the hardware places a cluster's CTAs within one GPU processing cluster, so fewer
// CTAs than the SMs' slots may run together); -1 when the query fails.
template <int D, int KV, int W, int HP = 1>
int decode_cluster_capacity_t(int cluster_y, int cluster_z) {
  using C = DecCfg<D, KV, W, HP>;
  auto kern = ua_decode_kernel<D, KV, false, KV == KV_E4M3 ? 2 : 1, W, HP>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, static_cast<unsigned>(cluster_y), static_cast<unsigned>(cluster_z));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(cluster_y);
  attr[0].val.clusterDim.z = static_cast<unsigned>(cluster_z);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return -1;
  return n;
}

template <int D, int W>
int decode_cluster_capacity_d(int kv, int cluster_y, int cluster_z) {
  return kv == KV_E4M3 ? decode_cluster_capacity_t<D, KV_E4M3, W>(cluster_y, cluster_z)
                       : decode_cluster_capacity_t<D, KV_BF16, W>(cluster_y, cluster_z);
}

template <int D>
int decode_ctas_per_sm_d(int kv) {
  if (kv == KV_E4M3) return DecCfg<D, KV_E4M3>::kMinBlocks;
  return DecCfg<D, KV_BF16>::kMinBlocks;
}

}  // namespace ua
