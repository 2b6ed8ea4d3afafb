// ua_prefill_tm.cuh -- the tensor-memory attention kernel of libua.so for prefill-shaped
// q-blocks with head_dim <= 128 (included by ua_prefill_d64.cu and ua_prefill_d128.cu).
//
// One CTA owns (q-block, kv-head g, key partition z).  A q-block is NQ (1 or 2) q tiles of
// 128 rows; a tile is TQ = floor(128 / G) consecutive query tokens times the G query heads
// that read kv-head g, so the GQA heads of a group share every K/V tile (vllm-rdna PR #34
// "FA-RDNA2 D=128 prefill", "Change" 1, on tensor cores), and the NQ tiles share them too.
// Per key tile of BN = 128 keys and q tile t:
//
//   S_t = Q_t K^T   tcgen05.mma (kind::f16, M=128, N=128, fp32) into tensor memory
//   softmax         one thread per row: pass 1 reads the S row from tensor memory for the
//                   row max (applying scale, softcap, ALiBi, QQ-bias and the causal/window
//                   mask where a tile needs them, and writing those scores back); pass 2
//                   reads it again and writes P = 2^(s - m) back over S as bf16 high part
//                   + remainder (or f16), 32 keys at a time
//   O_t += P_t V    tcgen05.mma with A = P read from tensor memory and V from shared memory
//
// Tensor memory per q tile: S/P (128 columns) and O (D columns); two tiles fill the 512
// columns at D = 128.  Because P overwrites S, a tile's next S is issued after its P.V;
// the MMA warp alternates the tiles (P.V then S of tile 0, P.V then S of tile 1) so the
// tensor cores work on one tile while the other tile's softmax runs.  Each commit tracks
// every earlier MMA of the issuing thread, so "S of step n is ready" also means "O holds
// P.V of step n-1": the softmax rescales O (only when a row's max grows by more than 2^8)
// right after that wait, with no extra barrier.
//
// Warp roles (128 * NQ + 96 threads): warps 0..4NQ-1 softmax + epilogue (warp w serves
// tile w / 4, tensor-memory lanes 32 (w % 4) ..; thread = row), warps 4NQ and 4NQ+1 TMA
// producers (Q once and K pages; V pages; pages of 16 keys found through the block table,
// each operand in its own ring, 128-byte swizzled), warp 4NQ+2 MMA issuer and
// tensor-memory owner.
//
// fp8-e4m3 caches (F8, head_dim 64 or 128): the producers copy fp8 K and V tiles into a staging
// buffer, and four more warps (thread = row) turn each into the f16 tile the MMA reads
// (every e4m3 value is an f16; V rows past kv_len become zeros), after converting a bf16
// Q to f16 in place once; the MMAs and the softmax then run the f16 path, with k_scale
// in the score scale and v_scale on the output.
#pragma once

#include <atomic>
#include <climits>
#include <type_traits>

#include <cuda.h>

#include "ua_device.cuh"
#include "ua_internal.h"
#include "ua_prefill.cuh"

#include "ua.h"

namespace ua {

// SW: softmax warps per tensor-memory lane quarter of a q tile (1, or 2 or 4 splitting the
// key columns of S and the columns of O between them).
template <int D, int NQ, bool F8 = false, int SW = 1>
struct PrefillTmCfg {
  static constexpr int kBM = 128;                        // MMA rows of one q tile
  static constexpr int kBN = 128;                        // keys per tile
  static constexpr int kCB = D / 64;                     // 128-byte column blocks of a row
  static constexpr int kQBytes = kCB * kBM * 128;        // one q tile
  static constexpr int kKVCB = kBN * 128;                // one column block of a K or V tile
  static constexpr int kTileBytes = kCB * kKVCB;         // one K (or V) tile
  static constexpr int kBarBytes = 512;
  // fp8 caches: one staging tile of fp8 codes per operand (128 keys x D bytes)
  static constexpr int kF8Tile = kBN * D;
  static constexpr int kF8Bytes = F8 ? 2 * kF8Tile : 0;
  static constexpr int kDeqWarps = F8 ? 4 : 0;
  // SW > 1: each tile's row maxima of the SW warps of a row, exchanged through shared
  // memory as bf16 values rounded up
  static constexpr int kXchBytes = SW > 1 ? NQ * SW * 2 * 128 * 2 : 0;  // two tiles in flight
  // K and V ring depths: as many tiles as fit beside Q (K gets the odd one, at most 4 each)
  static constexpr int kSlots =
      (227 * 1024 - 1024 - kBarBytes - NQ * kQBytes - kF8Bytes - kXchBytes) / kTileBytes;
  static constexpr int kRingK = (kSlots + 1) / 2 > 4 ? 4 : (kSlots + 1) / 2;
  static constexpr int kRingV = kSlots / 2 > 4 ? 4 : kSlots / 2;
  static constexpr int kSmemBytes =
      1024 + NQ * kQBytes + (kRingK + kRingV) * kTileBytes + kF8Bytes + kBarBytes + kXchBytes;
  static constexpr int kTmemStride = kBN + D;            // S/P, then O, of one q tile
  static constexpr int kTmemCols = 512;
  static constexpr int kSoftmaxWarps = 4 * NQ * SW;
  static_assert(SW == 1 || SW == 2 || (SW == 4 && D == 128),
                "one, two or (head_dim 128) four softmax warps per lane quarter");
  static constexpr int kThreads = 32 * kSoftmaxWarps + 96 + 32 * kDeqWarps;
  static_assert(D <= 128, "two 128-key K/V rings must fit");
  static_assert(NQ * kTmemStride <= kTmemCols, "tensor memory budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kRingK >= 2 && kRingV >= 2, "at least double-buffered K and V");
  static_assert(!F8 || D == 64 || D == 128, "fp8 caches: head_dim 64 or 128");
};

template <int D, int NQ, bool BF16, bool FEAT, bool F8 = false, int SW = 1>
__global__ void __launch_bounds__(PrefillTmCfg<D, NQ, F8, SW>::kThreads, 1)
    ua_prefill_tm_kernel(const __grid_constant__ PrefillParams pp) {
  using C = PrefillTmCfg<D, NQ, F8, SW>;
  constexpr int BN = C::kBN;
  constexpr int RK = C::kRingK, RV = C::kRingV;
  constexpr int kProducerK = C::kSoftmaxWarps, kProducerV = C::kSoftmaxWarps + 1;
  constexpr int kMma = C::kSoftmaxWarps + 2;
  constexpr int kDeq0 = C::kSoftmaxWarps + 3;  // fp8: dequant warps kDeq0 .. kDeq0 + 3
  const AttnParams& p = pp.p;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* const smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* const sQ = smem;                          // NQ q tiles
  uint8_t* const sK = sQ + NQ * C::kQBytes;          // RK K tiles
  uint8_t* const sV = sK + RK * C::kTileBytes;       // RV V tiles
  uint8_t* const sK8 = sV + RV * C::kTileBytes;      // fp8: staging K tile of codes
  uint8_t* const sV8 = sK8 + (F8 ? C::kF8Tile : 0);  // fp8: staging V tile of codes
  uint64_t* const bars = reinterpret_cast<uint64_t*>(sK8 + C::kF8Bytes);
  uint64_t* const q_full = bars + 0;
  uint64_t* const fin = bars + 1;
  uint64_t* const k_full = bars + 2;                 // [RK]
  uint64_t* const k_empty = k_full + RK;             // [RK]
  uint64_t* const v_full = k_empty + RK;             // [RV]
  uint64_t* const v_empty = v_full + RV;             // [RV]
  // fp8: Q converted, staging K / V full (copies) and empty (dequant warps)
  uint64_t* const q_ready = v_empty + RV;
  uint64_t* const k8_full = q_ready + 1;
  uint64_t* const k8_empty = q_ready + 2;
  uint64_t* const v8_full = q_ready + 3;
  uint64_t* const v8_empty = q_ready + 4;
  // [NQ][3]: s_full, p_full, pv_done; then (one q tile: S double-buffered) s_full and
  // p_full of the second S buffer
  uint64_t* const tile_bars = v_empty + RV + (F8 ? 5 : 0);
  auto s_full = [&](int qt) { return tile_bars + 3 * qt; };
  auto p_full = [&](int qt) { return tile_bars + 3 * qt + 1; };
  auto pv_done = [&](int qt) { return tile_bars + 3 * qt + 2; };
  auto s_full_b = [&](int buf) { return buf ? tile_bars + 3 * NQ : s_full(0); };
  auto p_full_b = [&](int buf) { return buf ? tile_bars + 3 * NQ + 1 : p_full(0); };
  uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(tile_bars + 3 * NQ + 2);
  // [NQ][2]: walk step + 1 of the tile's P when its low part matters
  int* const lo_flag = reinterpret_cast<int*>(tmem_holder + 1);
  // SW > 1: per (q tile, lane quarter) a barrier for the tile's row-max exchange and one for
  // the final row-sum exchange ([NQ][4][2]), and the exchanged maxima
  uint64_t* const xch_bars = reinterpret_cast<uint64_t*>(lo_flag + 2 * NQ + 1);  // 8-byte aligned
  uint16_t* const xch = reinterpret_cast<uint16_t*>(bars) + C::kBarBytes / 2;  // [NQ][2][SW][128]
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int z = blockIdx.z;
  const int G = p.group;
  const int TQ = pp.tq;          // tokens of one q tile
  const int TB = NQ * TQ;        // tokens of the CTA's q-block

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(fin, 1);
    // f16 tiles are made by the copies, or (fp8) by the dequant warps
    for (int i = 0; i < RK; ++i) {
      mbar_init(&k_full[i], F8 ? C::kDeqWarps : 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < RV; ++i) {
      mbar_init(&v_full[i], F8 ? C::kDeqWarps : 1);
      mbar_init(&v_empty[i], 1);
    }
    if constexpr (F8) {
      mbar_init(q_ready, C::kDeqWarps);
      mbar_init(k8_full, 1);
      mbar_init(k8_empty, C::kDeqWarps);
      mbar_init(v8_full, 1);
      mbar_init(v8_empty, C::kDeqWarps);
    }
    if constexpr (SW > 1)
      for (int i = 0; i < NQ * 4 * 2; ++i) mbar_init(&xch_bars[i], 32 * SW);
    mbar_init(s_full_b(1), 1);
    mbar_init(p_full_b(1), 4 * SW);
    for (int qt = 0; qt < NQ; ++qt) {
      mbar_init(s_full(qt), 1);
      mbar_init(p_full(qt), 4 * SW);
      mbar_init(pv_done(qt), 1);
      lo_flag[2 * qt] = lo_flag[2 * qt + 1] = 0;
    }
    s_abort = 0;
    mbar_fence_init();
  }
  // Q rows past the tokens of a tile stay zero (they are computed and dropped).
  {
    const int pad = (C::kBM - TQ * G) * 8;  // 16-byte chunks per column block
    for (int i = threadIdx.x; i < NQ * C::kCB * pad; i += C::kThreads) {
      const int qc = i / pad, rem = i % pad;
      *reinterpret_cast<uint4*>(sQ + qc * C::kBM * 128 + (TQ * G + rem / 8) * 128 + (rem % 8) * 16) =
          make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();
  if (warp == kMma) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerK && lane == 0) {
    tma_prefetch_desc(&pp.tmap_q);
    tma_prefetch_desc(&pp.tmap_k);
    tma_prefetch_desc(&pp.tmap_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  volatile int* abort_flag = &s_abort;
  // Everything above touches only this CTA's shared and tensor memory, so it overlaps the
  // previous kernel's tail (programmatic dependent launch); global memory is read below.
  grid_dependency_wait();
  grid_launch_dependents();

  // Longest walks first: slots are taken in reverse order.
  const int x = static_cast<int>(gridDim.x - 1 - blockIdx.x);
  const PfSeq sq = pf_seq_of_slot(p.cu_seqlens_q, p.seq_lens_k, p.num_seqs, x, TB);
  const int b = sq.b, q0 = sq.q0, q_len = sq.q_len, kv_len = sq.kv_len;
  const int t_first = (x - (q0 / TB + b)) * TB;  // first token of the block within the sequence
  if (t_first < 0 || t_first >= q_len) {  // idle slot: uniform for the CTA
    if (warp == kMma) tmem_dealloc(tmem, C::kTmemCols);
    return;
  }
  const int nq_act = min(NQ, (q_len - t_first + TQ - 1) / TQ);  // q tiles holding tokens
  const int ctx = kv_len - q_len;
  // The CTA's key range: the union of its tiles' ranges, split into n_part partitions.
  const int pos_first = ctx + t_first, pos_last = ctx + min(t_first + TB, q_len) - 1;
  const int hi = max(0, min(pos_last + 1, kv_len));
  const int lo = min(hi, p.window_left >= 0 ? max(0, pos_first - p.window_left) : 0) & ~15;
  int part = (hi - lo + p.n_part - 1) / p.n_part;
  part = (part + 15) & ~15;
  const int ks = min(lo + z * part, hi);
  const int ke = min(ks + part, hi);
  const int nt = (ke - ks + BN - 1) / BN;
  // Key tiles [jb, je) of q tile qt: those its own tokens attend to.
  auto tile_walk = [&](int qt, int& jb, int& je) {
    jb = je = 0;
    if (qt >= nq_act) return;
    const int tf = t_first + qt * TQ, tl = min(tf + TQ, q_len) - 1;
    const int a = max(ks, p.window_left >= 0 ? max(0, ctx + tf - p.window_left) : 0);
    const int e = min(ke, max(0, min(ctx + tl + 1, kv_len)));
    if (a < e) {
      jb = (a - ks) / BN;
      je = (e - ks + BN - 1) / BN;
    }
  };


  if (warp == kProducerK || warp == kProducerV) {
    // ======================================================== TMA producers (K, then V)
    // Each warp streams one operand through its own ring, so a K tile never waits behind
    // a V slot.  Block ids are loaded two tiles ahead and only checked when used, so the
    // loop never stalls on a block-table load.
    const bool is_k = warp == kProducerK;
    // fp8: one staging tile of codes per operand instead of the f16 ring
    const int R = F8 ? 1 : (is_k ? RK : RV);
    uint64_t* const full = F8 ? (is_k ? k8_full : v8_full) : (is_k ? k_full : v_full);
    uint64_t* const empty = F8 ? (is_k ? k8_empty : v8_empty) : (is_k ? k_empty : v_empty);
    uint8_t* const ring = F8 ? (is_k ? sK8 : sV8) : (is_k ? sK : sV);
    constexpr int kTileIn = F8 ? C::kF8Tile : C::kTileBytes;  // bytes of one copied tile
    constexpr int kCBIn = F8 ? 1 : C::kCB;                     // its column blocks
    constexpr int kBoxIn = F8 ? 16 * D : 2048;                 // one page box (16 rows)
    const CUtensorMap* const map = is_k ? &pp.tmap_k : &pp.tmap_v;
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    const int bs = p.block_size;
    const int oob = p.num_blocks * bs;
    if (is_k && lane == 0) {
      mbar_arrive_expect_tx(q_full, nq_act * C::kCB * TQ * G * 128);
      for (int qt = 0; qt < nq_act; ++qt)
        for (int cb = 0; cb < C::kCB; ++cb)
          tma_load_3d_pf(sQ + qt * C::kQBytes + cb * C::kBM * 128, &pp.tmap_q, 64 * cb, g * G,
                         q0 + t_first + qt * TQ, q_full);
    }
    // block id of this lane's 16-key page of key tile j (lanes 0 .. BN/16-1; -1: none)
    auto page_blk = [&](int j) -> int {
      const int key = ks + j * BN + 16 * lane;
      const int col = key / bs;
      return (j < nt && lane < BN / 16 && key < ke && col < p.max_blocks_per_seq) ? __ldg(bt + col) : -1;
    };
    // its cache row (the out-of-range row, zero-filled by the copy, where there is no key)
    auto page_row = [&](int j, int blk) -> int {
      const int key = ks + j * BN + 16 * lane;
      if (lane >= BN / 16 || key >= ke) return oob;
      if (static_cast<unsigned>(blk) >= static_cast<unsigned>(p.num_blocks)) {
        atomicOr(p.status, DEV_BAD_BLOCK);
        return oob;
      }
      return blk * bs + key % bs;
    };
    int blk0 = page_blk(0), blk1 = page_blk(1);
    int issued = 0;
    for (int j = 0; j < nt; ++j) {
      const int row = page_row(j, blk0);
      blk0 = blk1;
      blk1 = page_blk(j + 2);
      const int sl = j % R;
      if (j >= R && !pf_wait_warp(&empty[sl], ((j / R) - 1) & 1, abort_flag, p.status)) break;
      if (lane == 0) mbar_arrive_expect_tx(&full[sl], kTileIn);
      __syncwarp();
      if (lane < BN / 16)
#pragma unroll
        for (int cb = 0; cb < kCBIn; ++cb)
          tma_load_3d_pf(ring + sl * kTileIn + cb * C::kKVCB + lane * kBoxIn, map, 64 * cb, g,
                         row, &full[sl]);
      issued = j + 1;
    }
    // never leave copies in flight into this CTA's shared memory (even after an abort)
    for (int j = max(0, issued - R); j < issued; ++j)
      mbar_wait_bounded(&full[j % R], (j / R) & 1, p.status, DEV_TIMEOUT);
    if (is_k && lane == 0) mbar_wait_bounded(q_full, 0, p.status, DEV_TIMEOUT);
  } else if (warp == kMma) {
    // ======================================================== MMA issuer
    static_assert(!F8 || !BF16, "fp8 caches run the f16 MMAs");
    // Step j: for each q tile, O += P V_{j-1} (which frees the tile's S/P columns), then
    // S = Q K_j^T.  Tensor-core operations of one thread run in issue order.  The whole
    // warp runs this loop converged; one elected lane issues each MMA and commit.
    constexpr uint32_t kIdQK = umma_idesc_f16(128, BN, BF16, false);
    constexpr uint32_t kIdPV = umma_idesc_f16(128, D, BF16, true);
    int jb[NQ], je[NQ];
#pragma unroll
    for (int qt = 0; qt < NQ; ++qt) tile_walk(qt, jb[qt], je[qt]);
    bool ok = pf_wait_warp(F8 ? q_ready : q_full, 0, abort_flag, p.status);
    if constexpr (NQ == 1) {
      // One q tile: S double-buffered in tensor memory (columns 0 and BN; O from 2 BN), so
      // the tensor cores compute S_{j+1} while the softmax works on S_j.  Issue order
      // S_0, S_1, then for every j: [P_j ready] P.V_j, S_{j+2}; S_{j+2} overwrites P_j
      // only after P.V_j read it (tensor-core operations of one thread run in order).  One
      // pv_done phase per P.V.
      auto qk = [&](int j) -> bool {
        if (!pf_wait_warp(&k_full[j % RK], (j / RK) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t qb = smem_addr(sQ);
        const uint32_t kb = smem_addr(sK + (j % RK) * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = smem_desc_sw128(qb + (kk >> 2) * C::kBM * 128 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(kb + (kk >> 2) * C::kKVCB + (kk & 3) * 32, 16, 1024);
          umma_f16_ss_warp(tmem + (j & 1) * BN, ad, bd, kIdQK, kk > 0 ? 1u : 0u);
        }
        umma_commit_warp(s_full_b(j & 1));
        umma_commit_warp(&k_empty[j % RK]);
        return true;
      };
      auto pv = [&](int j) -> bool {
        if (!pf_wait_warp(p_full_b(j & 1), (j >> 1) & 1, abort_flag, p.status)) return false;
        if (!pf_wait_warp(&v_full[j % RV], (j / RV) & 1, abort_flag, p.status)) return false;
        uint8_t* vs = sV + (j % RV) * C::kTileBytes;
        const int k0 = ks + j * BN;
        if (!F8 && k0 + BN > kv_len) {  // NaN hygiene, as below
          const int r_lo = max(0, kv_len - k0), r_hi = min(BN, ((kv_len + 15) & ~15) - k0);
          for (int e = lane; e < (r_hi - r_lo) * C::kCB * 8; e += 32) {
            const int r = r_lo + e / (C::kCB * 8), c = e % (C::kCB * 8);
            *reinterpret_cast<uint4*>(vs + (c / 8) * C::kKVCB + r * 128 + (c % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        const bool use_lo = BF16 && lo_flag[j & 1] == j + 1;
        const uint32_t tP = tmem + (j & 1) * BN;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          if (part == 1 && !use_lo) break;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(smem_addr(vs) + kk * 16 * 128, C::kKVCB, 1024);
            umma_f16_ts_warp(tmem + 2 * BN, tP + 32 * (kk >> 1) + 8 * (kk & 1) + 16 * part, bd,
                             kIdPV, (j > 0 || kk > 0 || part > 0) ? 1u : 0u);
          }
        }
        umma_commit_warp(pv_done(0));
        umma_commit_warp(&v_empty[j % RV]);
        return true;
      };
      if (ok && nt > 0) ok = qk(0);
      if (ok && nt > 1) ok = qk(1);
      for (int j = 0; ok && j < nt; ++j) {
        ok = pv(j);
        if (ok && j + 2 < nt) ok = qk(j + 2);
      }
    }
    for (int j = 0; NQ > 1 && ok && j <= nt; ++j) {
      const int i = j - 1;  // key tile of this step's P.V
      uint8_t* vs = sV + (i >= 0 ? i % RV : 0) * C::kTileBytes;
      if (i >= 0) {
        if (!pf_wait_warp(&v_full[i % RV], (i / RV) & 1, abort_flag, p.status)) { ok = false; break; }
        // Cache slots at or past kv_len hold no key and may hold anything (NaN included):
        // zero those V rows before the tensor cores multiply them by P = 0 (fp8: the
        // dequant warps wrote them as zeros).
        const int k0 = ks + i * BN;
        if (!F8 && k0 + BN > kv_len) {
          const int r_lo = max(0, kv_len - k0), r_hi = min(BN, ((kv_len + 15) & ~15) - k0);
          for (int e = lane; e < (r_hi - r_lo) * C::kCB * 8; e += 32) {
            const int r = r_lo + e / (C::kCB * 8), c = e % (C::kCB * 8);
            *reinterpret_cast<uint4*>(vs + (c / 8) * C::kKVCB + r * 128 + (c % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
      }
      if (j < nt && !pf_wait_warp(&k_full[j % RK], (j / RK) & 1, abort_flag, p.status)) { ok = false; break; }
#pragma unroll
      for (int qt = 0; qt < NQ; ++qt) {
        if (i >= jb[qt] && i < je[qt]) {
          const int n = i - jb[qt];
          if (!pf_wait_warp(p_full(qt), n & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const bool use_lo = BF16 && lo_flag[2 * qt + (n & 1)] == n + 1;
          const uint32_t tP = tmem + qt * C::kTmemStride;
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            if (part == 1 && !use_lo) break;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              const uint64_t bd = smem_desc_sw128(smem_addr(vs) + kk * 16 * 128, C::kKVCB, 1024);
              umma_f16_ts_warp(tP + BN, tP + 32 * (kk >> 1) + 8 * (kk & 1) + 16 * part, bd, kIdPV,
                               (n > 0 || kk > 0 || part > 0) ? 1u : 0u);
            }
          }
          if (i == je[qt] - 1) umma_commit_warp(pv_done(qt));
        }
        if (j >= jb[qt] && j < je[qt]) {
          tc_fence_after();
          const uint32_t qb = smem_addr(sQ + qt * C::kQBytes);
          const uint32_t kb = smem_addr(sK + (j % RK) * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(qb + (kk >> 2) * C::kBM * 128 + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(kb + (kk >> 2) * C::kKVCB + (kk & 3) * 32, 16, 1024);
            umma_f16_ss_warp(tmem + qt * C::kTmemStride, ad, bd, kIdQK, kk > 0 ? 1u : 0u);
          }
          umma_commit_warp(s_full(qt));
        }
      }
      if (!ok) break;
      if (j < nt) umma_commit_warp(&k_empty[j % RK]);
      if (i >= 0) umma_commit_warp(&v_empty[i % RV]);
    }
    // nothing may still be in flight on the tensor cores when the memory is freed
    umma_commit_warp(fin);
    mbar_wait_bounded(fin, 0, p.status, DEV_TIMEOUT);
  } else if (F8 && warp >= kDeq0) {
    // ======================================================== fp8 dequant warps (thread = row)
    // Q (bf16) to f16 in place once; then per key tile, K and V: the staging tile of codes
    // (D-byte rows: 128-byte swizzled at d128, plain at d64) into the f16 ring slot
    // (128-byte swizzled column blocks), each e4m3 value exactly; V rows of keys at or past
    // kv_len become zeros.
    const int td = (warp - kDeq0) * 32 + lane;  // row of a tile
    bool ok = pf_wait_warp(q_full, 0, abort_flag, p.status);
    if (ok && p.q_dtype == UA_DT_BF16) {
#pragma unroll 1
      for (int qt = 0; qt < NQ; ++qt)
#pragma unroll 1
        for (int cb = 0; cb < C::kCB; ++cb) {
          uint4* row = reinterpret_cast<uint4*>(sQ + qt * C::kQBytes + cb * C::kBM * 128 + td * 128);
#pragma unroll
          for (int c0 = 0; c0 < 8; ++c0) {  // element-wise: the order only spreads the banks
            const int c = c0 ^ (td & 7);
            uint4 v = row[c];
            v.x = pack_f16(bf16_lo(v.x), bf16_hi(v.x));
            v.y = pack_f16(bf16_lo(v.y), bf16_hi(v.y));
            v.z = pack_f16(bf16_lo(v.z), bf16_hi(v.z));
            v.w = pack_f16(bf16_lo(v.w), bf16_hi(v.w));
            row[c] = v;
          }
        }
    }
    fence_proxy_async_smem();  // generic writes, read by the tensor cores
    __syncwarp();
    if (lane == 0) mbar_arrive(q_ready);
    // per-token scales: each key's K (V) row is written times its own scale, rounded once
    // to f16 (0 for keys past the partition's walk)
    const bool tok = p.k_scale_tok != nullptr;
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    auto key_scale = [&](int j, int op) -> float {
      const int key = ks + j * BN + td;
      if (key >= ke) return 0.f;
      const int col = key / p.block_size;
      const int blk = col < p.max_blocks_per_seq ? __ldg(bt + col) : -1;
      if (static_cast<unsigned>(blk) >= static_cast<unsigned>(p.num_blocks)) return 0.f;
      const long long slot = key % p.block_size;
      return op == 0 ? __ldg(p.k_scale_tok + blk * p.k_scale_stride[0] +
                             slot * p.k_scale_stride[1] + g * p.k_scale_stride[2])
                     : __ldg(p.v_scale_tok + blk * p.v_scale_stride[0] +
                             slot * p.v_scale_stride[1] + g * p.v_scale_stride[2]);
    };
#pragma unroll 1
    for (int j = 0; ok && j < nt; ++j) {
#pragma unroll 1
      for (int op = 0; op < 2; ++op) {
        const int R = op ? RV : RK;
        uint64_t* const f8_full = op ? v8_full : k8_full;
        uint64_t* const f8_empty = op ? v8_empty : k8_empty;
        const float ts = tok ? key_scale(j, op) : 1.f;
        if (!pf_wait_warp(f8_full, j & 1, abort_flag, p.status)) { ok = false; break; }
        // take the row of codes into registers and hand the staging tile back at once, so
        // the next tile's copy overlaps the conversion
        // 16-code chunk c of the loop is chunk cs(c) of the row.  At d64 (64-byte rows, two
        // to a bank line) the order turns with the row pair a = td / 2 % 4 by pi(a) (pi =
        // 0, 2, 3, 1: pi(a) and pi(a) ^ a both permute 0..3), so the eight rows of a quarter
        // warp hit eight distinct 16-byte bank groups in the loads and in the stores.
        constexpr int kCh = D / 16;
        const uint32_t sw = td & 7;
        const int rot = D == 128 ? 0 : (0x78 >> (2 * ((td >> 1) & 3))) & 3;
        auto cs = [&](int c) -> int { return c ^ rot; };
        uint4 raw[kCh];
        {
          const uint8_t* src = (op ? sV8 : sK8) + td * D;
#pragma unroll
          for (int c = 0; c < kCh; ++c)
            raw[c] = *reinterpret_cast<const uint4*>(
                src + ((D == 128 ? (cs(c) ^ sw) : cs(c)) << 4));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(f8_empty);
        if (j >= R && !pf_wait_warp(&(op ? v_empty : k_empty)[j % R], ((j / R) - 1) & 1,
                                    abort_flag, p.status)) {
          ok = false;
          break;
        }
        uint8_t* dst = (op ? sV : sK) + (j % R) * C::kTileBytes + td * 128;
        const bool zero = op == 1 && ks + j * BN + td >= kv_len;
#pragma unroll
        for (int c = 0; c < kCh; ++c) {  // 16 codes of the row -> f16 chunks 2cs, 2cs + 1
          const uint4 r = zero ? make_uint4(0, 0, 0, 0) : raw[c];
          const uint32_t w[4] = {r.x, r.y, r.z, r.w};
          uint32_t h[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) e4m3x4_to_f16x4(w[q], h[2 * q], h[2 * q + 1]);
          if (tok) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[q]));
              h[q] = pack_f16(f.x * ts, f.y * ts);
            }
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int cc = 2 * cs(c) + u;  // f16 chunk of the row: column block cc / 8
            *reinterpret_cast<uint4*>(dst + (cc >> 3) * C::kKVCB + (((cc & 7) ^ sw) << 4)) =
                make_uint4(h[4 * u], h[4 * u + 1], h[4 * u + 2], h[4 * u + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&(op ? v_full : k_full)[j % R]);
      }
    }
  } else {
    // ======================================================== softmax warps (thread = row)
    // SW warps share a tensor-memory lane quarter: warp `half` takes S columns
    // [half BN / SW, (half + 1) BN / SW) of every key tile and O columns
    // [half D / SW, (half + 1) D / SW).  Once per tile their row maxima meet in shared
    // memory, each rounded up to bf16, and every warp of the row takes the largest: the
    // same running max in every warp, never below the true one.  Their row sums meet at
    // the end through SW columns of the tile's S/P region, free after its last P.V.
    constexpr int kCols = BN / SW, kOCols = D / SW;
    const int qt = warp / (4 * SW);                        // q tile of this warp
    const int quad = warp & 3;                             // its tensor-memory lane quarter
    const int half = (warp % (4 * SW)) >> 2;               // its column slice
    const int r = 32 * quad + lane;                        // row within the q tile
    uint64_t* const xbar = xch_bars + 2 * (4 * qt + quad);  // [0]: row max, [1]: row sum
    uint16_t* const xrow = xch + (qt * 2 * SW) * 128 + r;   // + (slot * SW + h) * 128
    int jb, je;
    tile_walk(qt, jb, je);
    const int n_tiles = je - jb;
    const int tf = t_first + qt * TQ;
    // the row's token within the tile and head within the group (rows token * G + head)
    const int tl = r / G;
    const bool rv = qt < nq_act && r < TQ * G && tf + tl < q_len && q0 + tf + tl < p.total_q;
    // a warp none of whose rows holds a query row (a q tile's unused rows) only keeps the
    // tile barriers in step: what its rows of P and O hold is never stored
    const bool active = __any_sync(0xffffffffu, rv);
    const int i_q = tf + (rv ? tl : 0);                    // query index within the sequence
    const int h = g * G + r % G;
    const int pos = ctx + i_q;
    const int lo_r = p.window_left >= 0 ? max(0, pos - p.window_left) : 0;
    // warp-uniform bounds of this warp's valid rows, to mask only boundary tiles
    int pmin = rv ? pos : INT_MAX, lomax = rv ? lo_r : INT_MIN;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, o));
      lomax = max(lomax, __shfl_xor_sync(0xffffffffu, lomax, o));
    }
    float slope = 0.f;
    const float* qq_row = nullptr;
    if constexpr (FEAT) {
      if (p.alibi != nullptr && rv) slope = __ldg(p.alibi + h);
      if (p.qq_bias != nullptr && rv && i_q < p.max_seqlen_q)
        qq_row = p.qq_bias + static_cast<size_t>(i_q) * p.qq_stride;
    }
    // With no softcap or bias the log2-domain score is c * s with c = scale * log2(e) > 0:
    // the row max is taken on the raw dot products and the scale folds into the exponent's
    // FMA.  Otherwise scores are transformed first and c = log2(e).
    // fp8: the per-tensor k_scale joins the score scale, v_scale the output
    // (per-token scales are already in the f16 tiles)
    const bool tok8 = F8 && p.k_scale_tok != nullptr;
    const float kq = F8 && !tok8 ? p.scale * __ldg(p.kv_scale) : p.scale;
    const float v_mul = F8 && !tok8 ? __ldg(p.kv_scale + 1) : 1.f;
    const float c = FEAT ? kLog2e : kq * kLog2e;
    const bool sink = p.sinks != nullptr && z == 0 && rv;
    float m_used = sink ? __ldg(p.sinks + h) * kLog2e : -INFINITY;
    float l = sink && half == 0 ? 1.f : 0.f;  // the sink's share, counted once per row
    // one q tile: S buffers at columns 0 and BN, O at 2 BN; two: tile qt's S then O
    constexpr bool DB = NQ == 1;
    const uint32_t lane_off = (32u * quad) << 16;
    const uint32_t tS0 = tmem + (DB ? 0u : static_cast<uint32_t>(qt * C::kTmemStride)) + lane_off;
    const uint32_t tO = DB ? tmem + 2 * BN + lane_off : tS0 + BN;
    bool ok = true;

    // softcap / ALiBi / QQ-bias, then (MASK: a boundary tile) the causal / window /
    // partition mask
    // softcap: sc tanh(s / sc) = sc - 2 sc / (1 + 2^(2 log2(e) s / sc)), the score scale folded
    // into ksc (one exp2, one reciprocal, one FMA; +-inf exponents give +-sc); ALiBi:
    // slope (j - ctx) as slope e + abase, abase = slope (first key of the chunk - ctx)
    const float sc = p.softcap;
    const float ksc = sc > 0.f ? kq * 2.f * kLog2e / sc : 0.f;
    auto score = [&](float v, int jk, float abase, int e, auto mask) -> float {
      if constexpr (FEAT) {
        if (sc > 0.f) v = fmaf(-2.f * sc, fast_rcp(fast_exp2(v * ksc) + 1.f), sc);
        else v *= kq;
        v += fmaf(slope, static_cast<float>(e), abase);
        if (qq_row != nullptr && jk >= ctx && jk <= pos) v += __ldg(qq_row + (jk - ctx));
      }
      if constexpr (decltype(mask)::value) {
        if (!(rv && jk >= lo_r && jk <= pos && jk < ke)) v = -INFINITY;
      }
      return v;
    };

    for (int n = 0; n < n_tiles; ++n) {
      uint64_t* const sf = DB ? s_full_b(n & 1) : s_full(qt);
      uint64_t* const pf = DB ? p_full_b(n & 1) : p_full(qt);
      const uint32_t tS = DB ? tS0 + (n & 1) * BN : tS0;
      if (!pf_wait_warp(sf, DB ? (n >> 1) & 1 : n & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      if (!active) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pf);
        continue;
      }
      const int k0 = ks + (jb + n) * BN;
      const bool need_mask = k0 < lomax || k0 + BN - 1 > pmin || k0 + BN > ke;

      // ---- pass 1: row max (two 32-column loads in flight).  Scores that need a transform
      // or a mask get it here, once, and are written back over S for pass 2.
      const bool rewrite = FEAT || need_mask;
      float mx0 = -INFINITY, mx1 = -INFINITY;
      constexpr bool kTwo = kCols >= 64;  // two 32-column loads an iteration
#pragma unroll 1
      for (int c0 = half * kCols; c0 < (half + 1) * kCols; c0 += kTwo ? 64 : 32) {
        uint32_t ra[32], rb[32];
        tmem_ld32(tS + c0, ra);
        if constexpr (kTwo) tmem_ld32(tS + c0 + 32, rb);
        tmem_ld_wait();
        if (rewrite) {
          const float ab = FEAT ? slope * static_cast<float>(k0 + c0 - ctx) : 0.f;
          if (need_mask) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              ra[e] = __float_as_uint(score(__uint_as_float(ra[e]), k0 + c0 + e, ab, e, std::true_type{}));
              if constexpr (kTwo)
                rb[e] = __float_as_uint(score(__uint_as_float(rb[e]), k0 + c0 + 32 + e, ab, 32 + e, std::true_type{}));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              ra[e] = __float_as_uint(score(__uint_as_float(ra[e]), k0 + c0 + e, ab, e, std::false_type{}));
              if constexpr (kTwo)
                rb[e] = __float_as_uint(score(__uint_as_float(rb[e]), k0 + c0 + 32 + e, ab, 32 + e, std::false_type{}));
            }
          }
          tmem_st32(tS + c0, ra);
          if constexpr (kTwo) tmem_st32(tS + c0 + 32, rb);
        }
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          mx0 = fmax3(mx0, __uint_as_float(ra[e]), __uint_as_float(ra[e + 1]));
          if constexpr (kTwo) mx1 = fmax3(mx1, __uint_as_float(rb[e]), __uint_as_float(rb[e + 1]));
        }
      }
      if (rewrite) tmem_st_wait();
      float mx = fmaxf(mx0, mx1) * c;  // row max in log2 units (-inf stays -inf)
      if constexpr (SW > 1) {
        // the row's other column slices: every lane arrives once its value is written.  Two
        // slots: a warp writes tile n + 2's slot only after its S wait, which follows the
        // P.V of tile n, which waited for every warp's P of tile n, written after the reads.
        const uint32_t u = __float_as_uint(mx);
        uint16_t* const slot = xrow + (n & 1) * SW * 128;
        slot[half * 128] = static_cast<uint16_t>(
            ((u & 0xFFFFu) == 0u || (u >> 31)) ? (u >> 16) : (u >> 16) + 1u);  // round up
        mbar_arrive(&xbar[0]);
        if (!pf_wait_warp(&xbar[0], n & 1, abort_flag, p.status)) { ok = false; break; }
        mx = -INFINITY;
#pragma unroll
        for (int hh = 0; hh < SW; ++hh)
          mx = fmaxf(mx, __uint_as_float(static_cast<uint32_t>(slot[hh * 128]) << 16));
      }
      // ---- running max, used lazily: O and l are rescaled only when the max grows by
      // more than 8 in log2 units (P stays <= 256, far inside the fp32 and P ranges)
      float alpha = 1.f;
      const bool grow = mx > m_used + 8.f || (m_used == -INFINITY && mx > -INFINITY);
      if (grow) {
        alpha = m_used == -INFINITY ? 0.f : fast_exp2(m_used - mx);
        m_used = mx;
      }
      const float m_use = m_used == -INFINITY ? 0.f : m_used;
      // O holds P.V of step n-1: with one S buffer the commit of this step's S covered it;
      // with two (S_n issued before P.V_{n-1}) wait for that P.V's own phase, every step,
      // so the parity waits stay exact
      if (DB && n >= 1) {
        if (!pf_wait_warp(pv_done(0), (n - 1) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
      }
      if (n >= 1 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
        for (int c0 = half * kOCols; c0 < (half + 1) * kOCols; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(tO + c0, rr);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
          tmem_st32(tO + c0, rr);
        }
      }
      // the low part of P matters only where one key can still weigh more than 1/64 of the
      // row sum; l * alpha + pmax is a lower bound of the new sum
      const float pmax = mx == -INFINITY ? 0.f : fast_exp2(mx - m_use);
      const bool warp_lo = BF16 && __any_sync(0xffffffffu, pmax * 63.f > l * alpha);

      // ---- pass 2: P = 2^(c s - m) over S, 32 keys at a time: 16 columns of high part
      // (bf16 or f16 pairs), then 16 columns of bf16 remainder (zeros when not needed)
      const float2 cc = make_float2(c, c), mm = make_float2(-m_use, -m_use);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      // one 32-key group: P and its remainder over the group's S columns
      auto p_group = [&](int c0, uint32_t* rr) {
        float xv[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) xv[e] = __uint_as_float(rr[e]);
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float2 u = __ffma2_rn(make_float2(xv[e], xv[e + 1]), cc, mm);
          const float2 w = __ffma2_rn(make_float2(xv[e + 2], xv[e + 3]), cc, mm);
          xv[e] = fast_exp2(u.x);
          xv[e + 1] = fast_exp2(u.y);
          xv[e + 2] = fast_exp2(w.x);
          xv[e + 3] = fast_exp2(w.y);
          acc0 = __fadd2_rn(acc0, make_float2(xv[e], xv[e + 1]));
          acc1 = __fadd2_rn(acc1, make_float2(xv[e + 2], xv[e + 3]));
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint32_t hw = BF16 ? pack_bf16(xv[2 * e], xv[2 * e + 1]) : pack_f16(xv[2 * e], xv[2 * e + 1]);
          rr[e] = hw;
          if (BF16 && warp_lo) {
            const float2 rem = __fadd2_rn(make_float2(xv[2 * e], xv[2 * e + 1]),
                                          make_float2(-bf16_lo(hw), -bf16_hi(hw)));
            rr[16 + e] = pack_bf16(rem.x, rem.y);
          } else {
            rr[16 + e] = 0u;
          }
        }
        tmem_st32(tS + c0, *reinterpret_cast<uint32_t(*)[32]>(rr));
      };
#pragma unroll 1
      for (int c0 = half * kCols; c0 < (half + 1) * kCols; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(tS + c0, rr);
        tmem_ld_wait();
        p_group(c0, rr);
      }
      l = l * alpha + ((acc0.x + acc0.y) + (acc1.x + acc1.y));
      tmem_st_wait();
      if (warp_lo && lane == 0) lo_flag[2 * qt + (n & 1)] = n + 1;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pf);
    }

    // ---- epilogue: O / l for one partition, or the partition's max / sum / O
    // the last P.V (two S buffers: the tile's last pv_done phase; one: its only phase)
    if (ok && n_tiles > 0 && active)
      ok = pf_wait_warp(pv_done(qt), DB ? (n_tiles - 1) & 1 : 0, abort_flag, p.status);
    tc_fence_after();
    if constexpr (SW > 1) {
      if (ok && active) {  // the row sum over every column slice, through tensor memory
        tmem_st1(tS0 + half, __float_as_uint(l));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&xbar[1]);
        ok = pf_wait_warp(&xbar[1], 0, abort_flag, p.status);
        tc_fence_after();
        if constexpr (SW == 2) {
          uint32_t l0, l1;
          tmem_ld2(tS0, l0, l1);
          tmem_ld_wait();
          l = __uint_as_float(l0) + __uint_as_float(l1);
        } else {
          uint32_t l4[4];
          tmem_ld4(tS0, l4);
          tmem_ld_wait();
          l = (__uint_as_float(l4[0]) + __uint_as_float(l4[1])) +
              (__uint_as_float(l4[2]) + __uint_as_float(l4[3]));
        }
      }
    }
    if (ok && active) {
      const size_t orow = static_cast<size_t>(q0 + i_q) * p.hq + h;
      const size_t n_part = static_cast<size_t>(p.n_part);
      const float inv = l > 0.f ? v_mul / l : 0.f;
      // One q tile: a split's partial rows leave through a 4 KB slice of the K/V ring that
      // this warp alone owns now (the ring's last reader, the tile's last P.V, is complete),
      // so that each store writes whole 128-byte runs of four rows instead of 16 bytes of 32
      // rows; only for warps with more than a quarter of their rows valid (a decode row or
      // two store faster straight from their lanes).  (In the two-tile kernel the same code
      // measured 5 % slower on the fp8 long prefill, which never splits: left out there.)
      const long long wrow = rv ? static_cast<long long>(orow * n_part + z) : -1;
      const bool staged = NQ == 1 && n_part > 1 && n_tiles > 0 &&
                          __popc(__ballot_sync(0xffffffffu, rv)) > 8;
#pragma unroll 1
      for (int c0 = half * kOCols; c0 < (half + 1) * kOCols; c0 += 32) {
        uint32_t rr[32];
        if (n_tiles > 0) {
          tmem_ld32(tO + c0, rr);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = 0u;
        }
        if constexpr (NQ == 1) {
          if (staged) {
            // this lane's row, 16-byte chunk k at position k ^ (row mod 8) (conflict-free
            // both ways); then lane l copies chunk l mod 8 of rows l / 8 + 4 j
            float* const stg = reinterpret_cast<float*>(sK) + (warp % (4 * SW)) * 1024;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              *reinterpret_cast<float4*>(stg + lane * 32 + ((k ^ (lane & 7)) << 2)) =
                  make_float4(__uint_as_float(rr[4 * k]) * v_mul,
                              __uint_as_float(rr[4 * k + 1]) * v_mul,
                              __uint_as_float(rr[4 * k + 2]) * v_mul,
                              __uint_as_float(rr[4 * k + 3]) * v_mul);
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int rw = (lane >> 3) + 4 * j, ck = lane & 7;
              const unsigned hi32 = static_cast<unsigned>(
                  __shfl_sync(0xffffffffu, static_cast<int>(wrow >> 32), rw));
              const unsigned lo32 =
                  static_cast<unsigned>(__shfl_sync(0xffffffffu, static_cast<int>(wrow), rw));
              const long long wr =
                  static_cast<long long>((static_cast<unsigned long long>(hi32) << 32) | lo32);
              const float4 v =
                  *reinterpret_cast<const float4*>(stg + rw * 32 + ((ck ^ (rw & 7)) << 2));
              if (wr >= 0) *reinterpret_cast<float4*>(p.ws_acc + wr * D + c0 + 4 * ck) = v;
            }
            __syncwarp();
            if (rv && c0 == 0) {
              p.ws_m[wrow] = m_used;
              p.ws_l[wrow] = l;
            }
            continue;
          }
        }
        if (!rv) continue;
        if (n_part > 1) {  // the partition's max, sum and unnormalised row
          const size_t w = orow * n_part + z;
          if (c0 == 0) {
            p.ws_m[w] = m_used;
            p.ws_l[w] = l;
          }
          float4* dst = reinterpret_cast<float4*>(p.ws_acc + w * D + c0);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(rr[4 * e]) * v_mul, __uint_as_float(rr[4 * e + 1]) * v_mul,
                                 __uint_as_float(rr[4 * e + 2]) * v_mul, __uint_as_float(rr[4 * e + 3]) * v_mul);
        } else {
          if (p.out_dtype == UA_DT_F32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * D + c0);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(__uint_as_float(rr[4 * e]) * inv, __uint_as_float(rr[4 * e + 1]) * inv,
                                   __uint_as_float(rr[4 * e + 2]) * inv, __uint_as_float(rr[4 * e + 3]) * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow * D + c0);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint32_t w[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float a0 = __uint_as_float(rr[8 * e + 2 * q]) * inv;
                const float a1 = __uint_as_float(rr[8 * e + 2 * q + 1]) * inv;
                w[q] = p.out_dtype == UA_DT_BF16 ? pack_bf16(a0, a1) : pack_f16(a0, a1);
              }
              dst[e] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMma) tmem_dealloc(tmem, C::kTmemCols);
}

// One q tile a CTA: four softmax warps per lane quarter at head_dim 128 with a 16-bit cache
// (32 key columns a warp: the per-tile chain of a thread shortens; the mixed batch went
// from 24.5 to 22 us against two), two at head_dim 64 (O's 64 columns) and for fp8 caches
// (the dequant warps' registers).  A CTA would otherwise have one softmax warp per SM
// sub-partition.  Two q tiles already alternate on the tensor cores; splitting their
// softmax too measured slower on GB300 (the d128 long prefill went from 1.12 to 1.19 ms).
template <int D, int NQ, bool BF16, bool FEAT, bool F8 = false>
cudaError_t launch_prefill_tm_t(const PrefillParams& pp, dim3 grid, cudaStream_t stream) {
  constexpr int SW = NQ == 1 ? (D == 128 && !F8 ? 4 : 2) : 1;
  using C = PrefillTmCfg<D, NQ, F8, SW>;
  auto kern = ua_prefill_tm_kernel<D, NQ, BF16, FEAT, F8, SW>;
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
  return launch_pdl(kern, grid, dim3(C::kThreads), C::kSmemBytes, stream, 1, pp);
}

template <int D, int NQ>
cudaError_t launch_prefill_tm_nq(const PrefillParams& pp, dim3 grid, int kv, bool feat,
                                 cudaStream_t s) {
  if (kv == KV_BF16)
    return feat ? launch_prefill_tm_t<D, NQ, true, true>(pp, grid, s)
                : launch_prefill_tm_t<D, NQ, true, false>(pp, grid, s);
  if (kv == KV_F16)
    return feat ? launch_prefill_tm_t<D, NQ, false, true>(pp, grid, s)
                : launch_prefill_tm_t<D, NQ, false, false>(pp, grid, s);
  if (kv == KV_E4M3)
    return feat ? launch_prefill_tm_t<D, NQ, false, true, true>(pp, grid, s)
                : launch_prefill_tm_t<D, NQ, false, false, true>(pp, grid, s);
  return cudaErrorInvalidValue;
}

// nq: q tiles of 128 rows per CTA (1 or 2).
template <int D>
cudaError_t launch_prefill_tm_dispatch(const PrefillParams& pp, dim3 grid, int kv, bool feat, int nq,
                                       cudaStream_t s) {
  if (nq == 2) return launch_prefill_tm_nq<D, 2>(pp, grid, kv, feat, s);
  if (nq == 1) return launch_prefill_tm_nq<D, 1>(pp, grid, kv, feat, s);
  return cudaErrorInvalidValue;
}

}  // namespace ua
