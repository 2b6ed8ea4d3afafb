// ua_prefill_wide.cuh -- the tensor-memory attention kernel of libua.so for prefill-shaped
// q-blocks with head_dim 256 (included by ua_prefill_d256.cu).
//
// One CTA owns (q-block, kv-head g, key partition z).  A q-block is one q tile of 128
// rows: TQ = floor(128 / G) consecutive query tokens times the G query heads that read
// kv-head g, so the GQA heads of a group share every K/V tile (vllm-rdna PR #34 "FA-RDNA2
// D=128 prefill", "Change" 1, on tensor cores).  Per key tile j of BN = 128 keys:
//
//   S_j = Q K_j^T   tcgen05.mma (kind::f16, M=128, N=128, fp32) into tensor memory
//   softmax         as in ua_prefill_tm.cuh: one thread per row, pass 1 for the row max
//                   (scores transformed and masked once, written back), pass 2 writes
//                   P = 2^(s - m) over S as bf16 high part + remainder (or f16)
//   O += P_j V_j    two tcgen05.mma passes of N = 128 (O columns 0..127 and 128..255),
//                   A = P read from tensor memory, B = V from shared memory
//
// Tensor memory: S/P double-buffered (2 x 128 columns) and O (256 columns).  The MMA
// warp issues ... P.V_{j-1}, S_{j+1}, [P_j ready] P.V_j, S_{j+2} ..., so the tensor cores
// compute the next S and the previous P.V while the softmax warps work on tile j; S_{j+2}
// overwrites P_j only after P.V_j, in issue order.  Each commit covers every earlier MMA
// of the thread, so when S_j is ready P.V_{j-2} is done; the softmax rescales O (only
// when a row's max grows by more than 2^8) after also waiting for P.V_{j-1}.
//
// Shared memory: Q (64 KB) and a ring of five 32 KB slots.  A slot holds half of a K or V
// tile (128 keys x 128 of the 256 columns); slots are filled in the order the MMA warp
// reads them: K_0, then for every j: K_{j+1}, V_j.
//
// Warp roles (288 threads): warps 0..3 softmax + epilogue (thread = row = tensor-memory
// lane), warps 4..7 TMA producers (a 128-key step moves 128 KB as 64 page boxes, more
// than one warp issues in time), warp 8 MMA issuer and tensor-memory owner.
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

// F8: fp8-e4m3 caches.  The producers copy each half tile of codes (128 keys x 128 bytes)
// into a two-slot staging ring, and eight dequant warps (thread = one key's 64-column half)
// write it into its f16 slot, exactly (every e4m3 value is an f16), so the f16 MMAs and the softmax run
// unchanged; k_scale joins the score scale and v_scale the output (per-token scales:
// folded into each key's f16 row instead).
template <int D, bool F8 = false>
struct PrefillWideCfg {
  static constexpr int kBM = 128;                   // MMA rows of the q tile
  static constexpr int kBN = 128;                   // keys per tile
  static constexpr int kCB = D / 64;                // 128-byte column blocks of a row
  static constexpr int kQBytes = kCB * kBM * 128;
  static constexpr int kSlotCB = 2;                 // column blocks of one half tile
  static constexpr int kSlotCBBytes = kBN * 128;    // one column block of a half tile
  static constexpr int kSlotBytes = kSlotCB * kSlotCBBytes;
  static constexpr int kSlots = F8 ? 4 : 5;         // f16 half tiles
  static constexpr int kStage = F8 ? 2 : 0;         // fp8: staging slots of codes
  static constexpr int kStageBytes = kBN * 128;     // one staged half tile of codes
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes =
      1024 + kQBytes + kSlots * kSlotBytes + kStage * kStageBytes + kBarBytes;
  static constexpr int kTmemCols = 512;             // S0, S1, O
  // TMA producer warps: a 16-bit half tile is 16 page boxes, an fp8 one 8.  Each producer
  // reuses the staging slot of its own previous item, so the fp8 staging ring holds as many
  // items as there are producers (a producer's parity wait is then never more than one
  // phase behind).
  static constexpr int kProducers = F8 ? 2 : 4;
  // eight dequant warps: thread = (key, column half); with four (thread = key) each item's
  // conversion took twice as long on the critical path
  static constexpr int kDeqWarps = F8 ? 8 : 0;
  static constexpr int kThreads = 32 * (4 + kProducers + 1 + kDeqWarps);
  static_assert(D == 256, "two half tiles of 128 columns");
  static_assert(2 * kBN + D <= kTmemCols, "tensor memory budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(!F8 || kStage == kProducers, "one staging slot per producer warp");
};

// Position of half h of K tile j and of V tile j in the slot sequence
// K_0, then for j = 0 .. nt-1: K_{j+1} (when j + 1 < nt), V_j.
__device__ __forceinline__ int wide_item_k(int j, int h) { return j == 0 ? h : 4 * j - 2 + h; }
__device__ __forceinline__ int wide_item_v(int j, int h, int nt) {
  return j < nt - 1 ? 4 * j + 4 + h : 4 * j + 2 + h;
}

template <int D, bool BF16, bool FEAT, bool F8 = false>
__global__ void __launch_bounds__(PrefillWideCfg<D, F8>::kThreads, 1)
    ua_prefill_wide_kernel(const __grid_constant__ PrefillParams pp) {
  using C = PrefillWideCfg<D, F8>;
  constexpr int BN = C::kBN;
  constexpr int NS = C::kSlots;
  constexpr int kMma = 4 + C::kProducers;
  constexpr int kDeq0 = kMma + 1;  // fp8: dequant warps kDeq0 .. kDeq0 + 7
  static_assert(!F8 || !BF16, "fp8 caches run the f16 MMAs");
  const AttnParams& p = pp.p;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* const smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* const sQ = smem;
  uint8_t* const sR = sQ + C::kQBytes;                // NS slots
  uint8_t* const s8 = sR + NS * C::kSlotBytes;         // fp8: staging slots of codes
  uint64_t* const bars = reinterpret_cast<uint64_t*>(s8 + C::kStage * C::kStageBytes);
  uint64_t* const q_full = bars + 0;
  uint64_t* const fin = bars + 1;
  uint64_t* const pv_done = bars + 2;                 // one phase per P.V_j
  uint64_t* const s_full = bars + 3;                  // [2]: S buffer b ready
  uint64_t* const p_full = bars + 5;                  // [2]: P in S buffer b ready
  uint64_t* const full = bars + 7;                    // [NS]
  uint64_t* const empty = full + NS;                  // [NS]
  uint64_t* const lo_bar = empty + NS;                // the softmax warps agree on P's low part
  // fp8: Q converted (dequant warps), staging slot full (copies) and empty (dequant warps)
  uint64_t* const q_ready = lo_bar + 1;
  uint64_t* const s8_full = q_ready + 1;              // [kStage]
  uint64_t* const s8_empty = s8_full + C::kStage;     // [kStage]
  uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(s8_empty + C::kStage);
  int* const lo_flag = reinterpret_cast<int*>(tmem_holder + 1);  // [2]: step + 1 when P_lo matters
  __shared__ int s_abort;
  __shared__ int s_last[C::kProducers];  // last item each producer warp issued

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int z = blockIdx.z;
  const int G = p.group;
  const int TQ = pp.tq;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(fin, 1);
    mbar_init(pv_done, 1);
    mbar_init(lo_bar, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      lo_flag[i] = 0;
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], F8 ? C::kDeqWarps : 1);  // f16 slots: written by the copies or
      mbar_init(&empty[i], 1);                      // (fp8) the dequant warps
    }
    if constexpr (F8) {
      mbar_init(q_ready, C::kDeqWarps);
      for (int i = 0; i < C::kStage; ++i) {
        mbar_init(&s8_full[i], 1);
        mbar_init(&s8_empty[i], C::kDeqWarps);
      }
    }
    s_abort = 0;
    mbar_fence_init();
  }
  // Q rows past the block's tokens stay zero (they are computed and dropped).
  {
    const int pad = (C::kBM - TQ * G) * 8;
    for (int i = threadIdx.x; i < C::kCB * pad; i += C::kThreads) {
      const int cb = i / pad, rem = i % pad;
      *reinterpret_cast<uint4*>(sQ + cb * C::kBM * 128 + (TQ * G + rem / 8) * 128 + (rem % 8) * 16) =
          make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();
  if (warp == kMma) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&pp.tmap_q);
    tma_prefetch_desc(&pp.tmap_k);
    tma_prefetch_desc(&pp.tmap_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tO = tmem + 2 * BN;
  volatile int* abort_flag = &s_abort;
  // Everything above touches only this CTA's shared and tensor memory, so it overlaps the
  // previous kernel's tail (programmatic dependent launch); global memory is read below.
  grid_dependency_wait();
  grid_launch_dependents();

  // Longest walks first: slots are taken in reverse order.
  const int x = static_cast<int>(gridDim.x - 1 - blockIdx.x);
  const PfSeq sq = pf_seq_of_slot(p.cu_seqlens_q, p.seq_lens_k, p.num_seqs, x, TQ);
  const int b = sq.b, q0 = sq.q0, q_len = sq.q_len, kv_len = sq.kv_len;
  const int t_first = (x - (q0 / TQ + b)) * TQ;
  if (t_first < 0 || t_first >= q_len) {  // idle slot: uniform for the CTA
    if (warp == kMma) tmem_dealloc(tmem, C::kTmemCols);
    return;
  }
  const int t_last = min(t_first + TQ, q_len) - 1;
  const int ctx = kv_len - q_len;
  const int pos_first = ctx + t_first, pos_last = ctx + t_last;
  const int hi = max(0, min(pos_last + 1, kv_len));
  const int lo = min(hi, p.window_left >= 0 ? max(0, pos_first - p.window_left) : 0) & ~15;
  int part = (hi - lo + p.n_part - 1) / p.n_part;
  part = (part + 15) & ~15;
  const int ks = min(lo + z * part, hi);
  const int ke = min(ks + part, hi);
  const int nt = (ke - ks + BN - 1) / BN;

  if (warp >= 4 && warp < 4 + C::kProducers) {
    // ======================================================== TMA producers
    // Producer warp pw issues the items u = pw, pw + NP, ... of the slot sequence; lane
    // i < 16 issues page i / 2 (16 keys), column block i % 2 of the item's half tile
    // (fp8: lane i < 8 page i, the half tile's one 128-byte column block, into the staging
    // slot u % NP).
    constexpr int NP = C::kProducers;
    constexpr int NR = F8 ? C::kStage : NS;  // slots this warp's copies land in
    const int pw = warp - 4;
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    const int bs = p.block_size;
    const int oob = p.num_blocks * bs;
    const int page = F8 ? lane : lane >> 1, cbl = F8 ? 0 : lane & 1;
    constexpr int kBoxLanes = F8 ? 8 : 16;
    if (pw == 0 && lane == 0) {
      mbar_arrive_expect_tx(q_full, C::kCB * TQ * G * 128);
      for (int cb = 0; cb < C::kCB; ++cb)
        tma_load_3d_pf(sQ + cb * C::kBM * 128, &pp.tmap_q, 64 * cb, g * G, q0 + t_first, q_full);
    }
    const int n_items = 4 * nt;
    // item u: K or V, tile j, half h
    auto decode = [&](int u, bool& is_k, int& j, int& h) {
      if (u < 2) {
        is_k = true, j = 0, h = u;
        return;
      }
      const int v = u - 2, blk4 = v >> 2, r = v & 3;
      is_k = blk4 < nt - 1 && r < 2;
      j = is_k ? blk4 + 1 : blk4;
      h = r & 1;
    };
    // block id of this lane's page of tile j (-1: none), loaded an item ahead of its use
    auto page_blk = [&](int j) -> int {
      const int key = ks + j * BN + 16 * page;
      const int col = key / bs;
      return (j < nt && lane < kBoxLanes && key < ke && col < p.max_blocks_per_seq) ? __ldg(bt + col) : -1;
    };
    auto page_row = [&](int j, int blk) -> int {
      const int key = ks + j * BN + 16 * page;
      if (lane >= kBoxLanes || key >= ke) return oob;
      if (static_cast<unsigned>(blk) >= static_cast<unsigned>(p.num_blocks)) {
        atomicOr(p.status, DEV_BAD_BLOCK);
        return oob;
      }
      return blk * bs + key % bs;
    };
    bool is_k;
    int j, h;
    int blk_cur = -1;
    if (pw < n_items) {
      decode(pw, is_k, j, h);
      blk_cur = page_blk(j);
    }
    int last = -1;
    for (int u = pw; u < n_items; u += NP) {
      decode(u, is_k, j, h);
      const int row = page_row(j, blk_cur);
      if (u + NP < n_items) {
        bool k2;
        int j2, h2;
        decode(u + NP, k2, j2, h2);
        blk_cur = page_blk(j2);
      }
      const int sl = u % NR;
      uint64_t* const f = F8 ? &s8_full[sl] : &full[sl];
      uint64_t* const e = F8 ? &s8_empty[sl] : &empty[sl];
      if (u >= NR && !pf_wait_warp(e, ((u / NR) - 1) & 1, abort_flag, p.status)) break;
      if (lane == 0) mbar_arrive_expect_tx(f, F8 ? C::kStageBytes : C::kSlotBytes);
      __syncwarp();
      if (lane < kBoxLanes) {
        if constexpr (F8)
          tma_load_3d_pf(s8 + sl * C::kStageBytes + page * 2048, is_k ? &pp.tmap_k : &pp.tmap_v,
                         128 * h, g, row, f);
        else
          tma_load_3d_pf(sR + sl * C::kSlotBytes + cbl * C::kSlotCBBytes + page * 2048,
                         is_k ? &pp.tmap_k : &pp.tmap_v, 64 * (2 * h + cbl), g, row, f);
      }
      last = u;
    }
    // Never leave copies in flight into this CTA's shared memory (even after an abort).
    // An item whose slot was taken by item u + NS was consumed, so it landed; the others
    // are waited for.  Items are issued in order per warp, so item u + NS was issued iff
    // its warp's last item is at least u + NS.
    if (lane == 0) s_last[pw] = last;
    named_bar_sync(2, 32 * NP);
    for (int u = last; u >= 0 && u > last - NR; u -= NP)
      if (s_last[(u + NR) % NP] < u + NR)
        mbar_wait_bounded(F8 ? &s8_full[u % NR] : &full[u % NR], (u / NR) & 1, p.status,
                          DEV_TIMEOUT);
    if (pw == 0 && lane == 0) mbar_wait_bounded(q_full, 0, p.status, DEV_TIMEOUT);
  } else if (warp == kMma) {
    // ======================================================== MMA issuer (converged warp)
    constexpr uint32_t kIdQK = umma_idesc_f16(128, BN, BF16, false);
    constexpr uint32_t kIdPV = umma_idesc_f16(128, 128, BF16, true);
    bool ok = pf_wait_warp(F8 ? q_ready : q_full, 0, abort_flag, p.status);
    auto qk = [&](int j) -> bool {
      const uint32_t tS = tmem + (j & 1) * BN;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int u = wide_item_k(j, h), sl = u % NS;
        if (!pf_wait_warp(&full[sl], (u / NS) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t kb = smem_addr(sR + sl * C::kSlotBytes);
#pragma unroll
        for (int kl = 0; kl < 8; ++kl) {
          const int kk = 8 * h + kl;  // 16-column step over D
          const uint64_t ad = smem_desc_sw128(smem_addr(sQ) + (kk >> 2) * C::kBM * 128 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(kb + (kl >> 2) * C::kSlotCBBytes + (kl & 3) * 32, 16, 1024);
          umma_f16_ss_warp(tS, ad, bd, kIdQK, kk > 0 ? 1u : 0u);
        }
        umma_commit_warp(&empty[sl]);
      }
      umma_commit_warp(&s_full[j & 1]);
      return true;
    };
    auto pv = [&](int j) -> bool {
      if (!pf_wait_warp(&p_full[j & 1], (j >> 1) & 1, abort_flag, p.status)) return false;
      tc_fence_after();
      const bool use_lo = BF16 && lo_flag[j & 1] == j + 1;
      const uint32_t tP = tmem + (j & 1) * BN;
      const int k0 = ks + j * BN;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int u = wide_item_v(j, h, nt), sl = u % NS;
        if (!pf_wait_warp(&full[sl], (u / NS) & 1, abort_flag, p.status)) return false;
        uint8_t* vs = sR + sl * C::kSlotBytes;
        // Cache slots at or past kv_len hold no key and may hold anything (NaN included):
        // zero those V rows before the tensor cores multiply them by P = 0 (fp8: the
        // dequant warps wrote them as zeros).
        if (!F8 && k0 + BN > kv_len) {
          const int r_lo = max(0, kv_len - k0), r_hi = min(BN, ((kv_len + 15) & ~15) - k0);
          for (int e = lane; e < (r_hi - r_lo) * C::kSlotCB * 8; e += 32) {
            const int r = r_lo + e / (C::kSlotCB * 8), c = e % (C::kSlotCB * 8);
            *reinterpret_cast<uint4*>(vs + (c / 8) * C::kSlotCBBytes + r * 128 + (c % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          if (part == 1 && !use_lo) break;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(smem_addr(vs) + kk * 16 * 128, C::kSlotCBBytes, 1024);
            umma_f16_ts_warp(tO + 128 * h, tP + 32 * (kk >> 1) + 8 * (kk & 1) + 16 * part, bd, kIdPV,
                             (j > 0 || kk > 0 || part > 0) ? 1u : 0u);
          }
        }
        umma_commit_warp(&empty[sl]);
      }
      umma_commit_warp(pv_done);
      return true;
    };
    if (ok && nt > 0) ok = qk(0);
    if (ok && nt > 1) ok = qk(1);
    for (int j = 0; ok && j < nt; ++j) {
      ok = pv(j);
      if (ok && j + 2 < nt) ok = qk(j + 2);
    }
    // nothing may still be in flight on the tensor cores when the memory is freed
    umma_commit_warp(fin);
    mbar_wait_bounded(fin, 0, p.status, DEV_TIMEOUT);
  } else if (F8 && warp >= kDeq0) {
    // ======================================================== fp8 dequant warps
    // Thread (key td, column half hc): Q (bf16) to f16 in place once (row td, column blocks
    // of half hc); then every item of the slot sequence: codes 64 hc .. 64 hc + 63 of the
    // staged half tile (128-byte rows, 128-byte swizzled) into column block hc of its f16
    // slot, each e4m3 value exactly, or times the key's own scale (per-token scales); V
    // rows of keys at or past kv_len become zeros.
    const int tdh = (warp - kDeq0) * 32 + lane;
    const int td = tdh & (BN - 1), hc = tdh / BN;
    const uint32_t sw = td & 7;
    bool ok = pf_wait_warp(q_full, 0, abort_flag, p.status);
    if (ok && p.q_dtype == UA_DT_BF16) {
#pragma unroll 1
      for (int cb = hc * (C::kCB / 2); cb < (hc + 1) * (C::kCB / 2); ++cb) {
        uint4* row = reinterpret_cast<uint4*>(sQ + cb * C::kBM * 128 + td * 128);
#pragma unroll
        for (int c0 = 0; c0 < 8; ++c0) {  // element-wise: the order only spreads the banks
          const int c = c0 ^ static_cast<int>(sw);
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
    const bool tok = p.k_scale_tok != nullptr;
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    // the per-token scale of this thread's key of tile j (0 past the partition's keys)
    auto key_scale = [&](int j, bool is_k) -> float {
      const int key = ks + j * BN + td;
      if (key >= ke) return 0.f;
      const int col = key / p.block_size;
      const int blk = col < p.max_blocks_per_seq ? __ldg(bt + col) : -1;
      if (static_cast<unsigned>(blk) >= static_cast<unsigned>(p.num_blocks)) return 0.f;
      const long long slot = key % p.block_size;
      return is_k ? __ldg(p.k_scale_tok + blk * p.k_scale_stride[0] + slot * p.k_scale_stride[1] +
                          g * p.k_scale_stride[2])
                  : __ldg(p.v_scale_tok + blk * p.v_scale_stride[0] + slot * p.v_scale_stride[1] +
                          g * p.v_scale_stride[2]);
    };
    const int n_items = 4 * nt;
#pragma unroll 1
    for (int u = 0; ok && u < n_items; ++u) {
      bool is_k;
      int j, h;
      if (u < 2) {
        is_k = true, j = 0, h = u;
      } else {
        const int v = u - 2, blk4 = v >> 2, r = v & 3;
        is_k = blk4 < nt - 1 && r < 2;
        j = is_k ? blk4 + 1 : blk4;
        h = r & 1;
      }
      const float ts = tok ? key_scale(j, is_k) : 1.f;
      const int st = u % C::kStage;
      if (!pf_wait_warp(&s8_full[st], (u / C::kStage) & 1, abort_flag, p.status)) { ok = false; break; }
      // take the half row of codes into registers and hand the staging slot back at once
      uint4 raw[4];
      {
        const uint8_t* src = s8 + st * C::kStageBytes + td * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          raw[c] = *reinterpret_cast<const uint4*>(src + (((4 * hc + c) ^ sw) << 4));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s8_empty[st]);
      const int sl = u % NS;
      if (u >= NS && !pf_wait_warp(&empty[sl], ((u / NS) - 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      uint8_t* dst = sR + sl * C::kSlotBytes + td * 128;
      const bool zero = !is_k && ks + j * BN + td >= kv_len;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {  // 16 codes of the row -> f16 chunks 2c, 2c + 1
        const int c = 4 * hc + c4;
        const uint4 r = zero ? make_uint4(0, 0, 0, 0) : raw[c4];
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
        uint32_t hh[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) e4m3x4_to_f16x4(w[q], hh[2 * q], hh[2 * q + 1]);
        if (tok) {  // the key's scale, rounded once to f16 with each value
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hh[q]));
            hh[q] = pack_f16(f.x * ts, f.y * ts);
          }
        }
#pragma unroll
        for (int uu = 0; uu < 2; ++uu) {
          const int cc = 2 * c + uu;  // f16 chunk of the row: column block cc / 8
          *reinterpret_cast<uint4*>(dst + (cc >> 3) * C::kSlotCBBytes + (((cc & 7) ^ sw) << 4)) =
              make_uint4(hh[4 * uu], hh[4 * uu + 1], hh[4 * uu + 2], hh[4 * uu + 3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[sl]);
    }
  } else {
    // ======================================================== softmax warps (thread = row)
    const int r = 32 * warp + lane;
    // the row's token within the tile and head within the group (rows token * G + head)
    const int tl = r / G;
    const bool rv = r < TQ * G && tl <= t_last - t_first && q0 + t_first + tl < p.total_q;
    const int i_q = t_first + (rv ? tl : 0);
    const int h = g * G + r % G;
    const int pos = ctx + i_q;
    const int lo_r = p.window_left >= 0 ? max(0, pos - p.window_left) : 0;
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
    // fp8: the per-tensor k_scale joins the score scale, v_scale the output (per-token
    // scales are already in the f16 tiles)
    const bool tok8 = F8 && p.k_scale_tok != nullptr;
    const float kq = F8 && !tok8 ? p.scale * __ldg(p.kv_scale) : p.scale;
    const float v_mul = F8 && !tok8 ? __ldg(p.kv_scale + 1) : 1.f;
    const float c = FEAT ? kLog2e : kq * kLog2e;
    const bool sink = p.sinks != nullptr && z == 0 && rv;
    float m_used = sink ? __ldg(p.sinks + h) * kLog2e : -INFINITY;
    float l = sink ? 1.f : 0.f;
    const uint32_t lane_off = (32u * warp) << 16;
    const uint32_t tOr = tO + lane_off;
    bool ok = true;

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

    for (int j = 0; j < nt; ++j) {
      const int bb = j & 1;
      if (!pf_wait_warp(&s_full[bb], (j >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tS = tmem + bb * BN + lane_off;
      const int k0 = ks + j * BN;
      const bool need_mask = k0 < lomax || k0 + BN - 1 > pmin || k0 + BN > ke;

      // ---- pass 1: row max; transformed / masked scores written back over S
      const bool rewrite = FEAT || need_mask;
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 64) {
        uint32_t ra[32], rb[32];
        tmem_ld32(tS + c0, ra);
        tmem_ld32(tS + c0 + 32, rb);
        tmem_ld_wait();
        if (rewrite) {
          const float ab = FEAT ? slope * static_cast<float>(k0 + c0 - ctx) : 0.f;
          if (need_mask) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              ra[e] = __float_as_uint(score(__uint_as_float(ra[e]), k0 + c0 + e, ab, e, std::true_type{}));
              rb[e] = __float_as_uint(score(__uint_as_float(rb[e]), k0 + c0 + 32 + e, ab, 32 + e, std::true_type{}));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              ra[e] = __float_as_uint(score(__uint_as_float(ra[e]), k0 + c0 + e, ab, e, std::false_type{}));
              rb[e] = __float_as_uint(score(__uint_as_float(rb[e]), k0 + c0 + 32 + e, ab, 32 + e, std::false_type{}));
            }
          }
          tmem_st32(tS + c0, ra);
          tmem_st32(tS + c0 + 32, rb);
        }
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          mx0 = fmax3(mx0, __uint_as_float(ra[e]), __uint_as_float(ra[e + 1]));
          mx1 = fmax3(mx1, __uint_as_float(rb[e]), __uint_as_float(rb[e + 1]));
        }
      }
      if (rewrite) tmem_st_wait();
      const float mx = fmaxf(mx0, mx1) * c;
      float alpha = 1.f;
      const bool grow = mx > m_used + 8.f || (m_used == -INFINITY && mx > -INFINITY);
      if (grow) {
        alpha = m_used == -INFINITY ? 0.f : fast_exp2(m_used - mx);
        m_used = mx;
      }
      const float m_use = m_used == -INFINITY ? 0.f : m_used;
      // O holds P.V of every step up to j-2 (the commit of S_j covers them); P.V_{j-1}
      // may still run: wait for it before rescaling
      if (j >= 1 && __any_sync(0xffffffffu, grow)) {
        if (!pf_wait_warp(pv_done, (j - 1) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ro[32];
          tmem_ld32(tOr + c0, ro);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) ro[e] = __float_as_uint(__uint_as_float(ro[e]) * alpha);
          tmem_st32(tOr + c0, ro);
        }
      }
      const float pmax = mx == -INFINITY ? 0.f : fast_exp2(mx - m_use);
      // The tile's P carries a low part when any of its rows needs one: every warp of the
      // tile then writes both parts, otherwise only the high part (the MMA reads the
      // same flag).  The tile's four warps agree on it through an mbarrier.
      bool tile_lo = false;
      if constexpr (BF16) {
        if (__any_sync(0xffffffffu, pmax * 63.f > l * alpha) && lane == 0)
          lo_flag[bb] = j + 1;
        __syncwarp();
        if (lane == 0) mbar_arrive(lo_bar);
        if (!pf_wait_warp(lo_bar, j & 1, abort_flag, p.status)) { ok = false; break; }
        tile_lo = lo_flag[bb] == j + 1;
      }

      // ---- pass 2: P = 2^(c s - m) over S, 32 keys at a time (16 columns of high part,
      // then, when the tile needs it, 16 of bf16 remainder)
      const float2 cc = make_float2(c, c), mm = make_float2(-m_use, -m_use);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(tS + c0, rr);
        tmem_ld_wait();
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
        if (tile_lo) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint32_t hw = pack_bf16(xv[2 * e], xv[2 * e + 1]);
            rr[e] = hw;
            const float2 rem = __fadd2_rn(make_float2(xv[2 * e], xv[2 * e + 1]),
                                          make_float2(-bf16_lo(hw), -bf16_hi(hw)));
            rr[16 + e] = pack_bf16(rem.x, rem.y);
          }
          tmem_st32(tS + c0, rr);
        } else {
          uint32_t hw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            hw[e] = BF16 ? pack_bf16(xv[2 * e], xv[2 * e + 1]) : pack_f16(xv[2 * e], xv[2 * e + 1]);
          tmem_st16(tS + c0, hw);
        }
      }
      l = l * alpha + ((acc0.x + acc0.y) + (acc1.x + acc1.y));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[bb]);
    }

    // ---- epilogue: P.V_{nt-2} and P.V_{nt-1} done, then O / l or the partition's state
    if (ok && nt >= 2) ok = pf_wait_warp(pv_done, (nt - 2) & 1, abort_flag, p.status);
    if (ok && nt >= 1) ok = pf_wait_warp(pv_done, (nt - 1) & 1, abort_flag, p.status);
    tc_fence_after();
    if (ok) {
      const size_t orow = static_cast<size_t>(q0 + i_q) * p.hq + h;
      const size_t n_part = static_cast<size_t>(p.n_part);
      const float inv = l > 0.f ? v_mul / l : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t rr[32];
        if (nt > 0) {
          tmem_ld32(tOr + c0, rr);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = 0u;
        }
        if (!rv) continue;
        if (n_part == 1) {
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
        } else {
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
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMma) tmem_dealloc(tmem, C::kTmemCols);
}

template <int D, bool BF16, bool FEAT, bool F8 = false>
cudaError_t launch_prefill_wide_t(const PrefillParams& pp, dim3 grid, cudaStream_t stream) {
  using C = PrefillWideCfg<D, F8>;
  auto kern = ua_prefill_wide_kernel<D, BF16, FEAT, F8>;
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

template <int D>
cudaError_t launch_prefill_wide_dispatch(const PrefillParams& pp, dim3 grid, int kv, bool feat,
                                         cudaStream_t s) {
  if (kv == KV_BF16)
    return feat ? launch_prefill_wide_t<D, true, true>(pp, grid, s)
                : launch_prefill_wide_t<D, true, false>(pp, grid, s);
  if (kv == KV_F16)
    return feat ? launch_prefill_wide_t<D, false, true>(pp, grid, s)
                : launch_prefill_wide_t<D, false, false>(pp, grid, s);
  if (kv == KV_E4M3)
    return feat ? launch_prefill_wide_t<D, false, true, true>(pp, grid, s)
                : launch_prefill_wide_t<D, false, false, true>(pp, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace ua
