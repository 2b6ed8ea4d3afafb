// ua_prefill.cuh -- the tensor-memory attention kernel of libua.so for prefill-shaped
// q-blocks with head_dim 256 (included by ua_prefill_d256.cu), and the helpers it shares
// with the head_dim <= 128 kernel of ua_prefill_tm.cuh.  At head_dim 256 two 128-key K/V
// tiles do not fit in shared memory beside Q, so this kernel walks 64-key tiles and keeps P
// in shared memory, with S double-buffered in tensor memory.
//
// One CTA owns (q-block, kv-head g, key partition z).  A q-block is TQ consecutive query
// tokens of one sequence times the G query heads that read kv-head g, packed as
// M = 128 rows of a 5th-generation tensor-core tile (row r = token r / G, head r % G;
// TQ = floor(128 / G)), so the GQA heads of a group share every K/V tile (vllm-rdna PR
// #34 "FA-RDNA2 D=128 prefill", "Change" 1, on tensor cores).  Per key tile of BN keys:
//
//   S = Q K^T    tcgen05.mma (kind::f16, M=128, N=BN, fp32 accumulate) into tensor memory
//   softmax      one thread per row reads its S row from tensor memory, applies scale,
//                softcap, ALiBi, QQ-bias and the causal/window mask, updates the running
//                max and sum in base 2 (the sink is the initial max), and writes
//                P = 2^(s - m) to shared memory as bf16 (high part + remainder) or f16
//   O += P V     tcgen05.mma into tensor memory (V is the MN-major operand as it lands)
//
// S is double-buffered in tensor memory, so the MMA warp computes S of tile j+1 while the
// softmax warps work on tile j.  O is rescaled only when a row's max grows by more than
// 2^8 (the sum and O stay consistent with the max actually used), which keeps tensor
// memory round trips rare.
//
// Warp roles (192 threads):  warps 0..3 softmax + epilogue (thread = row = TMEM lane),
// warp 4 TMA producer (Q once, then K and V pages of 16 keys through the block table into
// two separate rings, 128-byte swizzled: a K slot is refilled as soon as its QK^T is done,
// a V slot once its P.V is done), warp 5 MMA issuer and tensor-memory owner.
#pragma once

#include <atomic>
#include <climits>

#include <cuda.h>

#include "ua_device.cuh"
#include "ua_internal.h"

#include "ua.h"

namespace ua {

template <int D, int NQ>
struct PrefillCfg {
  static constexpr int kBM = 128;                        // MMA rows of one q tile
  static constexpr int kBN = 64;                         // keys per tile
  static constexpr int kCB = D / 64;                     // 128-byte column blocks of a row
  static constexpr int kQBytes = kCB * kBM * 128;        // one q tile
  static constexpr int kKVCB = kBN * 128;                // one column block of a K or V tile
  static constexpr int kTileBytes = kCB * kKVCB;         // one K (or V) tile
  static constexpr int kPCB = kBM * 128;                 // one column block (64 keys) of P
  static constexpr int kPBytes = (kBN / 64) * kPCB;      // P of one q tile (one part)
  static constexpr int kBarBytes = 512;
  // ring depth: as many K and V tiles as fit beside Q and P (at most 4 each)
  static constexpr int kFree = 227 * 1024 - 1024 - kBarBytes - NQ * kQBytes - NQ * 2 * kPBytes;
  static constexpr int kRing = kFree / (2 * kTileBytes) > 4 ? 4 : kFree / (2 * kTileBytes);
  static constexpr int kSmemBytes =
      1024 + NQ * kQBytes + 2 * kRing * kTileBytes + NQ * 2 * kPBytes + kBarBytes;
  static constexpr int kTmemStride = 2 * kBN + D;        // S0, S1, O of one q tile
  static constexpr int kTmemCols = 512;
  static constexpr int kSoftmaxWarps = 4 * NQ;
  static constexpr int kThreads = 32 * kSoftmaxWarps + 64;
  static_assert(NQ * kTmemStride <= kTmemCols, "tensor memory budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kRing >= 2, "at least double-buffered K and V");
};

// Two q tiles per CTA need 2 x (S0, S1, O) columns of tensor memory.
constexpr bool prefill_two_tiles_fit(int d) { return 2 * (2 * 64 + d) <= 512; }

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

template <int D, int NQ, bool BF16, bool FEAT>
__global__ void __launch_bounds__(PrefillCfg<D, NQ>::kThreads, 1)
    ua_prefill_tc_kernel(const __grid_constant__ PrefillParams pp) {
  using C = PrefillCfg<D, NQ>;
  constexpr int BN = C::kBN;
  constexpr int R = C::kRing;
  constexpr int kProducer = C::kSoftmaxWarps, kMma = C::kSoftmaxWarps + 1;
  const AttnParams& p = pp.p;
  grid_dependency_wait();
  grid_launch_dependents();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* const smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* const sQ = smem;                          // NQ q tiles
  uint8_t* const sK = sQ + NQ * C::kQBytes;          // R K tiles
  uint8_t* const sV = sK + R * C::kTileBytes;        // R V tiles
  uint8_t* const sP = sV + R * C::kTileBytes;        // per q tile: P high part, P low part
  uint64_t* const bars = reinterpret_cast<uint64_t*>(sP + NQ * 2 * C::kPBytes);
  uint64_t* const q_full = bars + 0;
  uint64_t* const fin = bars + 1;
  uint64_t* const k_full = bars + 2;            // [R]
  uint64_t* const k_empty = bars + 2 + R;       // [R]
  uint64_t* const v_full = bars + 2 + 2 * R;    // [R]
  uint64_t* const v_empty = bars + 2 + 3 * R;   // [R]
  uint64_t* const tile_bars = bars + 2 + 4 * R; // [NQ][6]: s_full[2], s_free[2], p_full, pv_done
  auto s_full = [&](int qt, int s) { return tile_bars + 6 * qt + s; };
  auto s_free = [&](int qt, int s) { return tile_bars + 6 * qt + 2 + s; };
  auto p_full = [&](int qt) { return tile_bars + 6 * qt + 4; };
  auto pv_done = [&](int qt) { return tile_bars + 6 * qt + 5; };
  uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(tile_bars + 6 * NQ);
  // [NQ][2]: walk step + 1 of the tile's P when its low part matters
  int* const lo_flag = reinterpret_cast<int*>(tmem_holder + 1);
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int z = blockIdx.z;
  const int G = p.group;
  const int TQ = pp.tq;          // tokens of one q tile
  const int TB = NQ * TQ;        // tokens of the CTA's q-block

  // Longest walks first: slots are taken in reverse order.
  const int x = static_cast<int>(gridDim.x - 1 - blockIdx.x);
  const int b = pf_find_seq(p.cu_seqlens_q, p.num_seqs, x, TB);
  const int q0 = __ldg(p.cu_seqlens_q + b);
  const int q_len = __ldg(p.cu_seqlens_q + b + 1) - q0;
  const int kv_len = __ldg(p.seq_lens_k + b);
  const int t_first = (x - (q0 / TB + b)) * TB;  // first token of the block within the sequence
  if (t_first < 0 || t_first >= q_len) return;   // idle slot: uniform for the CTA
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

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(fin, 1);
    for (int i = 0; i < R; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int qt = 0; qt < NQ; ++qt) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(s_full(qt, i), 1);
        mbar_init(s_free(qt, i), 4);
        lo_flag[2 * qt + i] = 0;
      }
      mbar_init(p_full(qt), 4);
      mbar_init(pv_done(qt), 1);
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  volatile int* abort_flag = &s_abort;

  if (warp == kProducer) {
    // ======================================================== TMA producer
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    const int bs = p.block_size;
    const int oob = p.num_blocks * bs;
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, nq_act * C::kCB * TQ * G * 128);
      for (int qt = 0; qt < nq_act; ++qt)
        for (int cb = 0; cb < C::kCB; ++cb)
          tma_load_3d_pf(sQ + qt * C::kQBytes + cb * C::kBM * 128, &pp.tmap_q, 64 * cb, g * G,
                         q0 + t_first + qt * TQ, q_full);
    }
    auto page_row = [&](int j) -> int {
      const int key = ks + j * BN + 16 * lane;
      if (lane >= BN / 16 || key >= ke) return oob;
      const int col = key / bs;
      const int blk = col < p.max_blocks_per_seq ? __ldg(bt + col) : -1;
      if (static_cast<unsigned>(blk) >= static_cast<unsigned>(p.num_blocks)) {
        atomicOr(p.status, DEV_BAD_BLOCK);
        return oob;
      }
      return blk * bs + key % bs;
    };
    int row_next = nt > 0 ? page_row(0) : oob;
    int issued = 0;
    for (int j = 0; j < nt; ++j) {
      const int s = j % R;
      const uint32_t ph = ((j / R) - 1) & 1;  // phase of the release of tile j - R
      const int row = row_next;
      if (j + 1 < nt) row_next = page_row(j + 1);
      if (j >= R && !pf_wait_warp(&k_empty[s], ph, abort_flag, p.status)) break;
      if (lane == 0) mbar_arrive_expect_tx(&k_full[s], C::kTileBytes);
      __syncwarp();
      if (lane < BN / 16)
#pragma unroll
        for (int cb = 0; cb < C::kCB; ++cb)
          tma_load_3d_pf(sK + s * C::kTileBytes + cb * C::kKVCB + lane * 2048, &pp.tmap_k,
                         64 * cb, g, row, &k_full[s]);
      if (j >= R && !pf_wait_warp(&v_empty[s], ph, abort_flag, p.status)) break;
      if (lane == 0) mbar_arrive_expect_tx(&v_full[s], C::kTileBytes);
      __syncwarp();
      if (lane < BN / 16)
#pragma unroll
        for (int cb = 0; cb < C::kCB; ++cb)
          tma_load_3d_pf(sV + s * C::kTileBytes + cb * C::kKVCB + lane * 2048, &pp.tmap_v,
                         64 * cb, g, row, &v_full[s]);
      issued = j + 1;
    }
    // never leave copies in flight into this CTA's shared memory (even after an abort)
    for (int j = max(0, issued - R); j < issued; ++j) {
      mbar_wait_bounded(&k_full[j % R], (j / R) & 1, p.status, DEV_TIMEOUT);
      mbar_wait_bounded(&v_full[j % R], (j / R) & 1, p.status, DEV_TIMEOUT);
    }
    if (lane == 0) mbar_wait_bounded(q_full, 0, p.status, DEV_TIMEOUT);
  } else if (warp == kMma) {
    // ======================================================== MMA issuer
    // Per key tile j: S of every q tile (Q_t K_j^T), then O_t += P_t V_{j-1} of every q
    // tile, so the tensor cores work on one tile while the softmax warps of the other run.
    // The whole warp runs this converged; one elected lane issues each MMA and commit.
    constexpr uint32_t kIdQK = umma_idesc_f16(128, BN, BF16, false);
    constexpr uint32_t kIdPV = umma_idesc_f16(128, D, BF16, true);
    int jb[NQ], je[NQ];
#pragma unroll
    for (int qt = 0; qt < NQ; ++qt) tile_walk(qt, jb[qt], je[qt]);
    bool ok = pf_wait_warp(q_full, 0, abort_flag, p.status);
    auto do_pv = [&](int i) -> bool {
      const int vs_i = i % R;
      if (!pf_wait_warp(&v_full[vs_i], (i / R) & 1, abort_flag, p.status)) return false;
      uint8_t* vs = sV + vs_i * C::kTileBytes;
      // Cache slots at or past kv_len hold no key and may hold anything (NaN included):
      // zero those V rows before the tensor cores multiply them by P = 0.
      const int k0 = ks + i * BN;
      if (k0 + BN > kv_len) {
        const int r_lo = max(0, kv_len - k0), r_hi = min(BN, ((kv_len + 15) & ~15) - k0);
        for (int e = lane; e < (r_hi - r_lo) * C::kCB * 8; e += 32) {
          const int r = r_lo + e / (C::kCB * 8), c = e % (C::kCB * 8);
          *reinterpret_cast<uint4*>(vs + (c / 8) * C::kKVCB + r * 128 + (c % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
#pragma unroll
      for (int qt = 0; qt < NQ; ++qt) {
        if (i < jb[qt] || i >= je[qt]) continue;
        const int n = i - jb[qt];
        if (!pf_wait_warp(p_full(qt), n & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const bool use_lo = BF16 && lo_flag[2 * qt + (n & 1)] == n + 1;
        const uint32_t tO = tmem + qt * C::kTmemStride + 2 * BN;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          if (part == 1 && !use_lo) break;
          const uint32_t pbase = smem_addr(sP + (2 * qt + part) * C::kPBytes);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t ad =
                smem_desc_sw128(pbase + (kk >> 2) * C::kPCB + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(smem_addr(vs) + kk * 16 * 128, C::kKVCB, 1024);
            umma_f16_ss_warp(tO, ad, bd, kIdPV, (n > 0 || kk > 0 || part > 0) ? 1u : 0u);
          }
        }
        umma_commit_warp(pv_done(qt));
      }
      umma_commit_warp(&v_empty[vs_i]);
      return true;
    };
    for (int j = 0; ok && j < nt; ++j) {
      const int ks_j = j % R;
      if (!pf_wait_warp(&k_full[ks_j], (j / R) & 1, abort_flag, p.status)) { ok = false; break; }
#pragma unroll
      for (int qt = 0; qt < NQ; ++qt) {
        if (j < jb[qt] || j >= je[qt]) continue;
        const int n = j - jb[qt], s = n & 1;
        if (n >= 2 && !pf_wait_warp(s_free(qt, s), ((n >> 1) - 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t qb = smem_addr(sQ + qt * C::kQBytes);
        const uint32_t kb = smem_addr(sK + ks_j * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = smem_desc_sw128(qb + (kk >> 2) * C::kBM * 128 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(kb + (kk >> 2) * C::kKVCB + (kk & 3) * 32, 16, 1024);
          umma_f16_ss_warp(tmem + qt * C::kTmemStride + s * BN, ad, bd, kIdQK, kk > 0 ? 1u : 0u);
        }
        umma_commit_warp(s_full(qt, s));
      }
      if (!ok) break;
      umma_commit_warp(&k_empty[ks_j]);
      if (j >= 1 && !do_pv(j - 1)) { ok = false; break; }
    }
    if (ok && nt > 0) do_pv(nt - 1);
    // nothing may still be in flight on the tensor cores when the memory is freed
    umma_commit_warp(fin);
    mbar_wait_bounded(fin, 0, p.status, DEV_TIMEOUT);
  } else {
    // ======================================================== softmax warps (thread = row)
    const int qt = warp >> 2;                              // q tile of this warp
    const int quad = warp & 3;                             // its tensor-memory lane quarter
    const int r = 32 * quad + lane;                        // row within the q tile
    int jb, je;
    tile_walk(qt, jb, je);
    const int n_tiles = je - jb;
    const int tf = t_first + qt * TQ;
    const int tl = r / G;                                  // token within the q tile
    const bool rv = qt < nq_act && r < TQ * G && tf + tl < q_len && q0 + tf + tl < p.total_q;
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
    const float scale_log2 = p.scale * kLog2e;
    const float inv_softcap = p.softcap > 0.f ? 1.f / p.softcap : 0.f;
    float slope = 0.f;
    const float* qq_row = nullptr;
    if constexpr (FEAT) {
      if (p.alibi != nullptr && rv) slope = __ldg(p.alibi + h);
      if (p.qq_bias != nullptr && rv && i_q < p.max_seqlen_q)
        qq_row = p.qq_bias + static_cast<size_t>(i_q) * p.qq_stride;
    }
    const bool sink = p.sinks != nullptr && z == 0 && rv;
    float m_used = sink ? __ldg(p.sinks + h) * kLog2e : -INFINITY;
    float l = sink ? 1.f : 0.f;
    const uint32_t lane_off = (32u * quad) << 16;
    const uint32_t tS0 = tmem + qt * C::kTmemStride + lane_off;
    const uint32_t tO = tS0 + 2 * BN;
    bool ok = true;
    uint8_t* const pw_hi = sP + (2 * qt) * C::kPBytes + r * 128;
    uint8_t* const pw_lo = pw_hi + C::kPBytes;
    bool lo_dirty = true;  // the low P rows of this thread hold something other than zeros

    for (int n = 0; n < n_tiles; ++n) {
      const int s = n & 1;
      if (!pf_wait_warp(s_full(qt, s), (n >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      float x[BN];
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(tS0 + s * BN + c0, rr);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c0 + e] = __uint_as_float(rr[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(qt, s));

      // ---- scores: with no softcap or bias the log2-domain score is c * s with
      // c = scale * log2(e) > 0, so the row max is taken on the raw dot products and the
      // scale is folded into the exponent's FMA; softcap and biases are applied first
      const int k0 = ks + (jb + n) * BN;
      const bool need_mask = k0 < lomax || k0 + BN - 1 > pmin || k0 + BN > ke;
      float c = scale_log2;
      if constexpr (FEAT) {
        c = kLog2e;
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          const int jk = k0 + e;
          float v = x[e] * p.scale;
          if (p.softcap > 0.f) v = p.softcap * fast_tanh(v * inv_softcap);
          v += slope * static_cast<float>(jk - ctx);
          if (qq_row != nullptr && jk >= ctx && jk <= pos) v += __ldg(qq_row + (jk - ctx));
          x[e] = v;
        }
      }
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          const int jk = k0 + e;
          x[e] = (rv && jk >= lo_r && jk <= pos && jk < ke) ? x[e] : -INFINITY;
        }
      }
      float mx0 = x[0], mx1 = x[1];
#pragma unroll
      for (int e = 2; e < BN; e += 2) {
        mx0 = fmaxf(mx0, x[e]);
        mx1 = fmaxf(mx1, x[e + 1]);
      }
      const float mx = fmaxf(mx0, mx1) * c;  // row max in log2 units (-inf stays -inf)
      // ---- running max, used lazily: O and l are rescaled only when the max grows by
      // more than 8 in log2 units (P stays <= 256, far inside the fp32 and P ranges)
      float alpha = 1.f;
      const bool grow = mx > m_used + 8.f || (m_used == -INFINITY && mx > -INFINITY);
      if (grow) {
        alpha = m_used == -INFINITY ? 0.f : fast_exp2(m_used - mx);
        m_used = mx;
      }
      const float m_use = m_used == -INFINITY ? 0.f : m_used;
      // ---- P = 2^(c s - m): one packed FMA per two scores, one ex2 per score
      const float2 cc = make_float2(c, c), mm = make_float2(-m_use, -m_use);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < BN; e += 4) {
        const float2 u = __ffma2_rn(make_float2(x[e], x[e + 1]), cc, mm);
        const float2 w = __ffma2_rn(make_float2(x[e + 2], x[e + 3]), cc, mm);
        x[e] = fast_exp2(u.x);
        x[e + 1] = fast_exp2(u.y);
        x[e + 2] = fast_exp2(w.x);
        x[e + 3] = fast_exp2(w.y);
        acc0 = __fadd2_rn(acc0, make_float2(x[e], x[e + 1]));
        acc1 = __fadd2_rn(acc1, make_float2(x[e + 2], x[e + 3]));
      }
      const float rs = (acc0.x + acc0.y) + (acc1.x + acc1.y);
      const float pmax = mx == -INFINITY ? 0.f : fast_exp2(mx - m_use);  // largest P of the row
      l = l * alpha + rs;
      // the low part of P matters only where one key can still weigh more than 1/64
      const bool need_lo = BF16 && pmax * 64.f > l;

      // ---- P buffer free and O final for step n-1
      if (n >= 1) {
        if (!pf_wait_warp(pv_done(qt), (n - 1) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
      }
      if (n >= 1 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(tO + c0, rr);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
          tmem_st32(tO + c0, rr);
        }
        tmem_st_wait();
      }
      // ---- P rows to shared memory (128-byte swizzled, K-major A operand).  The low
      // part is computed only by warps with a row that needs it; a warp that does not
      // keeps zeros in its low rows (written once), so the MMA may use the low buffer
      // whenever any warp of the tile asks for it.
      const bool warp_lo = BF16 && __any_sync(0xffffffffu, need_lo);
#pragma unroll
      for (int cq = 0; cq < BN / 8; ++cq) {
        uint32_t hi4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float a0 = x[8 * cq + 2 * q], a1 = x[8 * cq + 2 * q + 1];
          hi4[q] = BF16 ? pack_bf16(a0, a1) : pack_f16(a0, a1);
        }
        const uint32_t off = (cq >> 3) * C::kPCB + ((((cq & 7) ^ (r & 7))) << 4);
        *reinterpret_cast<uint4*>(pw_hi + off) = make_uint4(hi4[0], hi4[1], hi4[2], hi4[3]);
        if (BF16 && warp_lo) {
          uint32_t lo4[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 rem = __fadd2_rn(make_float2(x[8 * cq + 2 * q], x[8 * cq + 2 * q + 1]),
                                          make_float2(-bf16_lo(hi4[q]), -bf16_hi(hi4[q])));
            lo4[q] = pack_bf16(rem.x, rem.y);
          }
          *reinterpret_cast<uint4*>(pw_lo + off) = make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
        } else if (BF16 && lo_dirty) {
          *reinterpret_cast<uint4*>(pw_lo + off) = make_uint4(0, 0, 0, 0);
        }
      }
      if (BF16) lo_dirty = warp_lo;
      if (warp_lo && lane == 0) lo_flag[2 * qt + (n & 1)] = n + 1;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(qt));
    }

    // ---- epilogue: O / l for one partition, or the partition's max / sum / O
    if (ok && n_tiles > 0) ok = pf_wait_warp(pv_done(qt), (n_tiles - 1) & 1, abort_flag, p.status);
    tc_fence_after();
    if (ok) {
      const size_t orow = static_cast<size_t>(q0 + i_q) * p.hq + h;
      const size_t n_part = static_cast<size_t>(p.n_part);
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t rr[32];
        if (n_tiles > 0) {
          tmem_ld32(tO + c0, rr);
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
            dst[e] = make_float4(__uint_as_float(rr[4 * e]), __uint_as_float(rr[4 * e + 1]),
                                 __uint_as_float(rr[4 * e + 2]), __uint_as_float(rr[4 * e + 3]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMma) tmem_dealloc(tmem, C::kTmemCols);
}

template <int D, int NQ, bool BF16, bool FEAT>
cudaError_t launch_prefill_t(const PrefillParams& pp, dim3 grid, cudaStream_t stream) {
  using C = PrefillCfg<D, NQ>;
  auto kern = ua_prefill_tc_kernel<D, NQ, BF16, FEAT>;
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
cudaError_t launch_prefill_nq(const PrefillParams& pp, dim3 grid, int kv, bool feat,
                              cudaStream_t s) {
  if (kv == KV_BF16)
    return feat ? launch_prefill_t<D, NQ, true, true>(pp, grid, s)
                : launch_prefill_t<D, NQ, true, false>(pp, grid, s);
  if (kv == KV_F16)
    return feat ? launch_prefill_t<D, NQ, false, true>(pp, grid, s)
                : launch_prefill_t<D, NQ, false, false>(pp, grid, s);
  return cudaErrorInvalidValue;
}

// nq: q tiles of 128 rows per CTA (1, or 2 where two tiles' tensor memory fits: D <= 128).
template <int D>
cudaError_t launch_prefill_dispatch(const PrefillParams& pp, dim3 grid, int kv, bool feat, int nq,
                                    cudaStream_t s) {
  if constexpr (prefill_two_tiles_fit(D)) {
    if (nq == 2) return launch_prefill_nq<D, 2>(pp, grid, kv, feat, s);
  }
  if (nq == 1) return launch_prefill_nq<D, 1>(pp, grid, kv, feat, s);
  return cudaErrorInvalidValue;
}

}  // namespace ua
