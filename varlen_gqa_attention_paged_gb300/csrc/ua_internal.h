// ua_internal.h -- definitions shared by the host dispatcher and the kernels of libua.so.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace ua {

enum KvKind { KV_F16 = 0, KV_BF16 = 1, KV_E4M3 = 2 };

// Bits of the device status word (OR-ed by kernels, read by ua_device_status).
enum : unsigned { DEV_BAD_BLOCK = 1u, DEV_TIMEOUT = 2u, DEV_BAD_SHAPE = 4u };

// Everything one launch of the attention tile kernel needs (passed by value).
struct AttnParams {
  const void* q;                // [total_q, hq, D]
  const void* k;                // [num_blocks, block_size, hkv, D]
  const void* v;
  void* out;                    // [total_q, hq, D]          (n_part == 1)
  const int32_t* cu_seqlens_q;  // [num_seqs + 1]
  const int32_t* seq_lens_k;    // [num_seqs]
  const int32_t* block_table;   // [num_seqs, max_blocks_per_seq]
  const float* alibi;           // [hq] or null
  const float* qq_bias;         // [*, qq_stride] or null
  const float* sinks;           // [hq] or null
  const float* kv_scale;        // {k_scale, v_scale} (fp8 cache) or null
  // fp8 per-token scales over (block, slot, kv-head) with element strides, or null (the
  // decode tile kernel reads them; kv_scale is then unused)
  const float* k_scale_tok;
  const float* v_scale_tok;
  long long k_scale_stride[3];
  long long v_scale_stride[3];
  float* ws_m;                  // [total_q, hq, n_part]     (n_part > 1)
  float* ws_l;                  // [total_q, hq, n_part]
  float* ws_acc;                // [total_q, hq, n_part, D]
  unsigned int* status;         // device status word
  int num_seqs, total_q, max_seqlen_q, max_blocks_per_seq, num_blocks, block_size;
  int hq, hkv, group;
  int qq_stride, window_left, n_part;
  int slot_per_seq;             // 1: grid slot x is sequence x (every sequence fits one q-block)
  int cluster_merge;            // 1: the n_part partitions (grid z) of a slot form one cluster
                                //    and merge through distributed shared memory
  int q_dtype, out_dtype;
  float scale, softcap;
};

// Tile-kernel launch argument: the attention parameters plus the TMA tensor maps of the
// K and V caches, each viewed as a 3-D tensor [num_blocks * block_size][H_kv][D]
// (used when block_size % 16 == 0; boxes of 16 cache rows x one column block).
struct TileParams {
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  AttnParams p;
};

// Tensor-memory prefill kernel launch argument: tensor maps of q (viewed as [total_q][H_q][D],
// box 64 elements x G heads x tq tokens, so a tile's row token * G + head) and of the two
// caches, the attention parameters, and tq = query tokens per 128-row q tile
// (floor(128 / G)); a CTA owns 1 or 2 such tiles of consecutive tokens.
struct PrefillParams {
  CUtensorMap tmap_q;
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  AttnParams p;
  int tq;
};

// The LSE-merge of split partitions (one output row per query token x head).
struct MergeParams {
  const float* ws_m;
  const float* ws_l;
  const float* ws_acc;
  void* out;
  int rows;        // total_q * hq
  int n_part;
  int head_dim;
  int out_dtype;
};

// Rows (query token x head of one kv group) per CTA of the tile kernel.
// rows of one q-block (kernel 2, the key-major decode tile: 8)
constexpr int tile_block_m(int wm) { return wm == 2 ? 8 : 16 * wm; }

cudaError_t launch_tile_d64(const TileParams& tp, dim3 grid, int wm, int kv, bool feat, bool tma,
                            int cluster_y, int cluster_z, cudaStream_t s);
cudaError_t launch_tile_d128(const TileParams& tp, dim3 grid, int wm, int kv, bool feat, bool tma,
                             int cluster_y, int cluster_z, cudaStream_t s);
cudaError_t launch_tile_d256(const TileParams& tp, dim3 grid, int wm, int kv, bool feat, bool tma,
                             int cluster_y, int cluster_z, cudaStream_t s);
// key-major decode tile (head_dim 64, 128; TMA page boxes; at most 8 rows per kv-head), with
// four consumer warps (64-key stages, three CTAs per SM) or eight (128-key stages, one CTA
// per SM, for small grids)
cudaError_t launch_decode_w4_d64(const TileParams& tp, dim3 grid, int kv, bool feat,
                                 int cluster_y, int cluster_z, cudaStream_t s);
cudaError_t launch_decode_w4_d128(const TileParams& tp, dim3 grid, int kv, bool feat,
                                  int cluster_y, int cluster_z, cudaStream_t s);
cudaError_t launch_decode_w8_d64(const TileParams& tp, dim3 grid, int kv, bool feat,
                                 int cluster_y, int cluster_z, cudaStream_t s);
cudaError_t launch_decode_w8_d128(const TileParams& tp, dim3 grid, int kv, bool feat,
                                  int cluster_y, int cluster_z, cudaStream_t s);
// the same tile with two kv-heads per CTA (fp8 caches, at most 4 rows per kv-head; tensor
// maps over the view [H_kv][rows][D] with boxes of two heads)
cudaError_t launch_decode_pair_d64(const TileParams& tp, dim3 grid, bool feat, int cluster_y,
                                   int cluster_z, cudaStream_t s);
cudaError_t launch_decode_pair_d128(const TileParams& tp, dim3 grid, bool feat, int cluster_y,
                                    int cluster_z, cudaStream_t s);
int decode_cluster_capacity_pair(int head_dim, int cluster_y, int cluster_z);
int decode_pair_ctas_per_sm(int head_dim);
// resident CTAs per SM of the four-warp decode tile
int decode_ctas_per_sm(int head_dim, int kv);
// co-resident clusters of cluster_y x cluster_z decode CTAs (four or, wide, eight consumer
// warps; pair: two kv-heads a CTA) on the current device (-1: unknown); cached per device
int decode_cluster_capacity(int head_dim, int kv, bool wide, bool pair, int cluster_y,
                            int cluster_z);
int decode_cluster_capacity_w8(int head_dim, int kv, int cluster_y, int cluster_z);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t s);
cudaError_t launch_prefill_d64(const PrefillParams& pp, dim3 grid, int kv, bool feat, int nq,
                               cudaStream_t s);
cudaError_t launch_prefill_d128(const PrefillParams& pp, dim3 grid, int kv, bool feat, int nq,
                               cudaStream_t s);
cudaError_t launch_prefill_d256(const PrefillParams& pp, dim3 grid, int kv, bool feat, int nq,
                               cudaStream_t s);

// Plan kernel codes.
enum : int { KERNEL_TILE16 = 1, KERNEL_DEC8 = 2, KERNEL_TILE64 = 4, KERNEL_TC128 = 8, KERNEL_TC256 = 16,
             KERNEL_DEC8W = 32, KERNEL_DEC8P = 64 };

// Resident CTAs per SM of the tile kernel variant for (head_dim, kv dtype, wm).
int tile_ctas_per_sm(int head_dim, int kv, int wm);

}  // namespace ua
