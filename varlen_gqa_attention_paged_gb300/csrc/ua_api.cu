// ua_api.cu -- C ABI of libua.so: argument checks, the dispatcher (2D vs split-KV from
// grid fill and key-walk length), the split workspace, and the kernel launches.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "ua.h"
#include "ua_internal.h"

namespace {

__device__ unsigned int g_device_status = 0;

// Keys per split partition below which splitting a q-block's walk does not pay: the
// partition must amortise its prologue and the extra merge traffic.
constexpr int kMinPartitionKeys = 256;
constexpr int kMaxPartitions = 128;

int device_sm_count(int* out) {
  static std::mutex mu;
  static std::map<int, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it == cache.end()) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return UA_ERR_CUDA;
    it = cache.emplace(dev, n).first;
  }
  *out = it->second;
  return UA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Recently encoded tensor maps, keyed by everything that goes into one (base address,
// element type, extents, box): a steady stream of calls on the same cache and query buffers
// reuses its maps instead of encoding them again.  Small, round-robin replacement.
struct MapKey {
  const void* base;
  int kind, dtype, d, heads, rows, box_y, box_z;
  bool operator==(const MapKey& o) const {
    return base == o.base && kind == o.kind && dtype == o.dtype && d == o.d && heads == o.heads &&
           rows == o.rows && box_y == o.box_y && box_z == o.box_z;
  }
};

class MapCache {
 public:
  bool find(const MapKey& k, CUtensorMap* out) {
    std::lock_guard<std::mutex> lock(mu_);
    for (int i = 0; i < used_; ++i)
      if (keys_[i] == k) {
        *out = maps_[i];
        return true;
      }
    return false;
  }
  void put(const MapKey& k, const CUtensorMap& m) {
    std::lock_guard<std::mutex> lock(mu_);
    const int i = used_ < kSize ? used_++ : (next_++ % kSize);
    keys_[i] = k;
    maps_[i] = m;
  }

 private:
  static constexpr int kSize = 32;
  std::mutex mu_;
  MapKey keys_[kSize];
  CUtensorMap maps_[kSize];
  int used_ = 0, next_ = 0;
};

MapCache& map_cache() {
  static MapCache* c = new MapCache();  // never destroyed
  return *c;
}

// q [total_q][H_q][D] as a 3-D TMA tensor (dims d, head, token); one box is the 64-element
// column block `x` of G heads x tq tokens, written as G*tq rows of 128 bytes (128-byte
// swizzle), row token * G + head: the rows of a short q-block (a decode token's G heads)
// sit together in the first lane quarters, and the warps of the others have no row.  (A
// head-major view, rows head * tq + token, spread them over every quarter instead: with
// four softmax warps a quarter it measured slower, 21.9 against 21.5 us on the mixed batch
// and 1.1 % on the d256 prefill.)
bool encode_q_map(CUtensorMap* map, const void* q, int q_dtype, int total_q, int hq, int d,
                  int group, int tq) {
  const MapKey key{q, 0, q_dtype, d, hq, total_q, group, tq};
  if (map_cache().find(key, map)) return true;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t tok_stride = static_cast<cuuint64_t>(d) * 2 * hq;
  const cuuint64_t head_stride = static_cast<cuuint64_t>(d) * 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hq),
                              static_cast<cuuint64_t>(total_q)};
  const cuuint64_t strides[2] = {head_stride, tok_stride};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tq)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r =
      enc(map, q_dtype == UA_DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
          3, const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  map_cache().put(key, *map);
  return true;
}

// A paged cache [num_blocks * block_size][H_kv][D] as a 3-D TMA tensor; one box is 16
// cache rows of one kv-head and one column block (128 bytes, swizzled; 64-byte rows
// unswizzled).  Rows past the tensor read as zero.  With heads_per_box > 1 the view is
// [H_kv][rows][D] (head outermost) and a box is 16 rows of heads_per_box consecutive
// kv-heads, landing head by head.
bool encode_cache_map(CUtensorMap* map, const void* base, int kv_dtype, int num_blocks,
                      int block_size, int hkv, int d, int heads_per_box = 1) {
  const MapKey key{base, 1, kv_dtype, d, hkv, num_blocks, block_size, heads_per_box};
  if (map_cache().find(key, map)) return true;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const int esz = kv_dtype == UA_DT_F8E4M3 ? 1 : 2;
  const int row_bytes = d * esz;
  const int cbw = row_bytes >= 128 ? 128 : row_bytes;
  const CUtensorMapDataType dt = kv_dtype == UA_DT_F8E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : kv_dtype == UA_DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t rows = static_cast<cuuint64_t>(num_blocks) * block_size;
  const cuuint64_t head_stride = static_cast<cuuint64_t>(row_bytes);
  const cuuint64_t row_stride = static_cast<cuuint64_t>(row_bytes) * hkv;
  const bool head_outer = heads_per_box > 1;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d),
                              head_outer ? rows : static_cast<cuuint64_t>(hkv),
                              head_outer ? static_cast<cuuint64_t>(hkv) : rows};
  const cuuint64_t strides[2] = {head_outer ? row_stride : head_stride,
                                 head_outer ? head_stride : row_stride};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(cbw / esz),
                             head_outer ? 16u : 1u,
                             head_outer ? static_cast<cuuint32_t>(heads_per_box) : 16u};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         cbw == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  map_cache().put(key, *map);
  return true;
}

// Device address of the status word on the current device (looked up once per device; the
// address does not survive cudaDeviceReset of that device).
int status_word(unsigned int** out) {
  static std::mutex mu;
  static std::map<int, unsigned int*> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it == cache.end()) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess || ptr == nullptr)
      return UA_ERR_CUDA;
    it = cache.emplace(dev, static_cast<unsigned int*>(ptr)).first;
  }
  *out = it->second;
  return UA_OK;
}

int check_sizes(const ua_shape_t* sh, int block_size, int hq, int hkv, int d, int kv_dtype,
                int backend) {
  if (sh == nullptr) return UA_ERR_INVALID_ARG;
  if (sh->num_seqs < 0 || sh->total_q < 0 || sh->max_seqlen_q < 0 || sh->max_seqlen_k < 0 ||
      sh->max_blocks_per_seq < 0 || sh->num_blocks < 0 || sh->num_splits < 0)
    return UA_ERR_INVALID_ARG;
  if (block_size < 1 || hq < 1 || hkv < 1 || hq % hkv != 0) return UA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return UA_ERR_INVALID_ARG;
  if (kv_dtype != UA_DT_F16 && kv_dtype != UA_DT_BF16 && kv_dtype != UA_DT_F8E4M3)
    return UA_ERR_INVALID_ARG;
  if (sh->q_dtype != UA_DT_F16 && sh->q_dtype != UA_DT_BF16) return UA_ERR_INVALID_ARG;
  if (sh->out_dtype != UA_DT_F16 && sh->out_dtype != UA_DT_BF16 && sh->out_dtype != UA_DT_F32)
    return UA_ERR_INVALID_ARG;
  if (backend != UA_BACKEND_AUTO && backend != UA_BACKEND_2D && backend != UA_BACKEND_SPLIT)
    return UA_ERR_INVALID_ARG;
  if (kv_dtype != UA_DT_F8E4M3 && sh->q_dtype != kv_dtype) return UA_ERR_UNSUPPORTED;
  return UA_OK;
}

// The dispatcher.  Split the key walk (UA_BACKEND_AUTO) only when the 2D grid leaves
// part of one wave of SMs idle and the walk spans at least two minimum partitions;
// then into as many partitions as still fit in that one wave (at least two): a
// second, partly filled wave costs more than the extra parallelism gives back.
//
// Kernel: decode calls with at most 8 rows per kv-head, head_dim <= 128 and page-sized
// TMA boxes take the key-major decode tile (keys on the MMA's M side, rows on N); other
// decode-shaped calls (every sequence's rows fit 16) take the warp-MMA tile kernel with
// 16-row q-blocks; other calls with 16 | block_size take the tensor-memory kernels with
// 128-row q tiles (floor(128 / G) tokens x G heads; fp8 caches dequantised to f16 tiles in
// shared memory), two tiles per CTA for head_dim <= 128 when that grid still fills the
// device; the rest (block sizes not a multiple of 16) take the tile kernel with 64-row
// q-blocks.  A decode grid of at most one CTA per SM takes the eight-warp decode tile.
bool is_tc(int kernel) { return kernel == ua::KERNEL_TC128 || kernel == ua::KERNEL_TC256; }

void make_plan(const ua_shape_t* sh, int block_size, int hq, int hkv, int d, int window_left,
               int kv_dtype, int backend, int num_sms, bool allow_tc, bool allow_dec,
               bool query_device, ua_plan_t* pl) {
  const int group = hq / hkv;
  const long long rows_max = static_cast<long long>(sh->max_seqlen_q) * group;
  const bool tc = allow_tc && rows_max > 16 && group <= 128 && block_size % 16 == 0;
  // decode with at most 8 rows per kv-head: the key-major decode tile (page boxes)
  const bool dec = allow_dec && !tc && rows_max <= 8 && d <= 128 && block_size % 16 == 0 &&
                   static_cast<long long>(sh->num_blocks) * block_size + 16 <= INT32_MAX;
  // fp8 decode with at most 4 rows per kv-head and per-tensor scales: two kv-heads a CTA
  // (their q-blocks fill the tile's 8 columns; one page box carries both heads' rows)
  const bool pair = dec && kv_dtype == UA_DT_F8E4M3 && rows_max <= 4 && hkv % 2 == 0 &&
                    sh->k_scale_tok == nullptr;
  const int gy = pair ? hkv / 2 : hkv;  // CTAs of one slot (grid y)
  const int wm = dec ? ua::KERNEL_DEC8 : rows_max <= 16 ? 1 : 4;
  const int tq = tc ? 128 / group : 0;               // tokens per 128-row tensor-memory tile
  // two tiles per CTA (sharing every K/V tile) where their tensor memory fits and the
  // grid still fills the device
  const int nq = tc && d <= 128 &&
                         (static_cast<long long>(sh->total_q) / (2 * tq) + sh->num_seqs) * hkv >= num_sms
                     ? 2
                     : 1;
  const int bm = tc ? nq * tq * group : ua::tile_block_m(wm);
  // every sequence fits one q-block: slot x is sequence x; else the monotone slot layout
  const bool per_seq = !tc && rows_max <= bm;
  const long long slots =
      tc ? static_cast<long long>(sh->total_q) / (nq * tq) + sh->num_seqs
         : per_seq ? sh->num_seqs
                   : static_cast<long long>(sh->total_q) * group / bm + sh->num_seqs;
  const long long active = per_seq ? std::min<long long>(sh->num_seqs, sh->total_q) : slots;
  const long long base = std::max<long long>(1, active * gy);
  // Longest key walk of one q-block: a window bounds it, otherwise the longest sequence.
  long long walk = sh->max_seqlen_k;
  if (window_left >= 0)
    walk = std::min<long long>(walk, static_cast<long long>(window_left) + 1 + (bm + group - 1) / group);
  const long long wave =
      static_cast<long long>(num_sms) *
      (tc    ? 1
       : pair ? ua::decode_pair_ctas_per_sm(d)
       : dec  ? ua::decode_ctas_per_sm(d, kv_dtype)
              : ua::tile_ctas_per_sm(d, kv_dtype, wm));
  const long long by_walk = std::max<long long>(1, walk / kMinPartitionKeys);
  const long long fit = std::max<long long>(2, std::min(wave / base, by_walk));
  int n_part = 1;
  bool fitted = false;  // n_part chosen here rather than by the caller
  if (backend == UA_BACKEND_SPLIT) {
    n_part = sh->num_splits > 0 ? sh->num_splits : static_cast<int>(fit);
    fitted = sh->num_splits <= 0;
  } else if (backend == UA_BACKEND_AUTO) {
    if (base < wave && walk >= 2LL * kMinPartitionKeys) {
      n_part = static_cast<int>(fit);
      fitted = true;
    }
  }
  n_part = std::min(n_part, kMaxPartitions);
  // Decode-shaped CTAs of one slot read the same cache pages for different kv-heads and
  // are launched as one cluster (cluster_y kv-heads) so they are scheduled together; a
  // split's partitions join that cluster (cluster_z = n_part; at most 8 CTAs, the portable
  // size, or up to 16 partitions alone) and merge through distributed shared memory: no
  // merge kernel, no workspace.
  auto cluster_shape = [&](int np, int& cy, int& cz) {
    cy = 1;
    if (!tc && wm != 4)
      for (int c = 8; c > 1; c >>= 1)
        if (gy % c == 0) {
          cy = c;
          break;
        }
    cz = 1;
    if (!tc && wm != 4 && np > 1 && np <= 16) {
      cz = np;
      while (cy * cz > (cz > 8 ? 16 : 8)) cy >>= 1;
    }
  };
  // A cluster's CTAs must be resident together, inside one GPU processing cluster, which
  // leaves fewer co-resident CTAs than the SMs' slots; a fitted partition count shrinks
  // until every cluster of the grid fits one wave (the decode tile asks the device; else
  // 90 % of the slots for clusters of three CTAs or more).
  if (fitted && !tc && wm != 4) {
    for (; n_part > 2; --n_part) {
      int cy, cz;
      cluster_shape(n_part, cy, cz);
      const int c = cy * cz;
      if (c <= 1) break;
      long long cap = -1;
      if (dec && query_device) cap = ua::decode_cluster_capacity(d, kv_dtype, false, pair, cy, cz);
      if (cap < 0) cap = c <= 2 ? wave / c : (wave * 9 / 10) / c;
      if (slots * (gy / cy) <= cap) break;
    }
  }
  // A decode grid of at most one CTA per SM runs the eight-warp decode tile (128-key
  // stages): twice the consumer warps on each CTA's key walk, half the pipeline stages,
  // when its clusters (one CTA per SM) are all resident together.
  bool wide = false;
  if (dec && !pair && slots * hkv * n_part <= num_sms) {
    int cy, cz;
    cluster_shape(n_part, cy, cz);
    wide = true;
    if (cy * cz > 1) {
      long long cap = -1;
      if (query_device) cap = ua::decode_cluster_capacity(d, kv_dtype, true, false, cy, cz);
      if (cap < 0) cap = (static_cast<long long>(num_sms) * 9 / 10) / (cy * cz);
      wide = slots * (hkv / cy) <= cap;
    }
  }
  pl->path = n_part > 1 ? UA_PATH_SPLIT : UA_PATH_2D;
  pl->kernel = tc     ? (nq == 2 ? ua::KERNEL_TC256 : ua::KERNEL_TC128)
               : pair ? ua::KERNEL_DEC8P
               : wide ? ua::KERNEL_DEC8W
                      : wm;
  pl->block_m = bm;
  pl->n_part = n_part;
  pl->grid_x = static_cast<int32_t>(slots);
  pl->grid_y = gy;
  pl->grid_z = n_part;
  pl->num_sms = num_sms;
  int cy, cz;
  cluster_shape(n_part, cy, cz);
  pl->cluster_y = cy;
  pl->cluster_z = cz;
  pl->slot_per_seq = per_seq ? 1 : 0;
  pl->workspace_bytes = 0;
  if (n_part > 1 && cz == 1) {
    const size_t rows = static_cast<size_t>(sh->total_q) * hq * n_part;
    // m and l, then acc; each piece rounded to 256 bytes
    const size_t ml = ((rows * sizeof(float) + 255) / 256) * 256;
    const size_t acc = ((rows * d * sizeof(float) + 255) / 256) * 256;
    pl->workspace_bytes = 2 * ml + acc;
  }
}

// Library-owned split workspace: one grow-only buffer per (device, stream).  A buffer
// that is replaced stays allocated, because earlier work (or a captured graph) on that
// stream may still use it.
struct WorkspacePool {
  std::mutex mu;
  std::map<std::pair<int, void*>, std::pair<void*, size_t>> live;
  std::vector<void*> retired;
};

WorkspacePool& pool() {
  static WorkspacePool* p = new WorkspacePool();  // never destroyed: kernels may outlive exit order
  return *p;
}

int library_workspace(void* stream, size_t bytes, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return UA_ERR_CUDA;
  WorkspacePool& wp = pool();
  std::lock_guard<std::mutex> lock(wp.mu);
  auto key = std::make_pair(dev, stream);
  auto it = wp.live.find(key);
  if (it != wp.live.end() && it->second.second >= bytes) {
    *out = it->second.first;
    return UA_OK;
  }
  size_t grow = 1 << 20;
  while (grow < bytes) grow <<= 1;
  void* ptr = nullptr;
  if (cudaMalloc(&ptr, grow) != cudaSuccess) return UA_ERR_CUDA;
  if (it != wp.live.end()) {
    wp.retired.push_back(it->second.first);
    it->second = std::make_pair(ptr, grow);
  } else {
    wp.live.emplace(key, std::make_pair(ptr, grow));
  }
  *out = ptr;
  return UA_OK;
}

int enqueue(const void* q, const void* k_cache, const void* v_cache, void* out,
            const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, const int32_t* block_table,
            int block_size, int hq, int hkv, int d, float scale, float softcap, int window_left,
            const float* alibi, const float* qq_bias, const float* sinks, int kv_dtype,
            const float* kv_scale, int backend, void* stream, const ua_shape_t* sh) {
  int rc = check_sizes(sh, block_size, hq, hkv, d, kv_dtype, backend);
  if (rc != UA_OK) return rc;
  if (sh->total_q == 0 || sh->num_seqs == 0) return UA_OK;
  if (!q || !k_cache || !v_cache || !out || !cu_seqlens_q || !seq_lens_k || !block_table)
    return UA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return UA_ERR_INVALID_ARG;
  const bool tok_scales = kv_dtype == UA_DT_F8E4M3 && sh->k_scale_tok != nullptr;
  if (kv_dtype == UA_DT_F8E4M3) {
    if ((sh->k_scale_tok == nullptr) != (sh->v_scale_tok == nullptr)) return UA_ERR_INVALID_ARG;
    if (!tok_scales && kv_scale == nullptr) return UA_ERR_INVALID_ARG;
    if (tok_scales) {
      if ((reinterpret_cast<uintptr_t>(sh->k_scale_tok) & 3) ||
          (reinterpret_cast<uintptr_t>(sh->v_scale_tok) & 3))
        return UA_ERR_INVALID_ARG;
      for (int i = 0; i < 3; ++i)
        if (sh->k_scale_stride[i] < 0 || sh->v_scale_stride[i] < 0) return UA_ERR_INVALID_ARG;
    }
  }
  if (qq_bias != nullptr && sh->qq_bias_stride < std::max(1, sh->max_seqlen_q))
    return UA_ERR_INVALID_ARG;
  if (sh->max_blocks_per_seq < 1 || sh->num_blocks < 1) return UA_ERR_INVALID_ARG;

  int num_sms = 0;
  if ((rc = device_sm_count(&num_sms)) != UA_OK) return rc;
  ua_plan_t pl;
  make_plan(sh, block_size, hq, hkv, d, window_left, kv_dtype, backend, num_sms, true, true, true,
            &pl);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  ua::TileParams tp{};
  ua::AttnParams& p = tp.p;
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.out = out;
  p.cu_seqlens_q = cu_seqlens_q;
  p.seq_lens_k = seq_lens_k;
  p.block_table = block_table;
  p.alibi = alibi;
  p.qq_bias = qq_bias;
  p.sinks = sinks;
  p.kv_scale = kv_scale;
  if (tok_scales) {
    p.k_scale_tok = sh->k_scale_tok;
    p.v_scale_tok = sh->v_scale_tok;
    for (int i = 0; i < 3; ++i) {
      p.k_scale_stride[i] = sh->k_scale_stride[i];
      p.v_scale_stride[i] = sh->v_scale_stride[i];
    }
  }
  p.num_seqs = sh->num_seqs;
  p.total_q = sh->total_q;
  p.max_seqlen_q = sh->max_seqlen_q;
  p.max_blocks_per_seq = sh->max_blocks_per_seq;
  p.num_blocks = sh->num_blocks;
  p.block_size = block_size;
  p.hq = hq;
  p.hkv = hkv;
  p.group = hq / hkv;
  p.qq_stride = sh->qq_bias_stride;
  p.window_left = window_left < 0 ? -1 : window_left;
  p.n_part = pl.n_part;
  p.slot_per_seq = pl.slot_per_seq;
  p.q_dtype = sh->q_dtype;
  p.out_dtype = sh->out_dtype;
  p.scale = scale;
  p.softcap = softcap > 0.f ? softcap : 0.f;
  if ((rc = status_word(&p.status)) != UA_OK) return rc;

  const int kv = kv_dtype == UA_DT_F16 ? ua::KV_F16 : kv_dtype == UA_DT_BF16 ? ua::KV_BF16 : ua::KV_E4M3;
  const bool feat = softcap > 0.f || alibi != nullptr || qq_bias != nullptr;
  // The tensor-memory kernel needs TMA maps of q and both caches; if one cannot be made,
  // the call is planned again for the tile kernel.
  ua::PrefillParams pp{};
  if (is_tc(pl.kernel)) {
    const int group = hq / hkv;
    const bool maps =
        static_cast<long long>(sh->num_blocks) * block_size + 16 <= INT32_MAX &&
        encode_q_map(&pp.tmap_q, q, sh->q_dtype, sh->total_q, hq, d, group, 128 / group) &&
        encode_cache_map(&pp.tmap_k, k_cache, kv_dtype, sh->num_blocks, block_size, hkv, d) &&
        encode_cache_map(&pp.tmap_v, v_cache, kv_dtype, sh->num_blocks, block_size, hkv, d);
    if (!maps) {
      make_plan(sh, block_size, hq, hkv, d, window_left, kv_dtype, backend, num_sms, false, true,
                true, &pl);
      p.n_part = pl.n_part;
    }
    pp.tq = 128 / group;
  }
  // Page-sized TMA boxes need 16 | block_size and row coordinates that fit in int32; the
  // decode tile needs them, else the call is planned again for the tile kernel.
  bool tma = !is_tc(pl.kernel) && block_size % 16 == 0 &&
             static_cast<long long>(sh->num_blocks) * block_size + 16 <= INT32_MAX;
  const int hbox = pl.kernel == ua::KERNEL_DEC8P ? 2 : 1;  // kv-heads per page box
  if (tma)
    tma = encode_cache_map(&tp.tmap_k, k_cache, kv_dtype, sh->num_blocks, block_size, hkv, d,
                           hbox) &&
          encode_cache_map(&tp.tmap_v, v_cache, kv_dtype, sh->num_blocks, block_size, hkv, d,
                           hbox);
  const bool dec_kernel = pl.kernel == ua::KERNEL_DEC8 || pl.kernel == ua::KERNEL_DEC8W ||
                          pl.kernel == ua::KERNEL_DEC8P;
  if (dec_kernel && !tma) {
    make_plan(sh, block_size, hq, hkv, d, window_left, kv_dtype, backend, num_sms, false, false,
              true, &pl);
    p.n_part = pl.n_part;
  }
  // per-token fp8 scales: the decode tile and the tensor-memory kernels read them (the tile
  // kernel, for decode batches of 9 to 16 rows a kv-head or head_dim 256, and for pages
  // not a multiple of 16, does not)
  if (tok_scales && pl.kernel != ua::KERNEL_DEC8 && pl.kernel != ua::KERNEL_DEC8W &&
      !is_tc(pl.kernel))
    return UA_ERR_UNSUPPORTED;
  p.cluster_merge = pl.cluster_z > 1 ? 1 : 0;
  if (pl.n_part > 1 && !p.cluster_merge) {
    void* ws = sh->workspace;
    if (ws != nullptr) {
      if (sh->workspace_bytes < pl.workspace_bytes || !aligned16(ws)) return UA_ERR_WORKSPACE;
    } else if ((rc = library_workspace(stream, pl.workspace_bytes, &ws)) != UA_OK) {
      return rc;
    }
    const size_t rows = static_cast<size_t>(sh->total_q) * hq * pl.n_part;
    const size_t ml = ((rows * sizeof(float) + 255) / 256) * 256;
    p.ws_m = static_cast<float*>(ws);
    p.ws_l = reinterpret_cast<float*>(static_cast<char*>(ws) + ml);
    p.ws_acc = reinterpret_cast<float*>(static_cast<char*>(ws) + 2 * ml);
  }
  const dim3 grid(pl.grid_x, pl.grid_y, pl.grid_z);
  cudaEvent_t* ev = static_cast<cudaEvent_t*>(sh->events);
  if (ev && cudaEventRecord(ev[0], st) != cudaSuccess) return UA_ERR_CUDA;
  cudaError_t err;
  if (is_tc(pl.kernel)) {
    pp.p = p;
    const int nq = pl.kernel == ua::KERNEL_TC256 ? 2 : 1;
    switch (d) {
      case 64: err = ua::launch_prefill_d64(pp, grid, kv, feat, nq, st); break;
      case 128: err = ua::launch_prefill_d128(pp, grid, kv, feat, nq, st); break;
      default: err = ua::launch_prefill_d256(pp, grid, kv, feat, nq, st); break;
    }
  } else if (pl.kernel == ua::KERNEL_DEC8) {
    err = d == 64 ? ua::launch_decode_w4_d64(tp, grid, kv, feat, pl.cluster_y, pl.cluster_z, st)
                  : ua::launch_decode_w4_d128(tp, grid, kv, feat, pl.cluster_y, pl.cluster_z, st);
  } else if (pl.kernel == ua::KERNEL_DEC8P) {
    err = d == 64 ? ua::launch_decode_pair_d64(tp, grid, feat, pl.cluster_y, pl.cluster_z, st)
                  : ua::launch_decode_pair_d128(tp, grid, feat, pl.cluster_y, pl.cluster_z, st);
  } else if (pl.kernel == ua::KERNEL_DEC8W) {
    err = d == 64 ? ua::launch_decode_w8_d64(tp, grid, kv, feat, pl.cluster_y, pl.cluster_z, st)
                  : ua::launch_decode_w8_d128(tp, grid, kv, feat, pl.cluster_y, pl.cluster_z, st);
  } else switch (d) {
    case 64: err = ua::launch_tile_d64(tp, grid, pl.kernel, kv, feat, tma, pl.cluster_y, pl.cluster_z, st); break;
    case 128: err = ua::launch_tile_d128(tp, grid, pl.kernel, kv, feat, tma, pl.cluster_y, pl.cluster_z, st); break;
    default: err = ua::launch_tile_d256(tp, grid, pl.kernel, kv, feat, tma, pl.cluster_y, pl.cluster_z, st); break;
  }
  if (err != cudaSuccess) return UA_ERR_CUDA;
  if (ev && cudaEventRecord(ev[1], st) != cudaSuccess) return UA_ERR_CUDA;
  if (pl.n_part > 1 && !p.cluster_merge) {
    ua::MergeParams mp{};
    mp.ws_m = p.ws_m;
    mp.ws_l = p.ws_l;
    mp.ws_acc = p.ws_acc;
    mp.out = out;
    mp.rows = sh->total_q * hq;
    mp.n_part = pl.n_part;
    mp.head_dim = d;
    mp.out_dtype = sh->out_dtype;
    if (ua::launch_merge(mp, st) != cudaSuccess) return UA_ERR_CUDA;
  }
  if (ev && cudaEventRecord(ev[2], st) != cudaSuccess) return UA_ERR_CUDA;
  return UA_OK;
}

}  // namespace

extern "C" {

int ua_unified_attention(const void* q, const void* k_cache, const void* v_cache, void* out,
                         const int32_t* cu_seqlens_q, const int32_t* seq_lens_k,
                         const int32_t* block_table, int block_size, int num_q_heads,
                         int num_kv_heads, int head_dim, float scale, float softcap,
                         int window_left, const float* alibi_slopes, const float* qq_bias,
                         const float* sinks, int kv_dtype, const float* kv_scale, int backend,
                         void* stream, const ua_shape_t* shape) {
  try {
    return enqueue(q, k_cache, v_cache, out, cu_seqlens_q, seq_lens_k, block_table, block_size,
                   num_q_heads, num_kv_heads, head_dim, scale, softcap, window_left, alibi_slopes,
                   qq_bias, sinks, kv_dtype, kv_scale, backend, stream, shape);
  } catch (...) {
    return UA_ERR_CUDA;
  }
}

int ua_plan(const ua_shape_t* shape, int block_size, int num_q_heads, int num_kv_heads,
            int head_dim, int window_left, int kv_dtype, int backend, int num_sms,
            ua_plan_t* plan) {
  try {
    if (plan == nullptr) return UA_ERR_INVALID_ARG;
    int rc = check_sizes(shape, block_size, num_q_heads, num_kv_heads, head_dim, kv_dtype, backend);
    if (rc != UA_OK) return rc;
    const bool on_device = num_sms <= 0;  // plan for this device (else host-only sizes)
    if (on_device && (rc = device_sm_count(&num_sms)) != UA_OK) return rc;
    make_plan(shape, block_size, num_q_heads, num_kv_heads, head_dim, window_left, kv_dtype,
              backend, num_sms, true, true, on_device, plan);
    return UA_OK;
  } catch (...) {
    return UA_ERR_CUDA;
  }
}

size_t ua_workspace_bytes(const ua_shape_t* shape, int block_size, int num_q_heads,
                          int num_kv_heads, int head_dim, int window_left, int kv_dtype,
                          int backend) {
  ua_plan_t pl;
  if (ua_plan(shape, block_size, num_q_heads, num_kv_heads, head_dim, window_left, kv_dtype,
              backend, 0, &pl) != UA_OK)
    return 0;
  return pl.workspace_bytes;
}

int ua_device_status(void* stream, int* status) {
  if (status == nullptr) return UA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return UA_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_device_status, sizeof(word)) != cudaSuccess) return UA_ERR_CUDA;
  *status = (word & (ua::DEV_BAD_BLOCK | ua::DEV_BAD_SHAPE)) ? UA_ERR_DEVICE_CHECK
            : (word & ua::DEV_TIMEOUT) ? UA_ERR_TIMEOUT
                                       : UA_OK;
  return UA_OK;
}

int ua_device_status_reset(void* stream) {
  const unsigned int zero = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st) !=
      cudaSuccess)
    return UA_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? UA_OK : UA_ERR_CUDA;
}

const char* ua_status_string(int status) {
  switch (status) {
    case UA_OK: return "ok";
    case UA_ERR_INVALID_ARG: return "invalid argument";
    case UA_ERR_UNSUPPORTED: return "unsupported combination";
    case UA_ERR_CUDA: return "CUDA runtime error";
    case UA_ERR_WORKSPACE: return "workspace too small";
    case UA_ERR_DEVICE_CHECK: return "device check failed: block id outside the cache";
    case UA_ERR_TIMEOUT: return "device wait timed out";
    case UA_ERR_SCRATCH_LIMIT:
      return "call needs more scratch than the fixed array of ua_unified_attention_noalloc";
    default: return "unknown status";
  }
}

int ua_version(void) { return UA_VERSION; }

}  // extern "C"
