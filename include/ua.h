/*
 * ua.h -- C ABI of libua.so: unified paged, variable-length GQA attention for
 * NVIDIA GB300 (sm_103a).
 *
 * One call computes attention for a batch of sequences whose keys and values sit
 * in a paged cache indexed by a block table ("RocKE unified_attention parity &
 * benchmark harness", gfx950 README, "Running" step 1: paged KV cache, block
 * tables, cumulative query lengths, optional sliding window, softcap, sinks, ALiBi
 * slopes, QQ-bias).  The library chooses between two execution paths ("2D": one
 * CTA per q-block x kv-head walks every key; "split": the key range is cut into
 * partitions whose max / sum / partial output are merged, as in the aiter PR #3962
 * "split-K long-context decode for shuffled fp8 SWA", "Changes" -- inside the
 * thread-block cluster of a decode slot's partitions, or by a second kernel).
 *
 * Semantics, for sequence b with q_len = cu_seqlens_q[b+1] - cu_seqlens_q[b],
 * kv_len = seq_lens_k[b] and ctx = kv_len - q_len, query row i (0 <= i < q_len)
 * of head h at position p = ctx + i, kv-head g = h / (num_q_heads / num_kv_heads):
 *   allowed keys   0 <= j < kv_len, j <= p, and p - j <= window_left if window_left >= 0
 *   s_j  = scale * q . K_j                 (fp8 cache: K_j = e4m3 * k_scale)
 *   s_j  = softcap * tanh(s_j / softcap)   if softcap > 0
 *   s_j += alibi_slopes[h] * (j - ctx)     if alibi_slopes != NULL
 *   s_j += qq_bias[i * qq_bias_stride + (j - ctx)]  if qq_bias != NULL and j >= ctx
 *   out  = sum_j e^{s_j} V_j / (e^{sinks[h]} (if sinks != NULL) + sum_j e^{s_j})
 *                                      (fp8 cache: V_j = e4m3 * v_scale; per-token
 *                                       scales, when given, replace k_scale / v_scale
 *                                       key by key: see ua_shape_t)
 * A row with no allowed key (possible only when kv_len < q_len, e.g. a decode slot
 * with kv_len 0) is written as 0.
 *
 * Layouts (all contiguous, row-major, device memory owned by the caller):
 *   q            [total_q, num_q_heads, head_dim]               q_dtype (F16 or BF16)
 *   k_cache      [num_blocks, block_size, num_kv_heads, head_dim] kv_dtype
 *   v_cache      same shape and type as k_cache
 *   out          [total_q, num_q_heads, head_dim]               out_dtype (F16, BF16, F32)
 *   cu_seqlens_q [num_seqs + 1] int32, non-decreasing, cu_seqlens_q[0] = 0
 *   seq_lens_k   [num_seqs] int32
 *   block_table  [num_seqs, max_blocks_per_seq] int32 physical block ids
 *   alibi_slopes [num_q_heads] float32, sinks [num_q_heads] float32
 *   qq_bias      float32 rows of qq_bias_stride elements, at least max_seqlen_q rows;
 *                qq_bias_stride >= max_seqlen_q
 *   kv_scale     float32[2] = {k_scale, v_scale}; required for the fp8 cache only
 *
 * Conventions: every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and never synchronises; the library keeps no pointer to
 * caller memory after the call returns.  Errors are returned as ua_status_t and no
 * C++ exception crosses the ABI.  Per device, the library keeps what it looks up once
 * (the SM count, the device address of its status word, recently encoded tensor maps of
 * the caller's buffers, keyed by address and layout); none of it survives cudaDeviceReset,
 * after which the library must not be called on that device again.
 * Block ids outside [0, num_blocks) are not read:
 * the kernel treats the key as zero and raises UA_ERR_DEVICE_CHECK in the device
 * status word (see ua_device_status).
 */
#ifndef UA_H_
#define UA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define UA_VERSION 100

/* Size of the fixed device scratch array used by ua_unified_attention_noalloc. */
#define UA_NOALLOC_SCRATCH_BYTES (16u << 20)

typedef enum {
  UA_OK = 0,
  UA_ERR_INVALID_ARG = 1,  /* a size, pointer, alignment or enum value is not accepted */
  UA_ERR_UNSUPPORTED = 2,  /* a valid combination this build has no kernel for */
  UA_ERR_CUDA = 3,         /* a CUDA runtime call failed (launch, allocation, query) */
  UA_ERR_WORKSPACE = 4,    /* the caller's workspace is smaller than ua_plan() asks */
  UA_ERR_DEVICE_CHECK = 5, /* a kernel saw a block id outside [0, num_blocks) */
  UA_ERR_TIMEOUT = 6,      /* a kernel gave up waiting on its own copy pipeline */
  UA_ERR_SCRATCH_LIMIT = 7 /* ua_unified_attention_noalloc: the call needs more scratch than
                              its fixed UA_NOALLOC_SCRATCH_BYTES */
} ua_status_t;

typedef enum { UA_DT_F16 = 0, UA_DT_BF16 = 1, UA_DT_F8E4M3 = 2, UA_DT_F32 = 3 } ua_dtype_t;

typedef enum {
  UA_BACKEND_AUTO = 0,  /* dispatcher picks from grid fill and key-walk length */
  UA_BACKEND_2D = 1,    /* force one pass per q-block x kv-head */
  UA_BACKEND_SPLIT = 2  /* force the split-KV partition + merge path */
} ua_backend_t;

typedef enum { UA_PATH_2D = 1, UA_PATH_SPLIT = 2 } ua_path_t;

/* Host-side sizes of one call (host ints, so the library never reads device data
 * to size its grids), plus optional caller workspace and profiling events. */
typedef struct {
  int32_t num_seqs;
  int32_t total_q;            /* = cu_seqlens_q[num_seqs] */
  int32_t max_seqlen_q;       /* >= every q_len */
  int32_t max_seqlen_k;       /* >= every kv_len */
  int32_t max_blocks_per_seq; /* row length of block_table */
  int32_t num_blocks;         /* physical blocks in each cache */
  int32_t qq_bias_stride;     /* elements per qq_bias row (ignored without qq_bias) */
  int32_t q_dtype;            /* ua_dtype_t: F16 or BF16 */
  int32_t out_dtype;          /* ua_dtype_t: F16, BF16 or F32 */
  int32_t num_splits;         /* 0: the dispatcher decides; > 0: partitions for the split path */
  void* workspace;            /* device scratch for the split path, or NULL: the library keeps
                                 a grow-only buffer per (device, stream) and never frees a
                                 replaced one while the process lives */
  size_t workspace_bytes;     /* bytes at `workspace` */
  void* events;               /* NULL, or cudaEvent_t[3] recorded on `stream` before the
                                 attention kernel, after it, and after the merge kernel */
  /* fp8 caches: per-token scales (aiter PR #3962 "split-K long-context decode for shuffled
   * fp8 SWA", test matrix: per-token scales, K and V scales with different strides), or
   * NULL for the per-tensor kv_scale.  Device float32 arrays over (block, slot, kv-head):
   * the scale of key slot s of physical block b, kv-head g, is
   * k_scale_tok[b * k_scale_stride[0] + s * k_scale_stride[1] + g * k_scale_stride[2]]
   * (strides in elements, each >= 0); V likewise with its own strides.  Both or neither;
   * ignored for fp16 / bf16 caches.  Read by the decode tile (at most 8 rows per kv-head,
   * head_dim <= 128, 16 | block_size); other calls with them return UA_ERR_UNSUPPORTED.
   * Every scale a call reads must be finite, and V scales below 256 (a key's P times its V
   * scale is an f16 MMA operand). */
  const float* k_scale_tok;
  const float* v_scale_tok;
  int64_t k_scale_stride[3];
  int64_t v_scale_stride[3];
} ua_shape_t;

/* What the dispatcher chose for a call (see ua_plan). */
typedef struct {
  int32_t path;        /* ua_path_t */
  int32_t kernel;      /* 1: warp-MMA tile kernel, 16 rows per CTA (decode-shaped q-blocks);
                          2: key-major decode tile, 8 rows per CTA (decode with at most 8
                          rows per kv-head, head_dim <= 128, 16 | block_size);
                          4: warp-MMA tile kernel, 64 rows per CTA (fp8 caches at head_dim
                          256, block sizes not a multiple of 16); 8: tensor-memory
                          (tcgen05) kernel with 128-row q-blocks of floor(128 / G) tokens x
                          G heads (16-bit caches, or fp8 at head_dim <= 128: codes dequantised
                          to f16 in shared memory as in RocKE "fp8 KV cache", a bf16 q
                          taken as f16); 16: the same
                          kernel with two such tiles of consecutive tokens per CTA; 32: the
                          key-major decode tile of code 2 with eight consumer warps (128-key
                          stages, one CTA per SM), for decode grids of at most one CTA per SM;
                          64: the decode tile of code 2 with two kv-heads per CTA (fp8 caches
                          with per-tensor scales, at most 4 rows per kv-head, an even
                          num_kv_heads): one page box carries both heads' rows */
  int32_t block_m;     /* (query token x head) rows per q-block */
  int32_t n_part;      /* key-range partitions (1 on the 2D path) */
  int32_t grid_x;      /* q-block slots: num_seqs when slot_per_seq, else
                          floor(total_q * G / block_m) + num_seqs */
  int32_t grid_y;      /* num_kv_heads (num_kv_heads / 2 for kernel 64) */
  int32_t grid_z;      /* n_part */
  int32_t num_sms;     /* SM count the plan was made for */
  int32_t cluster_y;   /* CTAs of one q-block slot (different kv-heads) launched as a cluster */
  int32_t cluster_z;   /* > 1: the n_part partitions of a slot are one cluster too (cluster
                          cluster_y x cluster_z, at most 16 CTAs) and merge through
                          distributed shared memory, with no merge kernel and no workspace */
  int32_t slot_per_seq; /* 1: every sequence fits one q-block and grid slot x is sequence x */
  size_t workspace_bytes; /* scratch the split path needs (0 on the 2D path) */
} ua_plan_t;

/*
 * ua_unified_attention -- the attention call described at the top of this file.
 *
 * scale         multiplies q . k (usually 1 / sqrt(head_dim))
 * softcap       > 0 enables s -> softcap * tanh(s / softcap); <= 0 disables it
 * window_left   >= 0: a query at position p sees keys p - window_left .. p
 *               (a window of W keys including the query itself is W - 1); < 0: off
 * alibi_slopes, qq_bias, sinks: device float32 arrays, or NULL to disable
 * kv_dtype      ua_dtype_t of both caches: F16, BF16 (q_dtype must match) or F8E4M3
 *               (OCP e4m3fn; q may be F16 or BF16, |q| < 65504)
 * kv_scale      device float32[2] {k_scale, v_scale}, required with F8E4M3
 * backend       ua_backend_t
 * stream        cudaStream_t to launch on
 * shape         host-side sizes (must not be NULL)
 *
 * Returns UA_OK after the kernels are enqueued.  UA_ERR_INVALID_ARG for: a NULL
 * required pointer or shape; a tensor pointer not 16-byte aligned; num_q_heads not
 * a positive multiple of num_kv_heads; head_dim not 64, 128 or 256; block_size < 1;
 * negative sizes; qq_bias with qq_bias_stride < max_seqlen_q; an unknown enum.
 * UA_ERR_UNSUPPORTED for q_dtype != kv_dtype with a 16-bit cache.  UA_ERR_WORKSPACE
 * when `shape->workspace` is given but smaller than the plan needs.  UA_ERR_CUDA
 * when a launch or allocation fails.
 */
int ua_unified_attention(const void* q, const void* k_cache, const void* v_cache, void* out,
                         const int32_t* cu_seqlens_q, const int32_t* seq_lens_k,
                         const int32_t* block_table, int block_size, int num_q_heads,
                         int num_kv_heads, int head_dim, float scale, float softcap,
                         int window_left, const float* alibi_slopes, const float* qq_bias,
                         const float* sinks, int kv_dtype, const float* kv_scale, int backend,
                         void* stream, const ua_shape_t* shape);

/*
 * ua_unified_attention_noalloc -- ua_unified_attention for callers that may not
 * allocate device memory (the pages have no counterpart: this is a library service).
 *
 * Some callers cannot call cudaMalloc: a serving runtime that gives all free device
 * memory to its own cache pool at start-up, a process held to a fixed memory budget,
 * or a latency-critical loop where an allocation (which can block and synchronise the
 * device) is not allowed.  ua_unified_attention allocates only when the split-KV path
 * runs without a caller workspace; this entry point runs the same kernels but keeps the
 * split path's scratch in one fixed device array of UA_NOALLOC_SCRATCH_BYTES that the
 * library holds on every GPU that loads it, until the process exits.  It never calls
 * cudaMalloc or cudaFree.
 *
 * Arguments and results are those of ua_unified_attention, except that
 * shape->workspace is ignored.  Extra behaviour:
 *   - UA_ERR_SCRATCH_LIMIT, before anything is launched, when the plan needs more than
 *     UA_NOALLOC_SCRATCH_BYTES of scratch (ua_plan reports workspace_bytes).
 *   - The first call on a device looks up the array's device address (with that device
 *     current); make that first call before any stream capture on the device.  The
 *     address is kept until the process exits and does not survive cudaDeviceReset:
 *     after a reset of the device, do not call this entry point again.
 *   - Every call on a device shares the one array: calls whose kernels overlap on the
 *     GPU (different streams, or several host threads) race on it and give wrong
 *     results.  Calls on one stream are ordered and safe.  The array keeps the last
 *     call's contents; nothing in it needs to start at zero.
 */
int ua_unified_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                 void* out, const int32_t* cu_seqlens_q,
                                 const int32_t* seq_lens_k, const int32_t* block_table,
                                 int block_size, int num_q_heads, int num_kv_heads, int head_dim,
                                 float scale, float softcap, int window_left,
                                 const float* alibi_slopes, const float* qq_bias,
                                 const float* sinks, int kv_dtype, const float* kv_scale,
                                 int backend, void* stream, const ua_shape_t* shape);

/*
 * ua_plan -- the dispatcher's decision for a call with these sizes, without touching
 * the GPU: path, kernel, partitions, grid and workspace bytes.  The split path is
 * taken (UA_BACKEND_AUTO) when the 2D grid fills less than one wave of SMs and the
 * longest key walk of a q-block spans at least two minimum partitions (grid fill and
 * walk length, as in the aiter PR #3962 gating and the RocKE harness "Why three
 * tables").  num_sms <= 0 asks the current CUDA device.  Returns UA_OK or
 * UA_ERR_INVALID_ARG / UA_ERR_CUDA (device query).
 */
int ua_plan(const ua_shape_t* shape, int block_size, int num_q_heads, int num_kv_heads,
            int head_dim, int window_left, int kv_dtype, int backend, int num_sms,
            ua_plan_t* plan);

/*
 * ua_workspace_bytes -- bytes of split-path scratch a call with these sizes needs on the
 * current device (0 when it takes the 2D path or merges its partitions inside a
 * thread-block cluster): fp32 max and sum per (query token, head, partition), then the
 * unnormalised partial output rows, each piece 256-byte aligned.  The scratch rules follow
 * the author's follow-up on the review of aiter PR #3962 ("split-K long-context decode for
 * shuffled fp8 SWA"): the partition count is capped, the scratch belongs to one stream at a
 * time (a caller workspace, or the library's own buffer per device and stream), and every
 * entry the merge reads is written by the same call, so the scratch needs no clearing.
 * Returns 0 on an invalid argument too.
 */
size_t ua_workspace_bytes(const ua_shape_t* shape, int block_size, int num_q_heads,
                          int num_kv_heads, int head_dim, int window_left, int kv_dtype,
                          int backend);

/*
 * ua_device_status -- synchronises `stream`, then stores in *status the device
 * check word the kernels of this library raised since the last reset, mapped to
 * UA_OK, UA_ERR_DEVICE_CHECK (a block id outside the cache, or a q_len
 * above max_seqlen_q in a decode-shaped call) or UA_ERR_TIMEOUT (a
 * bounded wait expired).  Returns UA_OK or UA_ERR_CUDA / UA_ERR_INVALID_ARG.
 * The word reports what the kernels refuse to read rather than faulting: a bad block id
 * is never dereferenced (its keys count as zero).  Slots of a sequence's last page at or
 * past kv_len are never an input either: whatever they hold (NaN included) gets weight
 * exactly 0 and its V values are zeroed before P.V, after the NaN-in-unused-V-slots
 * finding of the follow-up on aiter PR #3962's review.
 */
int ua_device_status(void* stream, int* status);

/* Clears the device check word (enqueued on `stream`). */
int ua_device_status_reset(void* stream);

/* Static text for a ua_status_t code. */
const char* ua_status_string(int status);

/* UA_VERSION of the loaded library. */
int ua_version(void);

#ifdef __cplusplus
}
#endif

#endif /* UA_H_ */
