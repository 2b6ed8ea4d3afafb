/*
 * ua_ref.c -- plain, slow fp64 CPU oracle for unified paged varlen GQA attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  It shares no code, header,
 * table or constant with the CUDA library, and it never calls it.
 *
 * What it computes (one output row per query token t and query head h):
 *
 *   Sources: "RocKE unified_attention parity & benchmark harness" (gfx950 README),
 *   section "Running" step 1 and "2D vs 2D" (ALiBi and QQ-bias offsets measured
 *   from context_len); the vllm-rdna PR #34 "FA-RDNA2 D=128 prefill" (paged varlen
 *   GQA prefill behind a prefix, head group g = h / G); the ROCm/aiter PR #3962
 *   "split-K long-context decode for shuffled fp8 SWA" (windowed key range
 *   [seq_len - window, seq_len), online-softmax update, per-partition
 *   max/sum/partial-O, a merge that skips partitions whose sum is 0, zero rows for
 *   rows without keys).
 *
 *   For sequence b with q_len = cu_seqlens_q[b+1] - cu_seqlens_q[b] and
 *   kv_len = seq_lens_k[b], context_len ctx = kv_len - q_len.
 *   Query row i (0 <= i < q_len) of head h sits at absolute position p = ctx + i
 *   and reads kv-head g = h / (H_q / H_kv).
 *   Allowed keys: 0 <= j < kv_len, j <= p, and p - j <= window_left when
 *   window_left >= 0.
 *   Key j lives at cache row block_table[b][j / block_size], slot j % block_size.
 *     s_j  = scale * sum_d q[t,h,d] * K_j[d]          (fp8: K_j = e4m3(k) * k_scale)
 *     s_j  = softcap * tanh(s_j / softcap)            if softcap > 0
 *     s_j += alibi_slopes[h] * (j - ctx)              if ALiBi is on
 *     s_j += qq_bias[i * stride + (j - ctx)]          if QQ-bias is on and j >= ctx
 *     m    = max(sink_h (if sinks), max_j s_j)
 *     den  = exp(sink_h - m) (if sinks) + sum_j exp(s_j - m)
 *     o    = sum_j exp(s_j - m) V_j / den             (fp8: V_j = e4m3(v) * v_scale)
 *   fp8 scales are per tensor (k_scale, v_scale) or, after the same aiter PR's test
 *   matrix ("scalar and per-token scales, K and V scales with different strides"), per
 *   cached token: the scale of key j's K (V) row of kv-head g is the element (block,
 *   slot, g) of its own array, block = block_table[b][j / block_size] and
 *   slot = j % block_size, at block * stride0 + slot * stride1 + g * stride2.
 *   A row with no allowed key is 0, with or without a sink (rows of a sequence
 *   with kv_len < q_len whose position p is negative have no key).
 *
 *   The order "scale, softcap, ALiBi, QQ-bias, mask" is this library's reading of
 *   the pages, which name the terms but do not print their order: parity unpinned
 *   for the composition of softcap with the biases (each term alone is pinned by the
 *   tests: closed forms, the row-shift invariance of ALiBi without sinks, softcap
 *   limits, brute force).
 *
 * Element decoders follow the published bit layouts: IEEE-754 binary16, bfloat16
 * (upper half of binary32) and OCP 8-bit e4m3fn (bias 7, no infinities, S.1111.111
 * is NaN, largest finite 448).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define REF_F16 0
#define REF_BF16 1
#define REF_E4M3 2
#define REF_F32 3

#define REF_OK 0
#define REF_ERR_ARG 1
#define REF_ERR_BLOCK 3 /* block id outside [0, num_blocks) */
#define REF_ERR_MEM 4

typedef struct {
  const void* q;            /* [total_q, H_q, D], q_dtype */
  const void* k_cache;      /* [num_blocks, block_size, H_kv, D], kv_dtype */
  const void* v_cache;      /* same layout as k_cache */
  const int32_t* cu_seqlens_q; /* [num_seqs + 1] */
  const int32_t* seq_lens_k;   /* [num_seqs] */
  const int32_t* block_table;  /* [num_seqs, max_blocks_per_seq] */
  const float* alibi_slopes;   /* [H_q] or NULL */
  const float* qq_bias;        /* [rows, qq_bias_stride] or NULL */
  const float* sinks;          /* [H_q] or NULL */
  int32_t q_dtype, kv_dtype;
  int32_t num_seqs, max_blocks_per_seq, num_blocks, block_size;
  int32_t num_q_heads, num_kv_heads, head_dim;
  int32_t window_left;   /* < 0: no window */
  int32_t qq_bias_stride;
  double scale, softcap; /* softcap <= 0: off */
  double k_scale, v_scale;
  /* fp8 per-token scales (NULL: the per-tensor k_scale / v_scale); element strides of
     block, slot and kv-head */
  const float* k_scale_tok;
  const float* v_scale_tok;
  int64_t k_scale_strides[3];
  int64_t v_scale_strides[3];
} ua_ref_problem;

double ua_ref_decode_f16(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)m, -24);          /* 0.m * 2^-14 */
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp(1.0 + m / 1024.0, e - 15);
  return s ? -v : v;
}

double ua_ref_decode_bf16(uint16_t b) {
  int s = b >> 15, e = (b >> 7) & 0xFF, m = b & 0x7F;
  double v;
  if (e == 0) v = ldexp((double)m, -133);         /* 0.m * 2^-126 */
  else if (e == 255) v = m ? NAN : INFINITY;
  else v = ldexp(1.0 + m / 128.0, e - 127);
  return s ? -v : v;
}

double ua_ref_decode_e4m3(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);           /* 0.m * 2^-6 */
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

static double load_elem(const void* base, int dtype, size_t idx) {
  switch (dtype) {
    case REF_F16: return ua_ref_decode_f16(((const uint16_t*)base)[idx]);
    case REF_BF16: return ua_ref_decode_bf16(((const uint16_t*)base)[idx]);
    case REF_E4M3: return ua_ref_decode_e4m3(((const uint8_t*)base)[idx]);
    default: return (double)((const float*)base)[idx];
  }
}

/* Sequence that owns global query token t (cu_seqlens_q is non-decreasing). */
static int seq_of_token(const ua_ref_problem* P, int t) {
  for (int b = 0; b < P->num_seqs; ++b)
    if (t >= P->cu_seqlens_q[b] && t < P->cu_seqlens_q[b + 1]) return b;
  return -1;
}

/* Cache row (in units of D-element rows) holding key j of sequence b, kv-head g. */
static int cache_row(const ua_ref_problem* P, int b, int j, int g, size_t* row) {
  int32_t blk = P->block_table[(size_t)b * P->max_blocks_per_seq + j / P->block_size];
  if (blk < 0 || blk >= P->num_blocks) return REF_ERR_BLOCK;
  *row = (((size_t)blk * P->block_size + (size_t)(j % P->block_size)) * P->num_kv_heads + g);
  return REF_OK;
}

/* The fp8 scale of key j's K (which = 0) or V (which = 1) row of kv-head g; 1 for 16-bit
   caches. */
static double kv_scale_of(const ua_ref_problem* P, int which, int b, int j, int g) {
  if (P->kv_dtype != REF_E4M3) return 1.0;
  const float* tok = which ? P->v_scale_tok : P->k_scale_tok;
  if (!tok) return which ? P->v_scale : P->k_scale;
  const int64_t* st = which ? P->v_scale_strides : P->k_scale_strides;
  int64_t blk = P->block_table[(size_t)b * P->max_blocks_per_seq + j / P->block_size];
  return (double)tok[blk * st[0] + (int64_t)(j % P->block_size) * st[1] + (int64_t)g * st[2]];
}

/*
 * Allowed key range [*lo, *hi) of query row i of sequence b.  A row whose position
 * p = ctx + i is negative (only when kv_len < q_len, e.g. a decode slot whose
 * sequence holds no key yet) has no key at all.
 */
static void key_range(const ua_ref_problem* P, int b, int i, int* ctx, int* lo, int* hi) {
  int q_len = P->cu_seqlens_q[b + 1] - P->cu_seqlens_q[b];
  int kv_len = P->seq_lens_k[b];
  *ctx = kv_len - q_len;
  int p = *ctx + i;
  *hi = p + 1 < kv_len ? p + 1 : kv_len;
  if (*hi < 0) *hi = 0;
  *lo = 0;
  if (P->window_left >= 0 && p - P->window_left > 0) *lo = p - P->window_left;
  if (*lo > *hi) *lo = *hi;
}

/* Transformed score of key j for row (t, i, h): the s_j of the header. */
static int score(const ua_ref_problem* P, int b, int t, int i, int h, int ctx, int j, double* s) {
  const int D = P->head_dim, G = P->num_q_heads / P->num_kv_heads;
  size_t row;
  int rc = cache_row(P, b, j, h / G, &row);
  if (rc) return rc;
  double kscale = kv_scale_of(P, 0, b, j, h / G);
  double dot = 0.0;
  for (int d = 0; d < D; ++d) {
    double qd = load_elem(P->q, P->q_dtype, ((size_t)t * P->num_q_heads + h) * D + d);
    double kd = load_elem(P->k_cache, P->kv_dtype, row * D + d) * kscale;
    dot += qd * kd;
  }
  double v = P->scale * dot;
  if (P->softcap > 0.0) v = P->softcap * tanh(v / P->softcap);
  if (P->alibi_slopes) v += (double)P->alibi_slopes[h] * (double)(j - ctx);
  if (P->qq_bias && j >= ctx) v += (double)P->qq_bias[(size_t)i * P->qq_bias_stride + (j - ctx)];
  *s = v;
  return REF_OK;
}

static int add_value_row(const ua_ref_problem* P, int b, int j, int g, double w, double* acc) {
  const int D = P->head_dim;
  size_t row;
  int rc = cache_row(P, b, j, g, &row);
  if (rc) return rc;
  double vscale = kv_scale_of(P, 1, b, j, g);
  for (int d = 0; d < D; ++d) acc[d] += w * load_elem(P->v_cache, P->kv_dtype, row * D + d) * vscale;
  return REF_OK;
}

/* One output row by the plain definition (one pass over the allowed keys). */
static int ref_row(const ua_ref_problem* P, int t, int h, double* o) {
  const int D = P->head_dim, G = P->num_q_heads / P->num_kv_heads;
  int b = seq_of_token(P, t);
  if (b < 0) return REF_ERR_ARG;
  int i = t - P->cu_seqlens_q[b], ctx, lo, hi, rc;
  key_range(P, b, i, &ctx, &lo, &hi);
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  int n = hi - lo;
  if (n == 0) return REF_OK; /* no keys: zero row whether or not a sink exists */
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  double* acc = (double*)calloc((size_t)D, sizeof(double));
  if (!s || !acc) { free(s); free(acc); return REF_ERR_MEM; }
  double m = P->sinks ? (double)P->sinks[h] : -INFINITY;
  for (int j = lo; j < hi; ++j) {
    if ((rc = score(P, b, t, i, h, ctx, j, &s[j - lo]))) goto done;
    if (s[j - lo] > m) m = s[j - lo];
  }
  double den = P->sinks ? exp((double)P->sinks[h] - m) : 0.0;
  for (int j = lo; j < hi; ++j) {
    double w = exp(s[j - lo] - m);
    den += w;
    if ((rc = add_value_row(P, b, j, h / G, w, acc))) goto done;
  }
  for (int d = 0; d < D; ++d) o[d] = acc[d] / den;
done:
  free(s);
  free(acc);
  return rc;
}

/*
 * The split-KV (flash-decoding) form of the same row, after the aiter PR #3962
 * "Changes" and its review fixes: the allowed range is cut into n_part
 * contiguous partitions of ceil(n / n_part) keys that together cover it; each
 * partition keeps its own max m_p, sum l_p and unnormalised acc_p (the sink joins
 * partition 0 only, as the initial max); the merge takes M = max m_p over the
 * partitions with l_p > 0, L = sum l_p exp(m_p - M), o = sum acc_p exp(m_p - M) / L,
 * and a row where every l_p is 0 is 0.
 */
static int ref_row_split(const ua_ref_problem* P, int t, int h, int n_part, double* o) {
  const int D = P->head_dim, G = P->num_q_heads / P->num_kv_heads;
  int b = seq_of_token(P, t);
  if (b < 0 || n_part < 1) return REF_ERR_ARG;
  int i = t - P->cu_seqlens_q[b], ctx, lo, hi, rc = REF_OK;
  key_range(P, b, i, &ctx, &lo, &hi);
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  int n = hi - lo;
  if (n == 0) return REF_OK;
  int chunk = (n + n_part - 1) / n_part;
  double* mp = (double*)malloc(sizeof(double) * (size_t)n_part);
  double* lp = (double*)malloc(sizeof(double) * (size_t)n_part);
  double* ap = (double*)calloc((size_t)n_part * D, sizeof(double));
  if (!mp || !lp || !ap) { rc = REF_ERR_MEM; goto done; }
  for (int pp = 0; pp < n_part; ++pp) {
    int a = lo + pp * chunk, e = a + chunk < hi ? a + chunk : hi;
    double m = (pp == 0 && P->sinks) ? (double)P->sinks[h] : -INFINITY;
    double s;
    for (int j = a; j < e; ++j) {
      if ((rc = score(P, b, t, i, h, ctx, j, &s))) goto done;
      if (s > m) m = s;
    }
    double l = (pp == 0 && P->sinks) ? exp((double)P->sinks[h] - m) : 0.0;
    for (int j = a; j < e; ++j) {
      if ((rc = score(P, b, t, i, h, ctx, j, &s))) goto done;
      double w = exp(s - m);
      l += w;
      if ((rc = add_value_row(P, b, j, h / G, w, ap + (size_t)pp * D))) goto done;
    }
    mp[pp] = m;
    lp[pp] = l;
  }
  {
    double M = -INFINITY, L = 0.0;
    for (int pp = 0; pp < n_part; ++pp)
      if (lp[pp] > 0.0 && mp[pp] > M) M = mp[pp];
    if (M == -INFINITY) goto done; /* every partition empty: zero row */
    for (int pp = 0; pp < n_part; ++pp)
      if (lp[pp] > 0.0) L += lp[pp] * exp(mp[pp] - M);
    for (int pp = 0; pp < n_part; ++pp) {
      if (!(lp[pp] > 0.0)) continue;
      double w = exp(mp[pp] - M) / L;
      for (int d = 0; d < D; ++d) o[d] += ap[(size_t)pp * D + d] * w;
    }
  }
done:
  free(mp);
  free(lp);
  free(ap);
  return rc;
}

static int check_problem(const ua_ref_problem* P) {
  if (!P || !P->q || !P->k_cache || !P->v_cache || !P->cu_seqlens_q || !P->seq_lens_k ||
      !P->block_table)
    return REF_ERR_ARG;
  if (P->num_q_heads <= 0 || P->num_kv_heads <= 0 || P->num_q_heads % P->num_kv_heads)
    return REF_ERR_ARG;
  if (P->head_dim <= 0 || P->block_size <= 0 || P->num_seqs < 0) return REF_ERR_ARG;
  if (P->qq_bias && P->qq_bias_stride <= 0) return REF_ERR_ARG;
  return REF_OK;
}

/*
 * Full output for query tokens [t_begin, t_end) and heads [h_begin, h_end).
 * out is [total_q, H_q, D] fp64; only the requested rows are written.
 * n_part <= 0 selects the one-pass definition, n_part >= 1 the split form.
 */
int ua_ref_attention(const ua_ref_problem* P, int t_begin, int t_end, int h_begin, int h_end,
                     int n_part, double* out) {
  int rc = check_problem(P);
  if (rc) return rc;
  const int D = P->head_dim, H = P->num_q_heads;
  for (int t = t_begin; t < t_end; ++t)
    for (int h = h_begin; h < h_end; ++h) {
      double* o = out + ((size_t)t * H + h) * D;
      rc = n_part >= 1 ? ref_row_split(P, t, h, n_part, o) : ref_row(P, t, h, o);
      if (rc) return rc;
    }
  return REF_OK;
}

/* Selected rows only: out[r] (D doubles) is the row of (tokens[r], heads[r]). */
int ua_ref_attention_rows(const ua_ref_problem* P, const int32_t* tokens, const int32_t* heads,
                          int n_rows, double* out) {
  int rc = check_problem(P);
  if (rc) return rc;
  for (int r = 0; r < n_rows; ++r) {
    if (heads[r] < 0 || heads[r] >= P->num_q_heads) return REF_ERR_ARG;
    rc = ref_row(P, tokens[r], heads[r], out + (size_t)r * P->head_dim);
    if (rc) return rc;
  }
  return REF_OK;
}
