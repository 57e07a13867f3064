/*
 * dsa_oracle.c -- plain fp64 CPU oracle for the DSA forward path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the bench's CPU-baseline leg load this library.  It shares no
 * code, header, table or helper with the CUDA path under
 * sparse_attention_gemm_gb300/csrc, and the CUDA path never calls it.
 *
 * Every function is the plain definition of one step, written out with
 * fp64 arithmetic and no blocking, fusion or reordering.  Inputs that the
 * GPU sees as bf16 are passed here already widened to double (exactly).
 * Rows are independent, so the outer loops run over rows with OpenMP.
 *
 * Sources (page title, section):
 *  [P1] NeMo AutoModel, nemo_automodel.components.models.glm_moe_dsa.
 *       kernels.cudnn_dsa: prepare_cudnn_dsa_packed_metadata (per-query
 *       storage starts and causal lengths), cudnn_indexer_topk (THD shapes,
 *       pre-scaled head weights, global ids), _compact_and_sort_indices,
 *       cudnn_sparse_attention (q [T,H,576], kv [T,1,576], -1 suffix).
 *  [P2] NeMo AutoModel, ...models.common.cudnn_sparse_attention:
 *       _compact_and_sort_indices (valid ids < key_count, ascending prefix).
 *  [P4] NeMo AutoModel, ...qwen3_8_flash_next.cudnn_qsa: _pack_indices,
 *       cudnn_sparse_gqa_attention.
 *  [P5] cuDNN Frontend, "DeepSeek Sparse Attention (DSA)": section 1
 *       (Sparse Attention Forward), section 3 (Indexer Forward), section 4
 *       (Combined Indexer Forward + Top-K, deterministic tie-break), section
 *       5 (Indexer Top-K), "Compact vs. non-compact sparse indices".
 *
 * Parity status: every function below is pinned by the not-gpu tests in
 * tests/test_oracle_pins.py (brute force, closed forms, library special
 * cases and invariants); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads the row loops below use from now on (n >= 1); for timing the
 * oracle on one core and on all of them.  Returns the previous count. */
int oracle_set_num_threads(int n) {
#ifdef _OPENMP
  const int prev = omp_get_max_threads();
  if (n >= 1) omp_set_num_threads(n);
  return prev;
#else
  (void)n;
  return 1;
#endif
}

/* ------------------------------------------------------------------------
 * THD metadata [P1 prepare_cudnn_dsa_packed_metadata, "Returns": per-query
 * storage starts and real causal lengths].  Tokens of document b occupy
 * rows cu[b] .. cu[b+1]-1; token t of that document has start[t] = cu[b]
 * and causal length len[t] = t - cu[b] + 1 (itself included).
 * Returns 0, or -1 when cu is not a valid prefix array covering [0, T).
 * ------------------------------------------------------------------------ */
int oracle_thd_metadata(const int32_t* cu, int n_docs, int T, int32_t* start,
                        int32_t* len) {
  if (n_docs < 1 || cu[0] != 0 || cu[n_docs] != T) return -1;
  for (int b = 0; b < n_docs; ++b)
    if (cu[b + 1] < cu[b]) return -1;
  for (int b = 0; b < n_docs; ++b) {
    for (int t = cu[b]; t < cu[b + 1]; ++t) {
      start[t] = cu[b];
      len[t] = t - cu[b] + 1;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------
 * Ratio-causal metadata of a compressed-key indexer [P5 section 3,
 * "ratio-causal mask" and q_causal_offsets; section 4, compact addressing
 * clamps rows that extend past the key prefix].  Query segment b occupies
 * rows cu_q[b] .. cu_q[b+1]-1 and its compressed keys rows cu_k[b] ..
 * cu_k[b+1]-1 (a prefix of the segment's compressed timeline, from
 * compressed column 0).  Local query row q (q = t - cu_q[b]) sees key
 * column j iff
 *     j < clamp( floor((q_off[b] + q + 1) / ratio), 0, cu_k[b+1] - cu_k[b] ),
 * q_off[b] being the global position of the segment's first query (0 when
 * q_off is NULL).  start[t] = cu_k[b] and len[t] = that bound.
 * Returns 0, or -1 when cu_q / cu_k are not valid prefix arrays over
 * [0, Tq) / [0, Tk) or ratio < 1.
 * ------------------------------------------------------------------------ */
int oracle_ratio_metadata(const int32_t* cu_q, const int32_t* cu_k,
                          const int32_t* q_off, int n_docs, int Tq, int Tk,
                          int ratio, int32_t* start, int32_t* len) {
  if (n_docs < 1 || ratio < 1 || cu_q[0] != 0 || cu_q[n_docs] != Tq ||
      cu_k[0] != 0 || cu_k[n_docs] != Tk)
    return -1;
  for (int b = 0; b < n_docs; ++b)
    if (cu_q[b + 1] < cu_q[b] || cu_k[b + 1] < cu_k[b]) return -1;
  for (int b = 0; b < n_docs; ++b) {
    const int64_t seqlen_k = cu_k[b + 1] - cu_k[b];
    const int64_t off = q_off ? q_off[b] : 0;
    for (int t = cu_q[b]; t < cu_q[b + 1]; ++t) {
      const int64_t num = off + (t - cu_q[b]) + 1;
      /* floor division (num may be negative for a negative offset) */
      int64_t bound = num >= 0 ? num / ratio : -((-num + ratio - 1) / ratio);
      if (bound < 0) bound = 0;
      if (bound > seqlen_k) bound = seqlen_k;
      start[t] = cu_k[b];
      len[t] = (int32_t)bound;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------
 * FP8 indexer inputs [P5 section 3, precision path "fp8": Q/K in E4M3 with
 * fp32 descales, one per token (and head for Q)].  E4M3 is the 8-bit float
 * with 1 sign, 4 exponent (bias 7) and 3 mantissa bits, no infinities, and
 * NaN only for exponent and mantissa all ones:
 *   e = 0:  (-1)^s * (m / 8) * 2^(1 - 7)      (zero and subnormals)
 *   e > 0:  (-1)^s * (1 + m / 8) * 2^(e - 7)
 * oracle_fp8_dequant writes out[r * len + i] = value(codes[r * len + i]) *
 * scales[r]: each row of `len` codes has one descale.  The dequantized
 * tensors then go through oracle_indexer_scores unchanged:
 *   score = sum_h w * ReLU( sum_c (q_scale * q) * (k_scale * k) ).
 * ------------------------------------------------------------------------ */
double oracle_e4m3_value(uint8_t code) {
  const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? ldexp((double)m / 8.0, 1 - 7) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

void oracle_fp8_dequant(const uint8_t* codes, const float* scales, int64_t rows, int len, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int i = 0; i < len; ++i)
      out[r * len + i] = oracle_e4m3_value(codes[r * len + i]) * (double)scales[r];
}

/* ------------------------------------------------------------------------
 * MXFP8 indexer inputs [P5 section 3, precision path "mxfp8": Q/K in E4M3
 * with block-scaled E8M0 scales, sf_vec_size 32].  An E8M0 scale is an
 * exponent alone: byte e stands for 2^(e - 127) (e = 0 .. 254); e = 255 is
 * NaN.  A row of `len` codes carries len / 32 scales, scale b applying to
 * elements 32 b .. 32 b + 31:
 *   x[i] = value(codes[i]) * 2^(scales[i / 32] - 127).
 * The dequantized tensors then go through oracle_indexer_scores unchanged,
 * so each dot product is the block-scaled sum
 *   sum_b 2^(eq_b - 127) * 2^(ek_b - 127) * sum_{i in block b} q[i] * k[i].
 * The page leaves the packed storage of the scales to its library; here they
 * are plain [rows, len / 32] bytes.
 * ------------------------------------------------------------------------ */
double oracle_e8m0_value(uint8_t e) {
  if (e == 255) return NAN;
  return ldexp(1.0, (int)e - 127);
}

void oracle_mxfp8_dequant(const uint8_t* codes, const uint8_t* scales, int64_t rows, int len, double* out) {
  const int nb = len / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int i = 0; i < len; ++i)
      out[r * len + i] = oracle_e4m3_value(codes[r * len + i]) * oracle_e8m0_value(scales[r * nb + i / 32]);
}

/* ------------------------------------------------------------------------
 * Lightning-indexer scores [P5 section 3; P1 cudnn_indexer_topk].
 * For one query row with inputs qi_row [Hi, d], w_row [Hi] and keys
 * ki [*, d]:
 *     score[j] = sum_h w[h] * ReLU( sum_c qi[h, c] * ki[start + j, c] )
 * for 0 <= j < len (ratio 1, zero causal offset: key j is visible iff
 * j < q_local + 1), and -inf for len <= j < s_max.  No scaling is applied:
 * the head weights arrive already scaled.
 *
 * abs_scale (optional) receives sum_h |w[h]| * sum_c |qi[h,c] * ki[s,c]|,
 * the magnitude that bounds the rounding error of any fp32 evaluation.
 * Rows are given compactly: qi_rows [n_rows, Hi, d], w_rows [n_rows, Hi],
 * start_rows / len_rows [n_rows]; ki is the full key tensor [T_k, d].
 * ------------------------------------------------------------------------ */
void oracle_indexer_scores(const double* qi_rows, const double* ki,
                           const double* w_rows, const int32_t* start_rows,
                           const int32_t* len_rows, int n_rows, int Hi, int d,
                           int s_max, double* scores, double* abs_scale) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < n_rows; ++r) {
    const double* qi = qi_rows + (int64_t)r * Hi * d;
    const double* w = w_rows + (int64_t)r * Hi;
    double* out = scores + (int64_t)r * s_max;
    double* mag = abs_scale ? abs_scale + (int64_t)r * s_max : NULL;
    for (int j = 0; j < s_max; ++j) {
      if (j >= len_rows[r]) {
        out[j] = -INFINITY;
        if (mag) mag[j] = 0.0;
        continue;
      }
      const double* k = ki + (int64_t)(start_rows[r] + j) * d;
      double s = 0.0, a = 0.0;
      for (int h = 0; h < Hi; ++h) {
        double dot = 0.0, adot = 0.0;
        for (int c = 0; c < d; ++c) {
          dot += qi[h * d + c] * k[c];
          adot += fabs(qi[h * d + c] * k[c]);
        }
        s += w[h] * (dot > 0.0 ? dot : 0.0);
        a += fabs(w[h]) * adot;
      }
      out[j] = s;
      if (mag) mag[j] = a;
    }
  }
}

/* ------------------------------------------------------------------------
 * Per-row top-k [P5 section 5 (per-row effective length), section 4
 * (deterministic: ties at the k-th boundary go to the smallest KV index;
 * padded slots are -1)].  The definition: order the candidates 0..len-1 by
 * score descending and, among equal scores, by index ascending; keep the
 * first min(K, len).  The kept ids are written in ascending id order (the
 * canonical compact prefix of P1 cudnn_sparse_attention) as start + j
 * (global ids) or j (start_rows == NULL, local ids), followed by -1.
 * topk_len receives min(K, len).
 * ------------------------------------------------------------------------ */
typedef struct {
  double score;
  int32_t j;
} oracle_pair;

static int cmp_score_desc_index_asc(const void* a, const void* b) {
  const oracle_pair* x = (const oracle_pair*)a;
  const oracle_pair* y = (const oracle_pair*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int cmp_i32_asc(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x < y) ? -1 : (x > y);
}

int oracle_topk(const double* scores, int64_t ld, const int32_t* len_rows,
                const int32_t* start_rows, int n_rows, int K, int32_t* idx,
                int32_t* topk_len) {
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int r = 0; r < n_rows; ++r) {
    int len = len_rows[r];
    if (len < 0) len = 0;
    if (len > ld) len = (int)ld;
    oracle_pair* p = (oracle_pair*)malloc(sizeof(oracle_pair) * (size_t)(len > 0 ? len : 1));
    if (!p) { bad = 1; continue; }
    for (int j = 0; j < len; ++j) {
      p[j].score = scores[(int64_t)r * ld + j];
      p[j].j = j;
    }
    qsort(p, (size_t)len, sizeof(oracle_pair), cmp_score_desc_index_asc);
    int n = len < K ? len : K;
    int32_t* out = idx + (int64_t)r * K;
    int32_t base = start_rows ? start_rows[r] : 0;
    for (int i = 0; i < n; ++i) out[i] = base + p[i].j;
    qsort(out, (size_t)n, sizeof(int32_t), cmp_i32_asc);
    for (int i = n; i < K; ++i) out[i] = -1;
    if (topk_len) topk_len[r] = n;
    free(p);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------
 * Compact and sort [P2 _compact_and_sort_indices: an id is valid iff
 * 0 <= id < key_count; P5 "Compact vs. non-compact sparse indices": the
 * valid ids form the prefix, every later slot holds -1, the id convention
 * is preserved].  Valid ids are sorted ascending; duplicates are kept.
 * ------------------------------------------------------------------------ */
/* cuDNN Frontend DSA page, section 4 (Combined Indexer Forward + Top-K):
 * with the indices come the aligned logits (the selected scores, -inf in
 * padded slots), their softmax and its log-sum-exp.  Reading: the softmax
 * and lse run over the row's selected slots j < topk_len[r]; padded slots
 * have probability 0; a row with no slot has lse = -inf. */
void oracle_topk_softmax(const double* scores, int64_t ld, const int32_t* idx,
                         const int32_t* start_rows, const int32_t* topk_len,
                         int n_rows, int K, double* logits, double* softmax,
                         double* lse) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < n_rows; ++r) {
    const int n = topk_len[r];
    const int32_t base = start_rows ? start_rows[r] : 0;
    double m = -INFINITY;
    for (int j = 0; j < K; ++j) {
      double l = -INFINITY;
      if (j < n) l = scores[(int64_t)r * ld + (idx[(int64_t)r * K + j] - base)];
      logits[(int64_t)r * K + j] = l;
      if (l > m) m = l;
    }
    double z = 0.0;
    for (int j = 0; j < n; ++j) z += exp(logits[(int64_t)r * K + j] - m);
    const double lz = n > 0 ? m + log(z) : -INFINITY;
    lse[r] = lz;
    for (int j = 0; j < K; ++j)
      softmax[(int64_t)r * K + j] = j < n ? exp(logits[(int64_t)r * K + j] - lz) : 0.0;
  }
}

void oracle_compact_sort(const int32_t* in, int T, int K, int64_t key_count,
                         int32_t* out, int32_t* lengths) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    int32_t* o = out + (int64_t)t * K;
    int n = 0;
    for (int j = 0; j < K; ++j) {
      int32_t id = in[(int64_t)t * K + j];
      if (id >= 0 && (int64_t)id < key_count) o[n++] = id;
    }
    qsort(o, (size_t)n, sizeof(int32_t), cmp_i32_asc);
    for (int j = n; j < K; ++j) o[j] = -1;
    lengths[t] = n;
  }
}

/* ------------------------------------------------------------------------
 * Route packing [P4 _pack_indices].  routes [B, S, W] hold batch-local ids;
 * an id is kept iff 0 <= id < S and becomes b*S + id, anything else is -1.
 * The output is [B*S, Wp] with Wp = ceil(W/4)*4; slots W..Wp-1 are -1.
 * ------------------------------------------------------------------------ */
void oracle_pack_routes(const int32_t* routes, int B, int S, int W,
                        int32_t* out) {
  int Wp = (W + 3) / 4 * 4;
  for (int b = 0; b < B; ++b)
    for (int s = 0; s < S; ++s)
      for (int j = 0; j < Wp; ++j) {
        int32_t v = -1;
        if (j < W) {
          int32_t id = routes[((int64_t)b * S + s) * W + j];
          if (id >= 0 && id < S) v = b * S + id;
        }
        out[((int64_t)b * S + s) * Wp + j] = v;
      }
}

/* ------------------------------------------------------------------------
 * Sparse MQA attention forward [P5 section 1].  For query row t, head h and
 * valid slot j (j < clamp(topk_length[t], 0, K) when lengths are given, and
 * 0 <= idx[t, j] < Tkv):
 *     s_j = scale * sum_{c < Dqk} q[t, h, c] * kv[idx_j, c]
 * Invalid or out-of-range slots contribute nothing (score -inf); duplicate
 * ids stay separate slots.  The sink enters the denominator only:
 *     Z = sum_j exp(s_j) + exp(sink[h])        (sink absent => -inf)
 *     out[t, h, :] = sum_j exp(s_j) * V[idx_j, :] / Z
 * with V = v (separate value tensor) or the first Dv columns of kv.
 * lse = log Z (the denominator that out uses, sink included);
 * lse_kv = log sum_j exp(s_j) (KV-only, the cuDNN "lse" statistic);
 * max_logits = max_j s_j.  Empty row: out = 0, lse_kv = +inf,
 * max_logits = -inf, lse = sink[h] (or -inf without a sink).
 * Computed two-pass (maximum first, then the sums) in fp64.
 *
 * Rows are compact: q_rows [n_rows, H, Dqk], idx_rows [n_rows, K],
 * len_rows [n_rows] or NULL; kv [Tkv, kv_ld] (kv_ld >= Dqk), v [Tkv, Dv].
 * ------------------------------------------------------------------------ */
void oracle_sparse_attn(const double* q_rows, const double* kv, int64_t kv_ld,
                        const double* v, const int32_t* idx_rows,
                        const int32_t* len_rows, const double* sink, int n_rows,
                        int Tkv, int H, int Dqk, int Dv, int K, double scale,
                        double* out, double* lse, double* lse_kv,
                        double* max_logits, int indexer_topk,
                        double* lse_indexer) {
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
    int32_t* slot = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t rh = 0; rh < (int64_t)n_rows * H; ++rh) {
      int r = (int)(rh / H), h = (int)(rh % H);
      int lim = K;
      if (len_rows) {
        lim = len_rows[r];
        if (lim < 0) lim = 0;
        if (lim > K) lim = K;
      }
      int n = 0;
      for (int j = 0; j < lim; ++j) {
        int32_t id = idx_rows[(int64_t)r * K + j];
        if (id >= 0 && id < Tkv) {
          slot[n] = j;
          ids[n++] = id;
        }
      }
      const double* qh = q_rows + ((int64_t)r * H + h) * Dqk;
      double m = -INFINITY;
      for (int j = 0; j < n; ++j) {
        const double* k = kv + (int64_t)ids[j] * kv_ld;
        double dot = 0.0;
        for (int c = 0; c < Dqk; ++c) dot += qh[c] * k[c];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
      }
      double sk = sink ? sink[h] : -INFINITY;
      double* o = out + ((int64_t)r * H + h) * Dv;
      for (int c = 0; c < Dv; ++c) o[c] = 0.0;
      if (lse_indexer) {
        /* cuDNN DSA page, section 1: the LSE of the KV logits of the first
         * indexer_topk slots (valid ids only, sink excluded); +inf when
         * there are none, as for an empty row. */
        int np = 0;  /* valid ids in slots below indexer_topk */
        while (np < n && slot[np] < indexer_topk) ++np;
        double mp = -INFINITY, zp = 0.0;
        for (int j = 0; j < np; ++j)
          if (s[j] > mp) mp = s[j];
        for (int j = 0; j < np; ++j) zp += exp(s[j] - mp);
        lse_indexer[rh] = zp > 0.0 ? mp + log(zp) : INFINITY;
      }
      if (n == 0) {
        if (lse) lse[rh] = sk;
        if (lse_kv) lse_kv[rh] = INFINITY;
        if (max_logits) max_logits[rh] = -INFINITY;
        continue;
      }
      double ref = (sk > m) ? sk : m;
      double zkv = 0.0;
      for (int j = 0; j < n; ++j) {
        double p = exp(s[j] - ref);
        zkv += p;
        const double* val = v ? v + (int64_t)ids[j] * Dv : kv + (int64_t)ids[j] * kv_ld;
        for (int c = 0; c < Dv; ++c) o[c] += p * val[c];
      }
      double z = zkv + exp(sk - ref);
      for (int c = 0; c < Dv; ++c) o[c] /= z;
      if (lse) lse[rh] = ref + log(z);
      if (lse_kv) lse_kv[rh] = ref + log(zkv);
      if (max_logits) max_logits[rh] = m;
    }
    free(s);
    free(ids);
    free(slot);
  }
}

/* ------------------------------------------------------------------------
 * Sparse attention backward [P5 section 2 Sparse Attention Backward: inputs
 * q, kv (K = V, MQA), out, dout, the KV-only lse, attn_sink, topk ids and
 * lengths; outputs dq, dkv, d_sink].  With the forward of section 1 --
 * s_j = scale * q . k_j over the valid slots j, the sink in the denominator
 * only -- and L = logaddexp(lse_kv, sink) the full normaliser:
 *     P_j     = exp(s_j - L),           P_sink = exp(sink - L)
 *     dP_j    = dout . v_j,             delta  = dout . out
 *     dS_j    = P_j * (dP_j - delta)
 *     dq      = scale * sum_j dS_j k_j
 *     dkv[id_j, 0:Dqk] += scale * dS_j q ;  dkv[id_j, 0:Dv] += P_j dout
 *     d_sink  += -P_sink * delta          (summed over rows)
 * (k_j = kv[id_j, 0:Dqk], v_j = kv[id_j, 0:Dv]).  Duplicate ids are separate
 * slots and both contribute; invalid ids and slots past the length are
 * absent; a row with no valid slot contributes nothing.  dq [n_rows, H,
 * Dqk] is written; dkv [Tkv, Dqk] and dsink [H] are accumulated (the caller
 * zeroes them), rows in order.
 * ------------------------------------------------------------------------ */
void oracle_sparse_attn_bwd(const double* q_rows, const double* kv, const int32_t* idx_rows, const int32_t* len_rows,
                            const double* sink, const double* out_rows, const double* dout_rows,
                            const double* lse_kv_rows, int n_rows, int Tkv, int H, int Dqk, int Dv, int K,
                            double scale, double* dq_rows, double* dkv, double* dsink) {
  for (int r = 0; r < n_rows; ++r) {
    int lim = K;
    if (len_rows) {
      lim = len_rows[r];
      if (lim < 0) lim = 0;
      if (lim > K) lim = K;
    }
    for (int h = 0; h < H; ++h) {
      const int64_t rh = (int64_t)r * H + h;
      const double* qh = q_rows + rh * Dqk;
      const double* o = out_rows + rh * Dv;
      const double* dout = dout_rows + rh * Dv;
      double* dq = dq_rows + rh * Dqk;
      for (int c = 0; c < Dqk; ++c) dq[c] = 0.0;
      int n = 0;
      for (int j = 0; j < lim; ++j) {
        const int32_t id = idx_rows[(int64_t)r * K + j];
        if (id >= 0 && id < Tkv) ++n;
      }
      if (n == 0) continue;
      const double sk = sink ? sink[h] : -INFINITY;
      const double lkv = lse_kv_rows[rh];
      const double L = lkv > sk ? lkv + log1p(exp(sk - lkv)) : sk + log1p(exp(lkv - sk));
      double delta = 0.0;
      for (int c = 0; c < Dv; ++c) delta += dout[c] * o[c];
      for (int j = 0; j < lim; ++j) {
        const int32_t id = idx_rows[(int64_t)r * K + j];
        if (id < 0 || id >= Tkv) continue;
        const double* k = kv + (int64_t)id * Dqk;
        double dot = 0.0, dp = 0.0;
        for (int c = 0; c < Dqk; ++c) dot += qh[c] * k[c];
        for (int c = 0; c < Dv; ++c) dp += dout[c] * k[c];
        const double p = exp(scale * dot - L);
        const double ds = p * (dp - delta);
        for (int c = 0; c < Dqk; ++c) dq[c] += scale * ds * k[c];
        double* g = dkv + (int64_t)id * Dqk;
        for (int c = 0; c < Dqk; ++c) g[c] += scale * ds * qh[c];
        for (int c = 0; c < Dv; ++c) g[c] += p * dout[c];
      }
      if (dsink && sink) dsink[h] += -exp(sk - L) * delta;
    }
  }
}
