/*
 * dsa.h -- C ABI of libdsa.so, the GB300 (sm_103a) DeepSeek Sparse Attention
 * (DSA) forward hot path.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor argument is a caller-owned, contiguous, row-major DEVICE
 *    pointer on the current CUDA device.  bf16 tensors are passed as void*
 *    (IEEE bfloat16 bit patterns), fp32 as float*, ids as int32_t*.
 *  - The library never allocates, frees or synchronises.  Work is enqueued
 *    on `stream` and the call returns immediately; scratch space is passed in
 *    by the caller and sized by a query function.
 *  - All host-visible arguments are validated before anything is launched or
 *    written.  On failure nothing is enqueued and an error code is returned;
 *    dsa_last_error() then describes it.  There is no fallback path.
 *  - Values inside device tensors (ids, cu_seqlens monotonicity, lengths) are
 *    a caller contract: the kernels clamp or skip what is out of range but do
 *    not report it.  Bounded device waits that give up, and candidate buffers
 *    that overflow, set bits in the device status word (dsa_device_status).
 *  - The library looks up device addresses of its own (the status word, the
 *    scratch array of dsa_indexer_topk_noalloc) once per device and keeps
 *    them for the life of the process: a process that calls cudaDeviceReset
 *    must not use the library on that device afterwards.
 *  - Layout names follow the pages: T = total (packed THD) query tokens,
 *    H = attention heads, Hi = indexer heads, d = indexer head dim,
 *    K = top-k / sparse width, Dqk = query/key dim, Dv = value dim.
 *
 * Sources, by page and section:
 *  [cuDNN-DSA] cuDNN Frontend, "DeepSeek Sparse Attention (DSA)":
 *      1 Sparse Attention Forward, 3 Indexer Forward, 4 Combined Indexer
 *      Forward + Top-K, 5 Indexer Top-K, "Compact vs. non-compact sparse
 *      indices".
 *  [NeMo-GLM] NeMo AutoModel, nemo_automodel.components.models.glm_moe_dsa.
 *      kernels.cudnn_dsa: prepare_cudnn_dsa_packed_metadata,
 *      cudnn_indexer_topk, cudnn_sparse_attention, _compact_and_sort_indices,
 *      _topk_wrapper_chunked and the module constants.
 *  [NeMo-common] NeMo AutoModel, ...models.common.cudnn_sparse_attention.
 *  [NeMo-QSA] NeMo AutoModel, ...models.qwen3_8_flash_next.cudnn_qsa:
 *      _pack_indices, cudnn_sparse_gqa_attention.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes (the pages' ValueError / RuntimeError split, [NeMo-GLM]
 * cudnn_indexer_topk and cudnn_sparse_attention "Raises"). */
#define DSA_OK 0
#define DSA_ERR_VALUE 1        /* bad shape, size, k, scale, pointer or alignment */
#define DSA_ERR_UNSUPPORTED 2  /* no CUDA device, or the device is not sm_103 */
#define DSA_ERR_CUDA 3         /* a CUDA runtime call or launch failed */
#define DSA_ERR_WORKSPACE 4    /* workspace pointer/size too small or misaligned */

/* Bits of the device status word (see dsa_device_status). */
#define DSA_STATUS_WAIT_TIMEOUT 0x1u   /* a bounded device wait gave up */
#define DSA_STATUS_CAND_OVERFLOW 0x2u  /* fused top-k candidate buffer overflowed */
#define DSA_STATUS_DRAIN_TIMEOUT 0x4u  /* an aborting CTA gave up waiting for its own copies / MMAs */
#define DSA_STATUS_CHECK_FAILED 0x8u   /* checked build only: an in-kernel range check failed (access skipped) */

/* Limits ([NeMo-GLM] _MAX_TOPK = 2048, _INDEX_HEAD_DIM = 128,
 * _ATTENTION_HEAD_DIM = 576, _VALUE_HEAD_DIM = 512; [cuDNN-DSA] 5: top_k <= 2048). */
#define DSA_MAX_TOPK 2048
#define DSA_MAX_COMPACT_WIDTH 16384

/* Thread-local description of the last error returned on this thread
 * (empty string after a successful call).  Never NULL. */
const char* dsa_last_error(void);

/* Reads (and when clear != 0, resets) the status word of the current
 * device: an OR of DSA_STATUS_* bits set by kernels since the last clear.
 * This call synchronises the device (it is a diagnostic, not part of the
 * hot path).  Returns DSA_OK or DSA_ERR_CUDA / DSA_ERR_UNSUPPORTED. */
int dsa_device_status(uint32_t* flags, int clear);

/* Failure-detection hook (no counterpart on the pages, which only describe
 * request-or-fail validation).  Every wait of a tcgen05 / TMA kernel on an
 * mbarrier gives up after a limit, raises DSA_STATUS_WAIT_TIMEOUT, and the
 * kernel then leaves in order: the CTA's roles agree to stop at their
 * barriers, each waits (bounded by 2 s regardless of this setting) for the
 * copies and MMAs it issued, TMEM is freed and the kernel returns, so the
 * context stays usable.  This call sets that limit for kernels launched
 * afterwards on the current device: 0 restores the default (2 s, far above
 * any legitimate wait); a tiny value (e.g. 1 ns) makes the first wait that is
 * not already satisfied give up, which is how the abort path is exercised
 * without a real hang.  Outputs of a call whose kernels aborted are
 * unspecified.  Synchronises the device; call it with none of this
 * library's kernels in flight.  Returns DSA_OK or DSA_ERR_CUDA /
 * DSA_ERR_UNSUPPORTED. */
int dsa_set_wait_limit_ns(uint64_t limit_ns);

/* THD metadata ([NeMo-GLM] prepare_cudnn_dsa_packed_metadata, "Returns":
 * per-query storage starts and real causal lengths).
 *   cu_seqlens int32 [n_docs + 1]: cumulative document lengths, cu[0] = 0,
 *       cu[n_docs] = T, non-decreasing (device contract).
 *   start int32 [T] (out): first row of the token's document.
 *   len   int32 [T] (out): causal length t - start[t] + 1.
 * Errors: DSA_ERR_VALUE for n_docs < 1, T < 0 or NULL pointers (T = 0 is a
 * no-op). */
int dsa_thd_metadata(const int32_t* cu_seqlens, int n_docs, int T, int32_t* start, int32_t* len,
                     cudaStream_t stream);

/* Lightning-indexer scores, dense ([cuDNN-DSA] 3 with ratio 1 and zero causal
 * offsets; THD form of [NeMo-GLM] cudnn_indexer_topk):
 *   scores[t, j] = sum_h w[t, h] * ReLU( sum_c qi[t, h, c] * ki[start[t] + j, c] )
 * for 0 <= j < len[t] and -inf for len[t] <= j < s_max.  The head weights
 * arrive already scaled; nothing is rescaled here.
 *   qi bf16 [T, Hi, d], ki bf16 [T, d], w fp32 [T, Hi],
 *   cu_seqlens int32 [n_docs + 1] (as in dsa_thd_metadata),
 *   s_max: the longest document (host value; columns written per row),
 *   scores fp32 [T, ld] (out), ld >= s_max, ld % 4 == 0.
 * Accumulation is fp32 on the tensor cores (products of bf16 are exact).
 * Shapes: d in {64, 128}, Hi in {8, 16, 32, 64}; qi, ki 16-byte aligned.
 * Errors: DSA_ERR_VALUE on any violated shape/alignment rule. */
int dsa_indexer_scores(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens,
                       int n_docs, int T, int Hi, int d, int s_max, float* scores, int64_t ld,
                       cudaStream_t stream);

/* Per-row top-k ([cuDNN-DSA] 5 radix top-k with per-row lengths, top_k <=
 * 2048; tie-break of [cuDNN-DSA] 4 deterministic=True; compact prefix of
 * [NeMo-GLM] cudnn_sparse_attention topk_length):
 * for row t the min(k, len[t]) largest of scores[t, 0:len[t]] are selected,
 * equal scores going to the smaller column.  Their ids (row_start[t] + j, or
 * j when row_start is NULL) are written in ASCENDING id order, then -1.
 *   scores fp32 [T, ld], len int32 [T] (clamped to [0, ld]),
 *   row_start int32 [T] or NULL, idx int32 [T, k] (out),
 *   topk_length int32 [T] or NULL (out, = min(k, len[t])),
 *   vals fp32 [T, k] or NULL (out: the score of each selected slot, -inf
 *   on padding).
 * Shapes: 1 <= k <= 2048, ld >= 1; NaN scores have no defined order.
 * Errors: DSA_ERR_VALUE. */
int dsa_topk(const float* scores, int64_t ld, const int32_t* len, const int32_t* row_start, int T,
             int k, int32_t* idx, int32_t* topk_length, float* vals, cudaStream_t stream);

/* Softmax of the top-k logits ([cuDNN-DSA] 4: the combined indexer + top-k
 * returns aligned logits, their softmax and an LSE).  Over the slots of a row
 * whose id is valid (idx >= 0):
 *   lse[t] = log sum_j exp(logits[t, j]);  softmax[t, j] = exp(logits[t, j] - lse[t]);
 * slots with idx < 0 get probability 0; a row with no valid slot has lse
 * -inf and probability 0 everywhere.  fp32 arithmetic (CUDA's expf/logf).
 *   logits fp32 [T, k] (e.g. dsa_topk's vals); idx int32 [T, k] (the ids
 *   they are aligned with); softmax fp32 [T, k] or NULL (out); lse fp32 [T]
 *   or NULL (out), not both NULL.  Shapes: T >= 0, k >= 1.
 * Errors: DSA_ERR_VALUE. */
int dsa_topk_softmax(const float* logits, const int32_t* idx, int T, int k, float* softmax, float* lse,
                     cudaStream_t stream);

/* Compact and sort ([NeMo-common] _compact_and_sort_indices; [cuDNN-DSA]
 * "Compact vs. non-compact sparse indices"): per row, ids with
 * 0 <= id < key_count are sorted ascending into a prefix (duplicates kept),
 * the rest of the row is -1, lengths[t] = number of valid ids.  The id
 * convention is preserved (local stays local).
 *   in int32 [T, K], out int32 [T, K] (may alias in), lengths int32 [T].
 * Shapes: 1 <= K <= DSA_MAX_COMPACT_WIDTH, key_count >= 0.
 * Errors: DSA_ERR_VALUE. */
int dsa_compact_sort_indices(const int32_t* in, int T, int K, int64_t key_count, int32_t* out,
                             int32_t* lengths, cudaStream_t stream);

/* Workspace bytes that dsa_indexer_topk (and dsa_indexer_topk_ratio, with
 * T = Tq) needs for these shapes: 0 when T, Hi, d or s_max is below 1 or k is
 * outside [1, DSA_MAX_TOPK].  Depends on shapes only, never on data. */
size_t dsa_indexer_topk_workspace_size(int T, int Hi, int d, int k, int s_max);

/* Fused indexer + top-k ([cuDNN-DSA] 4: one call, no dense [T, S] score
 * matrix, caller-owned candidate buffer, -1 padding, deterministic
 * tie-break; stage 2 is a separate selection as in [cuDNN-DSA] "Limitations").
 * Result: identical (bit for bit) to dsa_indexer_scores followed by dsa_topk
 * with global ids (row_start = start[t]).
 *   inputs as dsa_indexer_scores; idx int32 [T, k] (out, ascending global
 *   ids, -1 suffix); topk_length int32 [T] or NULL (out);
 *   workspace: device buffer of ws_bytes >= dsa_indexer_topk_workspace_size,
 *   256-byte aligned, contents ignored on entry.
 * Errors: DSA_ERR_VALUE, DSA_ERR_WORKSPACE.  The result is exact for any
 * data: a row's candidate space never overflows, because a segment of it
 * that fills up (scores rising along the row, long runs of equal scores) is
 * cut down in place to the keys that can still reach the row's top-k.
 * DSA_STATUS_CAND_OVERFLOW is therefore never expected; if it were ever set,
 * the flagged rows would hold -1 or an inexact selection. */
int dsa_indexer_topk(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens,
                     int n_docs, int T, int Hi, int d, int k, int s_max, int32_t* idx,
                     int32_t* topk_length, void* workspace, size_t ws_bytes, cudaStream_t stream);

/* dsa_indexer_topk with the other outputs of the pages' combined indexer +
 * top-k ([cuDNN-DSA] 4): logits fp32 [T, k] (out, required): the score of
 * each selected id, aligned with idx, -inf in padded slots -- bit for bit
 * the value dsa_indexer_scores computes for that key; softmax fp32 [T, k]
 * and lse fp32 [T] (out, each may be NULL): as dsa_topk_softmax over those
 * logits.  Other arguments and results as dsa_indexer_topk.
 * Errors: as dsa_indexer_topk, plus DSA_ERR_VALUE for NULL logits and
 * DSA_ERR_UNSUPPORTED when s_max exceeds 65536 (rows that long select
 * through a form that does not keep the values). */
int dsa_indexer_topk_ex(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens,
                        int n_docs, int T, int Hi, int d, int k, int s_max, int32_t* idx,
                        int32_t* topk_length, float* logits, float* softmax, float* lse,
                        void* workspace, size_t ws_bytes, cudaStream_t stream);

/* ---- Compressed-key (ratio-causal) indexer ([cuDNN-DSA] 3 Indexer Forward
 * with ratio and q_causal_offsets; [cuDNN-DSA] 4 for the combined call).
 * Query segment b holds query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1;
 * its keys are a compressed prefix, ki rows cu_seqlens_k[b] ..
 * cu_seqlens_k[b+1]-1, starting at compressed column 0.  Local query row q
 * sees key columns
 *     j < len = clamp( floor((q_causal_offsets[b] + q + 1) / ratio), 0,
 *                      cu_seqlens_k[b+1] - cu_seqlens_k[b] ),
 * q_causal_offsets[b] being the global position of the segment's first
 * query (all 0 when the pointer is NULL; the pages require offsets >= 0,
 * a negative one only shortens rows).  ratio = 1, zero offsets and
 * cu_seqlens_k = cu_seqlens_q give the plain causal form above.
 * cu_seqlens_q / cu_seqlens_k: int32 [n_docs + 1], device, non-decreasing,
 * from 0 to Tq / Tk (not checked: the call reads no device data on the host);
 * q_causal_offsets: int32 [n_docs], device, or NULL. */

/* Per-query-row start (= cu_seqlens_k[b]) and len of the mask above.
 *   start, len int32 [T] (out).  Errors: DSA_ERR_VALUE for n_docs < 1,
 *   T < 0, ratio < 1 or NULL pointers (T = 0 is a no-op). */
int dsa_thd_metadata_ratio(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                           const int32_t* q_causal_offsets, int n_docs, int T, int ratio,
                           int32_t* start, int32_t* len, cudaStream_t stream);

/* Dense scores over the compressed keys:
 *   scores[t, j] = sum_h w[t, h] * ReLU( qi[t, h, :] . ki[start[t] + j, :] )
 * for j < min(len[t], s_max), -inf for the other columns below s_max.
 *   qi bf16 [Tq, Hi, d], ki bf16 [Tk, d], w fp32 [Tq, Hi]; s_max: a host
 *   bound on the longest row, 1 <= s_max <= Tk (rows are cut at s_max);
 *   scores fp32 [Tq, ld] (out), ld >= s_max, ld % 4 == 0.
 * Shapes and errors as dsa_indexer_scores, plus DSA_ERR_VALUE for Tk < 1,
 * ratio < 1 or NULL cu_seqlens_k. */
int dsa_indexer_scores_ratio(const void* qi, const void* ki, const float* w,
                             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                             const int32_t* q_causal_offsets, int n_docs, int Tq, int Tk, int Hi,
                             int d, int ratio, int s_max, float* scores, int64_t ld,
                             cudaStream_t stream);

/* The combined indexer + top-k over the compressed keys: identical (bit for
 * bit) to dsa_indexer_scores_ratio followed by dsa_topk with row_start =
 * start[t] and len = min(len[t], s_max), without the dense matrix.  ids are
 * global ki rows (start[t] + j), ascending, -1 suffix.
 *   idx int32 [Tq, k] (out); topk_length int32 [Tq] or NULL (out);
 *   logits fp32 [Tq, k] or NULL (out, as dsa_indexer_topk_ex); softmax fp32
 *   [Tq, k] and lse fp32 [Tq] or NULL (out; need logits);
 *   workspace: dsa_indexer_topk_workspace_size(Tq, Hi, d, k, s_max) bytes,
 *   256-byte aligned.
 * Errors: as dsa_indexer_scores_ratio, plus DSA_ERR_WORKSPACE, and
 * DSA_ERR_UNSUPPORTED for logits with s_max > 65536. */
int dsa_indexer_topk_ratio(const void* qi, const void* ki, const float* w,
                           const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                           const int32_t* q_causal_offsets, int n_docs, int Tq, int Tk, int Hi, int d,
                           int ratio, int k, int s_max, int32_t* idx, int32_t* topk_length,
                           float* logits, float* softmax, float* lse, void* workspace,
                           size_t ws_bytes, cudaStream_t stream);

/* ---- FP8 indexer inputs ([cuDNN-DSA] 3, precision path "fp8": Q and K in
 * E4M3 with fp32 descales, one per (token, head) for Q and one per key row
 * for K).  With q = e4m3(qi8[t, h, :]) and k = e4m3(ki8[s, :]):
 *   scores[t, j] = sum_h w[t, h] * ReLU( q_scale[t, h] * k_scale[s] * (q . k) ),
 *   s = start[t] + j,
 * over the row geometry of the compressed-key calls above (pass
 * cu_seqlens_k = cu_seqlens_q, no offsets and ratio 1 for the plain causal
 * form).  The products of E4M3 values are exact and accumulate in fp32 on the
 * tensor cores; the descales are applied in fp32 after the dot product
 * (q_scale folded into w, k_scale after the head sum), which is the formula
 * above for positive descales -- descales must be positive and finite, codes
 * must not be NaN (S.1111.111).
 *   qi8 uint8 [Tq, Hi, d], ki8 uint8 [Tk, d] (16-byte aligned);
 *   q_scale fp32 [Tq, Hi], k_scale fp32 [Tk]; other arguments and outputs as
 *   dsa_indexer_scores_ratio / dsa_indexer_topk_ratio.
 * Shapes: d = 128, Hi in {32, 64} (the pages' fp8 head counts).
 * Errors: as the compressed-key calls, plus DSA_ERR_VALUE for NULL descales
 * or other d / Hi. */
int dsa_indexer_scores_fp8(const void* qi8, const void* ki8, const float* q_scale, const float* k_scale,
                           const float* w, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                           const int32_t* q_causal_offsets, int n_docs, int Tq, int Tk, int Hi, int d,
                           int ratio, int s_max, float* scores, int64_t ld, cudaStream_t stream);

int dsa_indexer_topk_fp8(const void* qi8, const void* ki8, const float* q_scale, const float* k_scale,
                         const float* w, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                         const int32_t* q_causal_offsets, int n_docs, int Tq, int Tk, int Hi, int d,
                         int ratio, int k, int s_max, int32_t* idx, int32_t* topk_length, float* logits,
                         float* softmax, float* lse, void* workspace, size_t ws_bytes, cudaStream_t stream);

/* ---- MXFP8 indexer inputs ([cuDNN-DSA] 3, precision path "mxfp8": Q and K
 * in E4M3 with block-scaled E8M0 scales, sf_vec_size 32).  Each row of 128
 * codes (a (token, head) row of qi8, a key row of ki8) carries 4 scale bytes,
 * byte b = e standing for 2^(e - 127) on elements 32 b .. 32 b + 31:
 *   q[c] = e4m3(qi8[t, h, c]) * 2^(q_sf[t, h, c / 32] - 127),
 *   k[c] = e4m3(ki8[s, c])    * 2^(k_sf[s, c / 32] - 127),
 *   scores[t, j] = sum_h w[t, h] * ReLU(q . k),  s = start[t] + j,
 * over the row geometry of the compressed-key calls (plain causal form:
 * cu_seqlens_k = cu_seqlens_q, no offsets, ratio 1).  The tensor cores apply
 * the scales per 32-element block (block-scaled MMA) and accumulate in fp32;
 * products of scaled E4M3 values are exact.  Codes must not be NaN
 * (S.1111.111) and scale bytes must not be 255 (NaN).
 *   qi8 uint8 [Tq, Hi, d], ki8 uint8 [Tk, d] (16-byte aligned);
 *   q_sf uint8 [Tq, Hi, d / 32], k_sf uint8 [Tk, d / 32] (4-byte aligned):
 *   plain row-major bytes; the page's packed scale layout is its library's
 *   own and is not needed here (the kernel stages the scales itself).
 *   Other arguments and outputs as dsa_indexer_scores_ratio /
 *   dsa_indexer_topk_ratio.
 * Shapes: d = 128, Hi in {32, 64} (the pages' MXFP8 head counts).
 * Errors: as the compressed-key calls, plus DSA_ERR_VALUE for NULL or
 * misaligned scales or other d / Hi. */
int dsa_indexer_scores_mxfp8(const void* qi8, const void* ki8, const uint8_t* q_sf, const uint8_t* k_sf,
                             const float* w, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                             const int32_t* q_causal_offsets, int n_docs, int Tq, int Tk, int Hi, int d,
                             int ratio, int s_max, float* scores, int64_t ld, cudaStream_t stream);

int dsa_indexer_topk_mxfp8(const void* qi8, const void* ki8, const uint8_t* q_sf, const uint8_t* k_sf,
                           const float* w, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                           const int32_t* q_causal_offsets, int n_docs, int Tq, int Tk, int Hi, int d,
                           int ratio, int k, int s_max, int32_t* idx, int32_t* topk_length,
                           float* logits, float* softmax, float* lse, void* workspace,
                           size_t ws_bytes, cudaStream_t stream);

/* The two stages of dsa_indexer_topk as separate calls, for callers that
 * schedule or time them apart ([cuDNN-DSA] "Limitations": the selection
 * over the candidate buffer is a stage of its own).  dsa_indexer_candidates
 * followed by dsa_select_candidates on the same workspace and stream gives
 * exactly the result of dsa_indexer_topk.
 *   dsa_indexer_candidates: arguments as dsa_indexer_topk without idx and
 *   topk_length; fills the workspace with the candidate buffer (stage 1).
 *   dsa_select_candidates: cu_seqlens, n_docs, T, Hi, d, k and s_max as
 *   given to dsa_indexer_candidates (they fix the workspace layout), the
 *   workspace it filled (read only), idx and topk_length as in
 *   dsa_indexer_topk (stage 2).
 * What the workspace holds between the two calls is private to this library.
 * Errors: DSA_ERR_VALUE, DSA_ERR_WORKSPACE. */
int dsa_indexer_candidates(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens, int n_docs,
                           int T, int Hi, int d, int k, int s_max, void* workspace, size_t ws_bytes,
                           cudaStream_t stream);
int dsa_select_candidates(const int32_t* cu_seqlens, int n_docs, int T, int Hi, int d, int k, int s_max,
                          const void* workspace, size_t ws_bytes, int32_t* idx, int32_t* topk_length,
                          cudaStream_t stream);

/* Bytes of the fixed device array used by dsa_indexer_topk_noalloc (64 MiB). */
#define DSA_NOALLOC_SCRATCH_BYTES (64u << 20)

/* dsa_indexer_topk for callers that cannot allocate device memory.  (The pages
 * have no counterpart; this is a convenience of this library.)
 * Some callers cannot call cudaMalloc at all: code running inside a host
 * framework whose own allocator owns the device memory, plug-ins of
 * inference runtimes that are handed only their input and output buffers,
 * and latency-critical loops where an allocation is not allowed because
 * cudaMalloc/cudaFree may synchronise the device.  This entry point takes the
 * same arguments as dsa_indexer_topk minus the workspace; its scratch lives
 * in one file-scope device array of DSA_NOALLOC_SCRATCH_BYTES, which every GPU
 * that loads this library keeps until the process exits.  The caller still
 * owns qi, ki, w, cu_seqlens, idx and topk_length.
 *  - Shapes whose workspace (dsa_indexer_topk_workspace_size) exceeds
 *    DSA_NOALLOC_SCRATCH_BYTES are rejected with DSA_ERR_WORKSPACE before
 *    anything is launched (e.g. T = s_max = 2048 fits, T = s_max = 4096
 *    does not).
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.  The cache is not keyed on the CUDA context: after a
 *    cudaDeviceReset the array may live at another address, so a process
 *    that resets a device must not call this entry point on it again.
 *  - Every call on a device shares the one array and it keeps whatever the
 *    last call left there.  Nothing needs clearing: each word the kernels read
 *    is written earlier in the same call.  Calls that overlap on the GPU
 *    (other streams, other host threads) race on the array and corrupt each
 *    other's results: serialise them.
 *  - Results are identical to dsa_indexer_topk.  It calls no allocating
 *    routine.  Errors: as dsa_indexer_topk, plus DSA_ERR_WORKSPACE for shapes
 *    beyond the fixed size. */
int dsa_indexer_topk_noalloc(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens,
                             int n_docs, int T, int Hi, int d, int k, int s_max, int32_t* idx,
                             int32_t* topk_length, cudaStream_t stream);

/* Sparse MQA attention forward ([cuDNN-DSA] 1; THD shapes of [NeMo-GLM]
 * cudnn_sparse_attention).  For row t, head h and valid slot j (j <
 * clamp(topk_length[t], 0, K) when lengths are given, and 0 <= idx[t,j] <
 * Tkv):  s_j = scale * q[t,h,:] . kv[idx[t,j], 0:Dqk]; invalid or
 * out-of-range slots count as absent, duplicates are separate slots.
 *   Z = sum_j exp(s_j) + exp(sink[h]);  out[t,h,:] = sum_j exp(s_j) V_j / Z
 * with V_j = v[idx_j, :] when v is given, else kv[idx_j, 0:Dv].
 *   q bf16 [T, H, Dqk]; kv bf16 [Tkv, Dqk]; v bf16 [Tkv, Dv] or NULL;
 *   idx int32 [T, K]; topk_length int32 [T] or NULL; sink fp32 [H] or NULL
 *   (NULL = -inf, i.e. no sink);
 *   out bf16 [T, H, Dv] (out);
 *   lse fp32 [T, H] (out, required): log Z, the denominator out uses (sink
 *       included; empty row: sink[h], or -inf without a sink);
 *   lse_kv fp32 [T, H] or NULL (out): log sum_j exp(s_j), KV only (empty
 *       row: +inf) -- the cuDNN "lse" statistic;
 *   max_logits fp32 [T, H] or NULL (out): max_j s_j (empty row: -inf).
 * Shapes: (Dqk, Dv) in {(576, 512), (512, 512)} with v == NULL, or
 * (256, 256) with a separate v; 1 <= H <= 128; K >= 0; scale finite > 0;
 * q, kv, v, out 16-byte aligned.
 * Errors: DSA_ERR_VALUE. */
int dsa_sparse_attn_fwd(const void* q, const void* kv, const void* v, const int32_t* idx,
                        const int32_t* topk_length, const float* sink, int T, int Tkv, int H,
                        int Dqk, int Dv, int K, float scale, void* out, float* lse, float* lse_kv,
                        float* max_logits, cudaStream_t stream);

/* Sparse attention backward ([cuDNN-DSA] 2 Sparse Attention Backward; the
 * deterministic variant).  Inputs are the forward's: q bf16 [T, H, 576], the
 * latent kv bf16 [Tkv, 576] (K = V = its first 512 dims), idx / topk_length
 * as for dsa_sparse_attn_fwd, the forward's out bf16 [T, H, 512], its
 * KV-only lse_kv fp32 [T, H] (+inf for an empty row), sink fp32 [H] or
 * NULL, and dout bf16 [T, H, 512].  With s_j = scale * q . k_j over the
 * valid slots and L = logaddexp(lse_kv, sink):
 *   P_j = exp(s_j - L),  dS_j = P_j * (dout . v_j - dout . out),
 *   dq = scale * sum_j dS_j k_j                  -> dq bf16 [T, H, 576] (out)
 *   dkv[id_j] += scale * dS_j q (+ P_j dout on dims 0..511)
 *                                                -> dkv fp32 [Tkv, 576] (out)
 *   d_sink = -sum over rows of exp(sink - L) * (dout . out)
 *                                                -> d_sink fp32 [H] or NULL
 * Duplicate ids are separate slots; invalid ids and slots past topk_length
 * are absent.  P and scale * dS are rounded to bf16 for the tensor-core
 * products (as P is in the forward); every sum is fp32.  The result is
 * bitwise reproducible: dkv is accumulated in 152 fp32 copies, each written
 * by one CTA in a fixed order, and summed in a fixed order; d_sink likewise.
 *   workspace: dsa_sparse_attn_bwd_workspace_size(T, Tkv, H, K) bytes,
 *   256-byte aligned (it holds P and dS of every slot and the 152 copies).
 * Shapes: Dqk = 576, Dv = 512, 1 <= H <= 128, K >= 1, scale finite > 0;
 * q, kv, out, dout, dkv 16-byte aligned.
 * Errors: DSA_ERR_VALUE, DSA_ERR_WORKSPACE. */
size_t dsa_sparse_attn_bwd_workspace_size(int T, int Tkv, int H, int K);
int dsa_sparse_attn_bwd(const void* q, const void* kv, const void* out, const void* dout,
                        const float* lse_kv, const float* sink, const int32_t* idx,
                        const int32_t* topk_length, int T, int Tkv, int H, int Dqk, int Dv, int K,
                        float scale, void* dq, float* dkv, float* d_sink, void* workspace,
                        size_t ws_bytes, cudaStream_t stream);

/* dsa_sparse_attn_bwd with the choice between the pages' two variants
 * ([cuDNN-DSA] 2 Sparse Attention Backward, "deterministic", whose default
 * is False: dKV accumulated with fp32 atomics, not bitwise reproducible):
 *   deterministic != 0: exactly dsa_sparse_attn_bwd.
 *   deterministic == 0: every valid slot adds its dkv row into dkv with fp32
 *       atomic adds (16-byte vector reductions, served by L2); no per-SM
 *       copies, so the workspace is
 *       dsa_sparse_attn_bwd_workspace_size_ex(T, Tkv, H, K, 0) bytes (P and
 *       dS of every slot).  dq and d_sink are computed as in the
 *       deterministic variant (bitwise equal to it); dkv equals it up to the
 *       order of its fp32 additions, which varies from run to run.
 * dkv is overwritten (zeroed, then accumulated) in both variants.  Other
 * arguments, results and errors as dsa_sparse_attn_bwd. */
size_t dsa_sparse_attn_bwd_workspace_size_ex(int T, int Tkv, int H, int K, int deterministic);
int dsa_sparse_attn_bwd_ex(const void* q, const void* kv, const void* out, const void* dout,
                           const float* lse_kv, const float* sink, const int32_t* idx,
                           const int32_t* topk_length, int T, int Tkv, int H, int Dqk, int Dv, int K,
                           float scale, void* dq, float* dkv, float* d_sink, int deterministic,
                           void* workspace, size_t ws_bytes, cudaStream_t stream);

/* dsa_sparse_attn_fwd plus the indexer-prefix statistic ([cuDNN-DSA] 1,
 * outputs "lse_indexer" and compile-time "indexer_topk"):
 *   lse_indexer fp32 [T, H] (out): log sum exp(s_j) over the valid slots j <
 *       indexer_topk (KV only, sink excluded), +inf when there are none
 *       (empty row, or a prefix of invalid ids).  A row whose topk_length is
 *       below indexer_topk uses all of its valid slots (the pages require
 *       topk_length >= indexer_topk; this is the plain reading otherwise).
 *   indexer_topk: 0 (no lse_indexer; the pointer is ignored) or a multiple
 *       of 64 in [64, K] (the pages' variants use 512, 1024, 2048).
 * Other arguments, results and errors as dsa_sparse_attn_fwd; lse_indexer
 * NULL with indexer_topk > 0, or an indexer_topk outside the rule above, is
 * DSA_ERR_VALUE. */
int dsa_sparse_attn_fwd_ex(const void* q, const void* kv, const void* v, const int32_t* idx,
                           const int32_t* topk_length, const float* sink, int T, int Tkv, int H,
                           int Dqk, int Dv, int K, float scale, void* out, float* lse, float* lse_kv,
                           float* max_logits, int indexer_topk, float* lse_indexer, cudaStream_t stream);

/* One forward step from host buffers: the fused indexer + top-k
 * (dsa_indexer_topk) and sparse attention (dsa_sparse_attn_fwd, latent
 * kv of the same T rows, ids global) with the host-device copies overlapped
 * with the kernels.  Not a step of the pages' method: the path of
 * dsa_indexer_topk and dsa_sparse_attn_fwd, enqueued so that the upload of q
 * and kv runs under the indexer and the download of each of `chunks` token
 * ranges of out/lse runs under the attention of the next range.
 *   b: host inputs qi [T,Hi,d] bf16, ki [T,d] bf16, w [T,Hi], cu_seqlens
 *      [n_docs+1], q [T,H,Dqk] bf16, kv [T,Dqk] bf16, sink [H] or NULL;
 *      caller-owned device buffers of the same shapes (*_d; sink_d NULL iff
 *      sink is NULL); device results idx_d [T,k], topk_length_d [T], out_d
 *      [T,H,Dv] bf16, lse_d [T,H]; the indexer workspace (as for
 *      dsa_indexer_topk); host results idx, topk_length, out, lse.  Host
 *      buffers should be page-locked: pageable ones are still correct but
 *      their copies do not overlap.
 *   chunks: 1..16 (and <= T) token ranges for attention.
 *   compute, copy: two streams; the call enqueues on both and returns.
 *      When `compute` has finished, every result is in the host buffers.
 * Results equal those of the two device calls on the same inputs, bit for
 * bit.  Shapes as those calls (Dqk in {576, 512}, Dv = 512, no separate v).
 * Events: a fixed set per device, created by the first call on that device
 * (make it before any stream capture); a lock serialises the enqueueing of
 * calls from several host threads.  Errors: DSA_ERR_VALUE,
 * DSA_ERR_WORKSPACE, DSA_ERR_CUDA, DSA_ERR_UNSUPPORTED; every argument is
 * validated before the first copy is enqueued. */
typedef struct dsa_forward_buffers {
  const void* qi;
  const void* ki;
  const float* w;
  const int32_t* cu_seqlens;
  const void* q;
  const void* kv;
  const float* sink;
  void* qi_d;
  void* ki_d;
  float* w_d;
  int32_t* cu_seqlens_d;
  void* q_d;
  void* kv_d;
  float* sink_d;
  int32_t* idx_d;
  int32_t* topk_length_d;
  void* out_d;
  float* lse_d;
  void* workspace;
  size_t ws_bytes;
  int32_t* idx;
  int32_t* topk_length;
  void* out;
  float* lse;
} dsa_forward_buffers;

int dsa_forward_host(const dsa_forward_buffers* b, int n_docs, int T, int Hi, int d, int k, int s_max,
                     int H, int Dqk, int Dv, float scale, int chunks, cudaStream_t compute,
                     cudaStream_t copy);

/* Route packing ([NeMo-QSA] _pack_indices): routes int32 [B, S, W] hold
 * batch-local ids; out int32 [B*S, Wp] with Wp = ceil(W/4)*4 receives
 * b*S + id for 0 <= id < S and -1 otherwise (including slots W..Wp-1).
 * Shapes: B, S >= 1, 1 <= W.  Errors: DSA_ERR_VALUE. */
int dsa_pack_routes(const int32_t* routes, int B, int S, int W, int32_t* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
