// small_ops.cu -- THD metadata, route packing, compact+sort and the softmax
// of the top-k logits.
//
// These are small, latency-bound steps: one thread per element for the
// metadata and the route packing, one CTA per row for compact+sort (the row
// is sorted in shared memory with a bitonic network), one warp per row for
// the top-k softmax.
#include <climits>

#include "block_sort.cuh"
#include "common.cuh"

namespace {

// Document of token t: the largest b with cu[b] <= t (binary search).
__device__ __forceinline__ int doc_of(const int32_t* __restrict__ cu, int n_docs, int t) {
  int lo = 0, hi = n_docs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// NeMo glm_moe_dsa prepare_cudnn_dsa_packed_metadata: per-token storage start
// of its document and causal length.
__global__ void thd_metadata_kernel(const int32_t* __restrict__ cu, int n_docs, int T, int32_t* __restrict__ start,
                                    int32_t* __restrict__ len) {
  int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int s = __ldg(cu + doc_of(cu, n_docs, t));
  start[t] = s;
  len[t] = t - s + 1;
}

// cuDNN DSA page, section 3 Indexer Forward, ratio-causal mask: query segment
// b's keys start at cu_k[b]; local row q sees
// clamp((q_off[b] + q + 1) / ratio, 0, cu_k[b+1] - cu_k[b]) of them.
__global__ void ratio_metadata_kernel(const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k,
                                      const int32_t* __restrict__ q_off, int n_docs, int T, int ratio,
                                      int32_t* __restrict__ start, int32_t* __restrict__ len) {
  int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int b = doc_of(cu_q, n_docs, t);
  const int k0 = __ldg(cu_k + b);
  const int64_t nk = __ldg(cu_k + b + 1) - k0;
  const int64_t num = (q_off ? static_cast<int64_t>(__ldg(q_off + b)) : 0) + (t - __ldg(cu_q + b)) + 1;
  int64_t n = num > 0 ? num / ratio : 0;
  n = n < nk ? n : nk;
  start[t] = k0;
  len[t] = n > 0 ? static_cast<int32_t>(n) : 0;
}

// NeMo qwen3_8_flash_next.cudnn_qsa _pack_indices: batch-local ids -> packed
// coordinates b*S + id; invalid ids and the width padding become -1.
__global__ void pack_routes_kernel(const int32_t* __restrict__ routes, int S, int W, int Wp, int64_t n_out,
                                   int32_t* __restrict__ out) {
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_out) return;
  int64_t row = i / Wp;
  int j = static_cast<int>(i - row * Wp);
  int32_t v = -1;
  if (j < W) {
    int32_t id = __ldg(routes + row * W + j);
    if (id >= 0 && id < S) v = static_cast<int32_t>((row / S) * S) + id;
  }
  out[i] = v;
}

// NeMo common.cudnn_sparse_attention _compact_and_sort_indices / cuDNN DSA
// "Compact vs. non-compact sparse indices": valid ids (0 <= id < key_count)
// sorted ascending into a prefix, -1 after it, lengths = number of valid ids.
__global__ void compact_sort_kernel(const int32_t* in, int K, int P, int64_t key_count, int32_t* out,
                                    int32_t* __restrict__ lengths) {
  extern __shared__ int32_t s[];
  __shared__ int scan_scratch[32];
  const int64_t row = blockIdx.x;
  int nvalid = 0;
  for (int j = threadIdx.x; j < P; j += blockDim.x) {
    int32_t v = INT_MAX;
    if (j < K) {
      int32_t id = in[row * K + j];
      if (id >= 0 && static_cast<int64_t>(id) < key_count) {
        v = id;
        ++nvalid;
      }
    }
    s[j] = v;
  }
  int total = 0;
  dsa::block_inclusive_scan(nvalid, scan_scratch, &total);
  dsa::bitonic_sort_smem(s, P);
  for (int j = threadIdx.x; j < K; j += blockDim.x) out[row * K + j] = j < total ? s[j] : -1;
  if (threadIdx.x == 0) lengths[row] = total;
}

}  // namespace

extern "C" int dsa_thd_metadata(const int32_t* cu_seqlens, int n_docs, int T, int32_t* start, int32_t* len,
                                cudaStream_t stream) {
  dsa::clear_error();
  if (n_docs < 1 || T < 0) return dsa::set_error(DSA_ERR_VALUE, "dsa_thd_metadata: need n_docs >= 1 and T >= 0");
  if (!cu_seqlens || (T > 0 && (!start || !len)))
    return dsa::set_error(DSA_ERR_VALUE, "dsa_thd_metadata: NULL pointer");
  int rc = dsa::check_device(nullptr);
  if (rc != DSA_OK) return rc;
  if (T == 0) return DSA_OK;
  thd_metadata_kernel<<<(T + 255) / 256, 256, 0, stream>>>(cu_seqlens, n_docs, T, start, len);
  return dsa::launch_error("thd_metadata_kernel");
}

extern "C" int dsa_thd_metadata_ratio(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                      const int32_t* q_causal_offsets, int n_docs, int T, int ratio, int32_t* start,
                                      int32_t* len, cudaStream_t stream) {
  dsa::clear_error();
  if (n_docs < 1 || T < 0 || ratio < 1)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_thd_metadata_ratio: need n_docs >= 1, T >= 0, ratio >= 1");
  if (!cu_seqlens_q || !cu_seqlens_k || (T > 0 && (!start || !len)))
    return dsa::set_error(DSA_ERR_VALUE, "dsa_thd_metadata_ratio: NULL pointer");
  int rc = dsa::check_device(nullptr);
  if (rc != DSA_OK) return rc;
  if (T == 0) return DSA_OK;
  ratio_metadata_kernel<<<(T + 255) / 256, 256, 0, stream>>>(cu_seqlens_q, cu_seqlens_k, q_causal_offsets, n_docs, T,
                                                             ratio, start, len);
  return dsa::launch_error("ratio_metadata_kernel");
}

extern "C" int dsa_pack_routes(const int32_t* routes, int B, int S, int W, int32_t* out, cudaStream_t stream) {
  dsa::clear_error();
  if (B < 1 || S < 1 || W < 1) return dsa::set_error(DSA_ERR_VALUE, "dsa_pack_routes: need B, S, W >= 1");
  if (!routes || !out) return dsa::set_error(DSA_ERR_VALUE, "dsa_pack_routes: NULL pointer");
  if (static_cast<int64_t>(B) * S > INT_MAX)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_pack_routes: B*S exceeds the int32 id range");
  int rc = dsa::check_device(nullptr);
  if (rc != DSA_OK) return rc;
  const int Wp = (W + 3) / 4 * 4;
  const int64_t n = static_cast<int64_t>(B) * S * Wp;
  pack_routes_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(routes, S, W, Wp, n, out);
  return dsa::launch_error("pack_routes_kernel");
}

namespace {

// cuDNN Frontend DSA page, section 4: the softmax of a row's top-k logits and
// its log-sum-exp, over the slots whose id is valid (>= 0); other slots get
// probability 0.  One warp per row: the maximum, then the sum of exp(l - max)
// (fp32, CUDA's expf/logf), then the probabilities.  A row with no valid slot
// has lse = -inf.
__global__ void __launch_bounds__(256) topk_softmax_kernel(const float* __restrict__ logits,
                                                           const int32_t* __restrict__ idx, int T, int k,
                                                           float* __restrict__ softmax, float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* l = logits + t * k;
  const int32_t* id = idx + t * k;
  float m = -INFINITY;
  for (int j = lane; j < k; j += 32)
    if (__ldg(id + j) >= 0) m = fmaxf(m, __ldg(l + j));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.f;
  if (m > -INFINITY)
    for (int j = lane; j < k; j += 32)
      if (__ldg(id + j) >= 0) z += expf(__ldg(l + j) - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  const float lz = z > 0.f ? m + logf(z) : -INFINITY;
  if (lse && lane == 0) lse[t] = lz;
  if (softmax) {
    float* s = softmax + t * k;
    for (int j = lane; j < k; j += 32) s[j] = (z > 0.f && __ldg(id + j) >= 0) ? expf(__ldg(l + j) - lz) : 0.f;
  }
}

}  // namespace

extern "C" int dsa_topk_softmax(const float* logits, const int32_t* idx, int T, int k, float* softmax, float* lse,
                                cudaStream_t stream) {
  dsa::clear_error();
  if (T < 0 || k < 1) return dsa::set_error(DSA_ERR_VALUE, "dsa_topk_softmax: need T >= 0 and k >= 1");
  if (T > 0 && (!logits || !idx || (!softmax && !lse)))
    return dsa::set_error(DSA_ERR_VALUE, "dsa_topk_softmax: NULL logits or idx, or neither softmax nor lse");
  int rc = dsa::check_device(nullptr);
  if (rc != DSA_OK) return rc;
  if (T == 0) return DSA_OK;
  topk_softmax_kernel<<<(T + 7) / 8, 256, 0, stream>>>(logits, idx, T, k, softmax, lse);
  return dsa::launch_error("topk_softmax_kernel");
}

extern "C" int dsa_compact_sort_indices(const int32_t* in, int T, int K, int64_t key_count, int32_t* out,
                                        int32_t* lengths, cudaStream_t stream) {
  dsa::clear_error();
  if (T < 0 || K < 1 || K > DSA_MAX_COMPACT_WIDTH || key_count < 0)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_compact_sort_indices: need T >= 0, 1 <= K <= %d, key_count >= 0",
                          DSA_MAX_COMPACT_WIDTH);
  if (T > 0 && (!in || !out || !lengths)) return dsa::set_error(DSA_ERR_VALUE, "dsa_compact_sort_indices: NULL pointer");
  int rc = dsa::check_device(nullptr);
  if (rc != DSA_OK) return rc;
  if (T == 0) return DSA_OK;
  int P = 1;
  while (P < K) P <<= 1;
  const size_t smem = static_cast<size_t>(P) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(compact_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return dsa::launch_error("compact_sort_kernel smem attribute");
  }
  const int threads = P >= 512 ? 512 : (P >= 32 ? P : 32);
  compact_sort_kernel<<<T, threads, smem, stream>>>(in, K, P, key_count, out, lengths);
  return dsa::launch_error("compact_sort_kernel");
}
