// topk.cu -- per-row top-k over dense fp32 scores (cuDNN Frontend DSA page,
// section 5 Indexer Top-K: radix top-k with per-row lengths, top_k <= 2048;
// section 4 deterministic tie-break toward the smallest index).
//
// One CTA of 512 threads per row.  Rows with len <= k are copied through.
// Longer rows go through dsa::select_topk (topk_select.cuh): one histogram
// pass and one collection pass over the row in HBM/L2, the rest in shared
// memory, then an ascending sort of the k selected columns.
#include "topk_select.cuh"

namespace {

template <bool VEC4>
__global__ void __launch_bounds__(dsa::kTopkThreads)
    topk_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ len,
                const int32_t* __restrict__ row_start, int k, int32_t* __restrict__ idx,
                int32_t* __restrict__ topk_length, float* __restrict__ vals) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  dsa::TopkShared& S = *reinterpret_cast<dsa::TopkShared*>(smem_raw);
  const int64_t row = blockIdx.x;
  int n = __ldg(len + row);
  if (n < 0) n = 0;
  if (n > ld) n = static_cast<int>(ld);
  const float* r = scores + row * ld;
  const int32_t base = row_start ? __ldg(row_start + row) : 0;
  int32_t* out = idx + row * k;
  float* vout = vals ? vals + row * k : nullptr;
  if (n <= k) {
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
      out[j] = j < n ? base + j : -1;
      if (vout) vout[j] = j < n ? __ldg(r + j) : -INFINITY;
    }
    if (threadIdx.x == 0 && topk_length) topk_length[row] = n;
    return;
  }
  const dsa::DenseRowSrc<VEC4> src{r, n};
  if (n <= 32 * dsa::kBitmapWords && dsa::select_topk_sampled(S, src, n, k, n)) {
    dsa::emit_bits_ascending(S, n, [&](int pos, int j) {
      out[pos] = base + j;
      if (vout) vout[pos] = __ldg(r + j);
    });
  } else {
    dsa::select_topk(S, src, k);
    for (int i = threadIdx.x; i < k; i += blockDim.x) {
      const int j = S.sel[i];
      out[i] = base + j;
      if (vout) vout[i] = __ldg(r + j);
    }
  }
  if (threadIdx.x == 0 && topk_length) topk_length[row] = k;
}

template <bool VEC4>
int launch_topk(const float* scores, int64_t ld, const int32_t* len, const int32_t* row_start, int T, int k,
                int32_t* idx, int32_t* topk_length, float* vals, cudaStream_t stream) {
  const size_t smem = sizeof(dsa::TopkShared);
  if (cudaFuncSetAttribute(topk_kernel<VEC4>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return dsa::launch_error("topk_kernel smem attribute");
  topk_kernel<VEC4><<<T, dsa::kTopkThreads, smem, stream>>>(scores, ld, len, row_start, k, idx, topk_length, vals);
  return dsa::launch_error("topk_kernel");
}

}  // namespace

extern "C" int dsa_topk(const float* scores, int64_t ld, const int32_t* len, const int32_t* row_start, int T, int k,
                        int32_t* idx, int32_t* topk_length, float* vals, cudaStream_t stream) {
  dsa::clear_error();
  if (T < 0 || ld < 1 || k < 1 || k > DSA_MAX_TOPK)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_topk: need T >= 0, ld >= 1, 1 <= k <= %d", DSA_MAX_TOPK);
  if (ld > INT32_MAX) return dsa::set_error(DSA_ERR_VALUE, "dsa_topk: ld exceeds the int32 column range");
  if (T > 0 && (!scores || !len || !idx)) return dsa::set_error(DSA_ERR_VALUE, "dsa_topk: NULL pointer");
  int rc = dsa::check_device(nullptr);
  if (rc != DSA_OK) return rc;
  if (T == 0) return DSA_OK;
  if (ld % 4 == 0 && dsa::aligned(scores, 16))
    return launch_topk<true>(scores, ld, len, row_start, T, k, idx, topk_length, vals, stream);
  return launch_topk<false>(scores, ld, len, row_start, T, k, idx, topk_length, vals, stream);
}
