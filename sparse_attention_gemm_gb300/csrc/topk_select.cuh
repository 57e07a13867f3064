// topk_select.cuh -- block-wide exact top-k selection by radix digits.
//
// Selects, from n (key, index) pairs, the k pairs that come first under the
// order "key descending, then index ascending" (cuDNN DSA section 4,
// deterministic tie-break toward the smallest KV index) and returns their
// indices sorted ascending (the canonical compact prefix).
//
// Method: the 32-bit key is split into digits of 11, 11 and 10 bits.  A
// histogram of the top digit finds the bin that holds the k-th key; keys in
// higher bins are selected outright, keys in that bin are copied to shared
// memory (fast path) and the next digits are resolved there.  When the bin
// does not fit, the remaining digits are resolved by further passes over the
// source.  The k-th key value tau is then exact; the need_eq pairs with key
// == tau and the smallest indices are found by sorting them in shared memory
// or, when there are too many, by a second radix selection on ~index.
#pragma once

#include <climits>

#include "block_sort.cuh"
#include "common.cuh"

namespace dsa {

constexpr int kTopkThreads = 512;
constexpr int kTopkBins = 2048;
constexpr int kTopkCandCap = 8192;
constexpr int kSampleBins = 4096;     // 12-bit histogram of the sampled keys
constexpr int kSample = 2048;         // keys sampled to place the collection threshold
constexpr int kBitmapWords = 2048;    // selected-column bitmap: rows of up to 65536 columns

struct TopkShared {
  uint32_t hist[kSampleBins];
  uint32_t bits[kBitmapWords];
  uint32_t tiebits[kBitmapWords];
  int32_t sel[DSA_MAX_TOPK];
  uint32_t ckey[kTopkCandCap];
  int32_t cidx[kTopkCandCap];
  int scan[32];
  int n_sel;
  int n_cand;
  int n_eq;
  int bin;
  int above;
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Warp-aggregated histogram increment (all 32 lanes call it).
__device__ __forceinline__ void hist_add_warp(uint32_t* hist, uint32_t bin, bool active) {
  const uint32_t act = __ballot_sync(0xffffffffu, active);
  if (active) {
    const uint32_t peers = __match_any_sync(act, bin);
    if ((threadIdx.x & 31) == static_cast<uint32_t>(__ffs(peers) - 1)) atomicAdd(&hist[bin], __popc(peers));
  }
}

// Warp-aggregated append: returns the slot of this lane (or -1 when !pred).
__device__ __forceinline__ int warp_append(int* counter, bool pred) {
  const uint32_t b = __ballot_sync(0xffffffffu, pred);
  int base = 0;
  if ((threadIdx.x & 31) == 0 && b) base = atomicAdd(counter, __popc(b));
  base = __shfl_sync(0xffffffffu, base, 0);
  return pred ? base + __popc(b & lanemask_lt()) : -1;
}

__device__ __forceinline__ void hist_clear(TopkShared& S, int nbins) {
  for (int i = threadIdx.x; i < nbins; i += blockDim.x) S.hist[i] = 0;
  __syncthreads();
}

// Largest bin b with (count of bins >= b) >= k_rem; S.bin = b and S.above =
// count of bins > b.  nbins is a multiple of blockDim.x.
__device__ __forceinline__ void find_threshold_bin(TopkShared& S, int nbins, int k_rem) {
  __syncthreads();
  const int g = nbins / blockDim.x;
  const int hi = nbins - threadIdx.x * g;
  int s = 0;
  for (int b = hi - 1; b >= hi - g; --b) s += static_cast<int>(S.hist[b]);
  int total = 0;
  const int incl = block_inclusive_scan(s, S.scan, &total);
  const int excl = incl - s;
  if (excl < k_rem && incl >= k_rem) {
    int acc = excl;
    for (int b = hi - 1; b >= hi - g; --b) {
      const int c = static_cast<int>(S.hist[b]);
      if (acc + c >= k_rem) {
        S.bin = b;
        S.above = acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// Source of n (key, index) pairs visited in warp-uniform steps.  f(key, idx,
// active) is called by every lane of every warp in each step.
struct PairSrc {
  const uint32_t* key;  // may be shared or global memory
  const int32_t* idx;
  int n;
  __device__ __forceinline__ uint32_t key_at(int i) const { return key[i]; }
  template <class F>
  __device__ __forceinline__ void for_each(F&& f) const {
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + threadIdx.x;
      const bool a = i < n;
      f(a ? key[i] : 0u, a ? idx[i] : 0, a);
    }
  }
};

// Dense fp32 row: key = f32_key(row[j]), index = j.  VEC4 requires the row to
// be 16-byte aligned and readable up to round_up(n, 4).
template <bool VEC4>
struct DenseRowSrc {
  const float* row;
  int n;
  __device__ __forceinline__ uint32_t key_at(int i) const { return f32_key(__ldg(row + i)); }
  template <class F>
  __device__ __forceinline__ void for_each(F&& f) const {
    if constexpr (VEC4) {
      // four independent 16-byte loads per thread are in flight before any
      // element is processed, so a step costs one memory latency, not four
      constexpr int U = 4;
      const int step = blockDim.x * 4;
      for (int base = 0; base < n; base += step * U) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = base + u * step + threadIdx.x * 4;
          v[u] = j < n ? __ldcs(reinterpret_cast<const float4*>(row + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = base + u * step + threadIdx.x * 4;
          f(f32_key(v[u].x), j, j < n);
          f(f32_key(v[u].y), j + 1, j + 1 < n);
          f(f32_key(v[u].z), j + 2, j + 2 < n);
          f(f32_key(v[u].w), j + 3, j + 3 < n);
        }
      }
    } else {
      constexpr int U = 8;
      for (int base = 0; base < n; base += blockDim.x * U) {
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = base + u * blockDim.x + threadIdx.x;
          v[u] = j < n ? __ldcs(row + j) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int j = base + u * blockDim.x + threadIdx.x;
          f(f32_key(v[u]), j, j < n);
        }
      }
    }
  }
};

// Resolves one digit: histogram of ((key >> shift) & (nbins-1)) over pairs
// whose key matches (key & mask) == match, then the threshold bin for k_rem.
template <class Src>
__device__ __forceinline__ void digit_pass(TopkShared& S, const Src& src, uint32_t mask, uint32_t match, int shift,
                                           int nbins, int k_rem) {
  hist_clear(S, nbins);
  src.for_each([&](uint32_t key, int32_t, bool a) {
    hist_add_warp(S.hist, (key >> shift) & static_cast<uint32_t>(nbins - 1), a && ((key & mask) == match));
  });
  find_threshold_bin(S, nbins, k_rem);
}

// View of the pairs of src whose key equals tau, keyed by ~index, so that a
// top-k by key selects the smallest indices.
template <class Src>
struct TiedSrc {
  const Src& s;
  uint32_t tau;
  template <class F>
  __device__ __forceinline__ void for_each(F&& f) const {
    const uint32_t tv = tau;
    s.for_each([&](uint32_t key, int32_t idx, bool a) { f(~static_cast<uint32_t>(idx), idx, a && key == tv); });
  }
};

// Among pairs with key == tau (from src), appends the `need` smallest indices
// to S.sel.  Uses S.cidx as a sort buffer when they fit, else radix-selects
// on ~index with passes over src.
template <class Src>
__device__ void take_smallest_tied(TopkShared& S, const Src& src, uint32_t tau, int need) {
  if (need <= 0) return;
  if (threadIdx.x == 0) S.n_eq = 0;
  __syncthreads();
  src.for_each([&](uint32_t key, int32_t idx, bool a) {
    const int p = warp_append(&S.n_eq, a && key == tau);
    if (p >= 0 && p < kTopkCandCap) S.cidx[p] = idx;
  });
  __syncthreads();
  const int n_eq = S.n_eq;
  if (n_eq <= kTopkCandCap) {
    if (n_eq > need) {
      int P = 1;
      while (P < n_eq) P <<= 1;
      for (int i = n_eq + threadIdx.x; i < P; i += blockDim.x) S.cidx[i] = INT_MAX;
      bitonic_sort_smem(S.cidx, P);
    }
    for (int i = threadIdx.x; i < need; i += blockDim.x) S.sel[S.n_sel + i] = S.cidx[i];
    __syncthreads();
    if (threadIdx.x == 0) S.n_sel += need;
    __syncthreads();
    return;
  }
  // Too many ties for shared memory: radix-select the `need` largest ~index
  // (= smallest index) among the tied pairs, digit by digit over src.
  const TiedSrc<Src> tied{src, tau};
  int k_rem = need;
  digit_pass(S, tied, 0u, 0u, 21, kTopkBins, k_rem);
  uint32_t prefix = static_cast<uint32_t>(S.bin) << 21;
  k_rem -= S.above;
  digit_pass(S, tied, 0xFFE00000u, prefix, 10, kTopkBins, k_rem);
  prefix |= static_cast<uint32_t>(S.bin) << 10;
  k_rem -= S.above;
  digit_pass(S, tied, 0xFFFFFC00u, prefix, 0, 1024, k_rem);
  const uint32_t thr = prefix | static_cast<uint32_t>(S.bin);  // all ~index distinct: take >= thr
  tied.for_each([&](uint32_t nk, int32_t idx, bool a) {
    const int p = warp_append(&S.n_sel, a && nk >= thr);
    if (p >= 0) S.sel[p] = idx;
  });
  __syncthreads();
}

// Fast-path variant of take_smallest_tied: the pairs are the shared-memory
// candidates ckey/cidx [0, n_cand).  Non-tied slots of cidx are overwritten
// with INT_MAX by the thread that owns them (no cross-thread hazard); the
// tied indices are then either all taken or sorted to find the smallest.
__device__ __forceinline__ void take_smallest_tied_in_cand(TopkShared& S, uint32_t tau, int need) {
  const int n = S.n_cand;
  int mine = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    if (S.ckey[i] == tau) ++mine; else S.cidx[i] = INT_MAX;
  }
  int n_eq = 0;
  block_inclusive_scan(mine, S.scan, &n_eq);
  if (n_eq == need) {
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + threadIdx.x;
      const bool tied = i < n && S.ckey[i] == tau;
      const int p = warp_append(&S.n_sel, tied);
      if (p >= 0) S.sel[p] = S.cidx[i];
    }
    __syncthreads();
    return;
  }
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = n + threadIdx.x; i < P; i += blockDim.x) S.cidx[i] = INT_MAX;
  bitonic_sort_smem(S.cidx, P);
  const int base = S.n_sel;
  for (int i = threadIdx.x; i < need; i += blockDim.x) S.sel[base + i] = S.cidx[i];
  __syncthreads();
  if (threadIdx.x == 0) S.n_sel = base + need;
  __syncthreads();
}

// Exact top-k of src (n > k assumed, k <= DSA_MAX_TOPK).  On return
// S.sel[0 .. k) holds the selected indices sorted ascending.
template <class Src>
__device__ void select_topk(TopkShared& S, const Src& src, int k) {
  if (threadIdx.x == 0) {
    S.n_sel = 0;
    S.n_cand = 0;
  }
  // digit 1: bits 31..21
  digit_pass(S, src, 0u, 0u, 21, kTopkBins, k);
  const uint32_t b1 = static_cast<uint32_t>(S.bin);
  int k_rem = k - S.above;
  src.for_each([&](uint32_t key, int32_t idx, bool a) {
    const uint32_t bin = key >> 21;
    const int ps = warp_append(&S.n_sel, a && bin > b1);
    if (ps >= 0) S.sel[ps] = idx;
    const int pc = warp_append(&S.n_cand, a && bin == b1);
    if (pc >= 0 && pc < kTopkCandCap) {
      S.ckey[pc] = key;
      S.cidx[pc] = idx;
    }
  });
  __syncthreads();
  uint32_t tau;
  if (S.n_cand <= kTopkCandCap) {
    // fast path: the threshold bin lives in shared memory
    const PairSrc cand{S.ckey, S.cidx, S.n_cand};
    digit_pass(S, cand, 0u, 0u, 10, kTopkBins, k_rem);
    const uint32_t b2 = static_cast<uint32_t>(S.bin);
    k_rem -= S.above;
    digit_pass(S, cand, 0x001FFC00u, b2 << 10, 0, 1024, k_rem);
    tau = (b1 << 21) | (b2 << 10) | static_cast<uint32_t>(S.bin);
    k_rem -= S.above;
    // keys above tau within the bin are selected; ties are resolved in place
    cand.for_each([&](uint32_t key, int32_t idx, bool a) {
      const int p = warp_append(&S.n_sel, a && key > tau);
      if (p >= 0) S.sel[p] = idx;
    });
    __syncthreads();
    take_smallest_tied_in_cand(S, tau, k_rem);
  } else {
    digit_pass(S, src, 0xFFE00000u, b1 << 21, 10, kTopkBins, k_rem);
    const uint32_t b2 = static_cast<uint32_t>(S.bin);
    k_rem -= S.above;
    digit_pass(S, src, 0xFFFFFC00u, (b1 << 21) | (b2 << 10), 0, 1024, k_rem);
    tau = (b1 << 21) | (b2 << 10) | static_cast<uint32_t>(S.bin);
    k_rem -= S.above;
    src.for_each([&](uint32_t key, int32_t idx, bool a) {
      const int p = warp_append(&S.n_sel, a && (key >> 21) == b1 && key > tau);
      if (p >= 0) S.sel[p] = idx;
    });
    __syncthreads();
    take_smallest_tied(S, src, tau, k_rem);
  }
  // canonical order: ascending indices
  int P = 1;
  while (P < k) P <<= 1;
  for (int i = k + threadIdx.x; i < P; i += blockDim.x) S.sel[i] = INT_MAX;
  bitonic_sort_smem(S.sel, P);
}

// ---------------------------------------------------------------------------
// Faster exact path with a sampled threshold and a bitmap output.
//
// 1. A 12-bit histogram of kSample evenly spaced keys places a threshold
//    tau_s at or below the key whose sample rank is about 1.25 * k * m / n
//    (with m = n every key is sampled and tau_s is at or below the k-th key).
// 2. One pass over the source copies the pairs with key >= tau_s into shared
//    memory.  When at least k and at most kTopkCandCap were copied, tau_s is
//    at or below the k-th key (at least k keys reach it), so every member of
//    the top-k, ties included, is among the copies; otherwise the function
//    returns false and the caller runs select_topk instead.
// 3. The exact k-th key tau follows from radix digits over the copies; keys
//    above tau and the `need` smallest-index keys equal to tau are marked in
//    the column bitmap S.bits.
// The block then reads the bitmap in column order (emit_bits_ascending).
// Requires every column index < 32 * kBitmapWords.
template <class Src>
__device__ bool select_topk_sampled(TopkShared& S, const Src& src, int n, int k, int len) {
  const int m = n < kSample ? n : kSample;
  for (int i = threadIdx.x; i < kSampleBins; i += blockDim.x) S.hist[i] = 0;
  if (threadIdx.x == 0) S.n_cand = 0;
  __syncthreads();
  for (int sidx = threadIdx.x; sidx < m; sidx += blockDim.x) {
    const int pos = static_cast<int>((static_cast<int64_t>(sidx) * n) / m);
    atomicAdd(&S.hist[src.key_at(pos) >> 20], 1u);
  }
  int r = m == n ? k : static_cast<int>((static_cast<int64_t>(k) * m * 5) / (static_cast<int64_t>(n) * 4)) + 16;
  if (r > m) r = m;
  find_threshold_bin(S, kSampleBins, r);
  const uint32_t tau_s = static_cast<uint32_t>(S.bin) << 20;
  src.for_each([&](uint32_t key, int32_t idx, bool a) {
    const int pc = warp_append(&S.n_cand, a && key >= tau_s);
    if (pc >= 0 && pc < kTopkCandCap) {
      S.ckey[pc] = key;
      S.cidx[pc] = idx;
    }
  });
  __syncthreads();
  const int nc = S.n_cand;
  __syncthreads();  // every thread has read n_cand before a fallback resets it
  if (nc < k || nc > kTopkCandCap) return false;
  // exact k-th key among the copies
  const PairSrc cand{S.ckey, S.cidx, nc};
  digit_pass(S, cand, 0u, 0u, 21, kTopkBins, k);
  const uint32_t b1 = static_cast<uint32_t>(S.bin);
  int k_rem = k - S.above;
  digit_pass(S, cand, 0xFFE00000u, b1 << 21, 10, kTopkBins, k_rem);
  const uint32_t b2 = static_cast<uint32_t>(S.bin);
  k_rem -= S.above;
  digit_pass(S, cand, 0xFFFFFC00u, (b1 << 21) | (b2 << 10), 0, 1024, k_rem);
  const uint32_t tau = (b1 << 21) | (b2 << 10) | static_cast<uint32_t>(S.bin);
  const int need = k_rem - S.above;  // how many keys equal to tau are taken
  const int words = (len + 31) >> 5;
  for (int w = threadIdx.x; w < words; w += blockDim.x) {
    S.bits[w] = 0u;
    S.tiebits[w] = 0u;
  }
  __syncthreads();
  int mine_eq = 0;
  for (int i = threadIdx.x; i < nc; i += blockDim.x) {
    const uint32_t key = S.ckey[i];
    const int j = S.cidx[i];
    if (key > tau) atomicOr(&S.bits[j >> 5], 1u << (j & 31));
    else if (key == tau) {
      atomicOr(&S.tiebits[j >> 5], 1u << (j & 31));
      ++mine_eq;
    }
  }
  int n_eq = 0;
  block_inclusive_scan(mine_eq, S.scan, &n_eq);  // ends with __syncthreads
  // the `need` tied columns with the smallest indices: walk the tie bitmap in order
  const int per = (words + blockDim.x - 1) / blockDim.x;
  const int w0 = threadIdx.x * per;
  int cnt = 0;
  for (int w = w0; w < w0 + per && w < words; ++w) cnt += __popc(S.tiebits[w]);
  int total = 0;
  const int excl = block_inclusive_scan(cnt, S.scan, &total) - cnt;
  if (n_eq == need) {
    for (int w = w0; w < w0 + per && w < words; ++w) S.bits[w] |= S.tiebits[w];
  } else if (excl < need) {
    int taken = excl;
    for (int w = w0; w < w0 + per && w < words && taken < need; ++w) {
      uint32_t v = S.tiebits[w], keep = 0u;
      while (v && taken < need) {
        const uint32_t low = v & (0u - v);
        keep |= low;
        v ^= low;
        ++taken;
      }
      S.bits[w] |= keep;
    }
  }
  __syncthreads();
  return true;
}

// Calls emit(position, column) for every set bit of S.bits[0 .. words) in
// increasing column order (positions 0, 1, ...).
template <class F>
__device__ __forceinline__ void emit_bits_ascending(TopkShared& S, int len, F&& emit) {
  const int words = (len + 31) >> 5;
  const int per = (words + blockDim.x - 1) / blockDim.x;
  const int w0 = threadIdx.x * per;
  int cnt = 0;
  for (int w = w0; w < w0 + per && w < words; ++w) cnt += __popc(S.bits[w]);
  int total = 0;
  int pos = block_inclusive_scan(cnt, S.scan, &total) - cnt;
  for (int w = w0; w < w0 + per && w < words; ++w) {
    uint32_t v = S.bits[w];
    while (v) {
      const int b = __ffs(v) - 1;
      v &= v - 1;
      emit(pos++, (w << 5) + b);
    }
  }
}

}  // namespace dsa
