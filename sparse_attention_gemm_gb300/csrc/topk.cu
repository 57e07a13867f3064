// topk.cu -- per-row top-k over dense fp32 scores (cuDNN Frontend DSA page,
// section 5 Indexer Top-K: radix top-k with per-row lengths, top_k <= 2048;
// section 4 deterministic tie-break toward the smallest index).
//
// Two kernels:
//
// topk_stream_kernel (rows of at most 65536 columns, 16-byte aligned rows):
// one 256-thread CTA per row, five CTAs resident per SM (the candidates keep
// 16-bit columns and the tie bitmap shares the histogram's space, so that
// five fit and the L1 cache keeps room for the loads in flight), rows taken
// longest first.  A row is read from HBM once:
//   1. a sample of 4096 keys (512 runs of 8 adjacent columns, so that every
//      sampled 32-byte sector is one the main pass reads next) places a
//      threshold tau0 a few standard deviations below the expected k-th key;
//      rows of at most 4096 columns are sampled whole, which makes tau0 a
//      lower bound of the k-th key by construction;
//   2. one streaming pass (six 16-byte loads per thread in flight, no block
//      barrier) appends every (key, column) with key >= tau0 to a shared
//      candidate buffer, one atomic per warp; when it starts, the row's next
//      two rounds are requested into L2, and when it ends, the sampled runs
//      and first round of the row one resident wave later;
//   3. the exact k-th key follows from radix passes over the candidates' key
//      range, the last few keys ranked by one warp;
//   4. the selected columns are set in a bitmap over the row, which one block
//      scan turns into ascending ids, staged in shared memory and stored
//      coalesced.
// Histograms use plain shared-memory atomics: warp-aggregated increments
// (match.any) measured ten times slower on this GPU.  When the sample
// misjudges the row (fewer than k candidates, or more than the buffer holds,
// as with long runs of equal scores) the row falls back to exact radix
// passes over the row itself: slower, same result.
//
// topk_kernel (any other row length or alignment): one 512-thread CTA per
// row through dsa::select_topk_sampled / dsa::select_topk (topk_select.cuh).
#include "topk_select.cuh"

namespace {

// ------------------------------------------------------------ streaming form
namespace st {
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCtasPerSm = 5;              // resident CTAs per SM (shared memory and registers)
constexpr int kU = 6;                      // 16-byte loads per thread per round
constexpr int kRound = kThreads * 4 * kU;  // 6144 columns per round
constexpr int kCap = 3584;                 // candidate buffer (k <= 2048)
constexpr int kBins = 2048;
constexpr int kMaxLen = 65536;
constexpr int kWords = kMaxLen / 32;
constexpr int kWordsPer = kWords / kThreads;  // bitmap words owned by a thread
constexpr int kRuns = 512;                    // sampled runs of 8 columns
constexpr int kSample = kRuns * 8;            // 4096 keys

struct Shared {
  // The histogram is all zero after every selection pass (find_bin clears
  // the bins it reads), so once the k-th key is known its space holds the
  // bitmap of the columns tied with it.
  union {
    uint32_t hist[kBins];
    uint32_t tie[kWords];
  };
  uint32_t bits[kWords];
  // sampled keys; then candidate keys | 16-bit columns; then the staged ids
  uint32_t cbuf[kCap + kCap / 2];
  int wsum[2][kWarps];
  uint32_t wlo[kWarps], whi[kWarps];
  uint32_t lkey[32];
  int lcnt, nc, fail;
  int bin, above, cnt;
  uint32_t tau;
  int need, n_eq;
};

// Candidates in shared memory: keys and 16-bit columns (rows have at most
// 65536 columns).  Keeping the buffer small leaves room for the L1 cache,
// which holds the streaming pass's loads in flight.
static_assert(kMaxLen <= 65536, "columns are stored in 16 bits");
struct CandSrc {
  const uint32_t* key;
  const uint16_t* col;
  int n;
  template <class F>
  __device__ __forceinline__ void for_each(F&& f) const {
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + threadIdx.x;
      const bool a = i < n;
      f(a ? key[i] : 0u, a ? static_cast<int32_t>(col[i]) : 0, a);
    }
  }
};

// Exclusive block prefix of v (one barrier).  Two consecutive calls must use
// different `par`; *total receives the block sum.
__device__ __forceinline__ int excl_scan(int v, Shared& S, int par, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) S.wsum[par][warp] = incl;
  __syncthreads();
  const int x = lane < kWarps ? S.wsum[par][lane] : 0;
  int wincl = x;
#pragma unroll
  for (int o = 1; o < kWarps; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, wincl, o);
    if (lane >= o) wincl += y;
  }
  if (total) *total = __shfl_sync(0xffffffffu, wincl, kWarps - 1);
  return __shfl_sync(0xffffffffu, wincl - x, warp) + incl - v;
}

// Bins are read from the top: thread t owns bins 2047-8t down to 2040-8t.
// Finds the bin holding the r-th largest counted key; S.bin, S.above (keys
// in higher bins) and S.cnt (keys in the bin) are valid after the call.
// Every bin is zeroed on the way.  Two barriers.
__device__ __forceinline__ void find_bin(Shared& S, int r, int par) {
  const int hi = kBins - 1 - 8 * static_cast<int>(threadIdx.x);
  uint32_t c[8];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    c[i] = S.hist[hi - i];
    S.hist[hi - i] = 0u;
    sum += static_cast<int>(c[i]);
  }
  const int excl = excl_scan(sum, S, par, nullptr);
  if (excl < r && excl + sum >= r) {
    int acc = excl;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int ci = static_cast<int>(c[i]);
      if (acc < r && acc + ci >= r) {
        S.bin = hi - i;
        S.above = acc;
        S.cnt = ci;
      }
      acc += ci;
    }
  }
  __syncthreads();
}

// L2 prefetches: fire-and-forget, no registers or shared memory held.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes));
}
__device__ __forceinline__ void prefetch_l2_line(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// Bytes of columns [c0, min(c0 + cols, n)) of a 16-byte aligned row that a
// bulk prefetch may cover (a multiple of 16; 0 when nothing is left).
__device__ __forceinline__ uint32_t prefetch_bytes(int c0, int cols, int n) {
  const int c1 = c0 + cols < n ? c0 + cols : n;
  return c1 > c0 ? (static_cast<uint32_t>(c1 - c0) * 4u) & ~15u : 0u;
}

__device__ __forceinline__ uint32_t block_max(uint32_t v, Shared& S) {
  v = __reduce_max_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) S.whi[threadIdx.x >> 5] = v;
  __syncthreads();
  return __reduce_max_sync(0xffffffffu, S.whi[threadIdx.x & (kWarps - 1)]);
}

// Exact k-th largest key of src, whose keys all lie in [lo, hi]: radix
// passes of at most 11 bits over key - lo, top down; once the bin holding
// the k-th key has at most 32 keys one warp ranks them.  Sets S.tau, S.need
// (keys equal to tau that are taken) and S.n_eq (keys equal to tau).
template <class Src>
__device__ void exact_kth(Shared& S, const Src& src, int n, uint32_t lo, uint32_t hi, int k, int& par) {
  int shift = hi > lo ? 32 - __clz(hi - lo) : 0;
  uint32_t prefix = 0u, mask = 0u;
  int k_rem = k, cnt = n;
  while (shift > 0) {
    const int db = shift < 11 ? shift : 11;
    shift -= db;
    const uint32_t nb1 = (1u << db) - 1u;
    src.for_each([&](uint32_t key, int32_t, bool a) {
      const uint32_t v = key - lo;
      if (a && (v & mask) == prefix) atomicAdd(&S.hist[(v >> shift) & nb1], 1u);
    });
    __syncthreads();
    find_bin(S, k_rem, par);
    par ^= 1;
    prefix |= static_cast<uint32_t>(S.bin) << shift;
    mask |= nb1 << shift;
    k_rem -= S.above;
    cnt = S.cnt;
    if (shift > 0 && cnt <= 32) {
      if (threadIdx.x == 0) S.lcnt = 0;
      __syncthreads();
      src.for_each([&](uint32_t key, int32_t, bool a) {
        const int p = dsa::warp_append(&S.lcnt, a && ((key - lo) & mask) == prefix);
        if (p >= 0) S.lkey[p] = key;
      });
      __syncthreads();
      if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const uint32_t mine = lane < cnt ? S.lkey[lane] : 0u;
        int greater = 0, equal = 0;
        for (int j = 0; j < cnt; ++j) {
          const uint32_t o = S.lkey[j];
          greater += o > mine;
          equal += o == mine;
        }
        const bool hit = lane < cnt && greater < k_rem && k_rem <= greater + equal;
        const uint32_t hits = __ballot_sync(0xffffffffu, hit);
        if (hits && lane == __ffs(hits) - 1) {
          S.tau = mine;
          S.need = k_rem - greater;
          S.n_eq = equal;
        }
      }
      __syncthreads();
      return;
    }
  }
  if (threadIdx.x == 0) {
    S.tau = lo + prefix;
    S.need = k_rem;
    S.n_eq = cnt;
  }
  __syncthreads();
}

// Sets the bitmap bits of the selected columns of src.
template <class Src>
__device__ __forceinline__ void mark(Shared& S, const Src& src) {
  const uint32_t tau = S.tau;
  const bool all_ties = S.n_eq == S.need;
  src.for_each([&](uint32_t key, int32_t col, bool a) {
    if (!a) return;
    if (key > tau || (key == tau && all_ties)) atomicOr(&S.bits[col >> 5], 1u << (col & 31));
    else if (key == tau) atomicOr(&S.tie[col >> 5], 1u << (col & 31));
  });
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    topk_stream_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ len,
                       const int32_t* __restrict__ row_start, int T, int k, int32_t* __restrict__ idx,
                       int32_t* __restrict__ topk_length, float* __restrict__ vals, int ahead,
                       uint32_t* status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Shared& S = *reinterpret_cast<Shared*>(smem_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = T - 1 - static_cast<int64_t>(blockIdx.x);  // longest rows first when lengths grow with t
  int n = __ldg(len + row);
  if (n < 0) n = 0;
  if (n > ld) n = static_cast<int>(ld);
  const float* r = scores + row * ld;
  const int32_t base = row_start ? __ldg(row_start + row) : 0;
  int32_t* out = idx + row * k;
  float* vout = vals ? vals + row * k : nullptr;
  if (n <= k) {
    for (int j = threadIdx.x; j < k; j += kThreads) {
      out[j] = j < n ? base + j : -1;
      if (vout) vout[j] = j < n ? __ldg(r + j) : -INFINITY;
    }
    if (threadIdx.x == 0 && topk_length) topk_length[row] = n;
    return;
  }

  // ---- 1. sample -> tau0
  const int m = n < kSample ? n : kSample;
  uint32_t* const ckey = S.cbuf;
  uint16_t* const ccol = reinterpret_cast<uint16_t*>(S.cbuf + kCap);
  uint32_t* const samp = S.cbuf;  // [16][256]: key i of thread t at samp[256 * i + t]
  static_assert(kCap + kCap / 2 >= kSample, "sample does not fit the candidate buffer");
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  {
    float4 v[4];
    if (m == n) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = 16 * threadIdx.x + 4 * u;
        v[u] = j < n ? __ldg(reinterpret_cast<const float4*>(r + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int run = 2 * threadIdx.x + h;
        const int p = static_cast<int>((static_cast<int64_t>(run) * n) / kRuns) & ~3;
        v[2 * h] = __ldg(reinterpret_cast<const float4*>(r + p));
        v[2 * h + 1] = __ldg(reinterpret_cast<const float4*>(r + p + 4));
      }
    }
    const bool whole = m == n;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t key = dsa::f32_key(x[e]);
        samp[256 * (4 * u + e) + threadIdx.x] = key;
        if (!whole || 16 * static_cast<int>(threadIdx.x) + 4 * u + e < n) {
          lo = min(lo, key);
          hi = max(hi, key);
        }
      }
    }
  }
  auto svalid = [&](int i) { return m != n || 16 * static_cast<int>(threadIdx.x) + i < n; };
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  for (int i = threadIdx.x; i < kBins; i += kThreads) S.hist[i] = 0u;
  for (int i = threadIdx.x; i < kWords; i += kThreads) S.bits[i] = 0u;
  if (lane == 0) {
    S.wlo[warp] = lo;
    S.whi[warp] = hi;
  }
  if (threadIdx.x == 0) {
    S.nc = 0;
    S.fail = 0;
  }
  __syncthreads();
  lo = __reduce_min_sync(0xffffffffu, S.wlo[lane & (kWarps - 1)]);
  hi = __reduce_max_sync(0xffffffffu, S.whi[lane & (kWarps - 1)]);
  const int sbits = hi > lo ? 32 - __clz(hi - lo) : 0;
  const int sshift = sbits > 11 ? sbits - 11 : 0;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (svalid(i)) atomicAdd(&S.hist[(samp[256 * i + threadIdx.x] - lo) >> sshift], 1u);
  __syncthreads();
  int rank;
  if (m == n) {
    rank = k;  // the whole row: tau0 is at or below the k-th key
  } else {
    const double mu = static_cast<double>(k) * m / n;
    rank = static_cast<int>(ceil(mu + 4.0 * sqrt(mu))) + 2;
    if (rank > m) rank = m;
  }
  int par = 0;
  find_bin(S, rank, par);
  par ^= 1;
  uint32_t tau0 = lo + (static_cast<uint32_t>(S.bin) << sshift);
  if (sshift > 0) {
    // The sample's key range spans many octaves when small scores are
    // present, so one 11-bit pass leaves bins ~1/8 octave wide; a second pass
    // over the sampled keys inside that bin narrows tau0 to 2^-22 of the range.
    const uint32_t b1 = static_cast<uint32_t>(S.bin);
    const int rank2 = rank - S.above;
    const int sshift2 = sshift > 11 ? sshift - 11 : 0;
    const uint32_t nb1 = (1u << (sshift - sshift2)) - 1u;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t v = samp[256 * i + threadIdx.x] - lo;
      if (svalid(i) && (v >> sshift) == b1) atomicAdd(&S.hist[(v >> sshift2) & nb1], 1u);
    }
    __syncthreads();
    find_bin(S, rank2, par);
    par ^= 1;
    tau0 += static_cast<uint32_t>(S.bin) << sshift2;
  }

  // ---- 2. one pass over the row: keys >= tau0 into the candidate buffer.
  // One thread asks L2 for the next two rounds (a bulk prefetch) while the
  // first is loaded (measured: 3% faster; prefetching further rounds from
  // inside the loop cost registers and was slower).
  if (threadIdx.x == 0) {
    const uint32_t b = prefetch_bytes(kRound, 2 * kRound, n);
    if (b) prefetch_l2_bulk(r + kRound, b);
  }
  // The pass compares floats: for every non-NaN x, key(x) >= tau0 exactly
  // when x >= tau0f (the key order is the float order with -0 == +0; a
  // threshold at or below the key of -inf admits every x).  NaN scores have
  // no defined order; they are never candidates here.  Columns past the row
  // (the tail of the last float4, which is still inside the ld-wide row) are
  // dropped by one mask per round, not by a test per element (measured:
  // 4.28 -> 3.81 ms for both changes on 65536 rows of 65536 columns).
  const float tau0f = tau0 <= 0x007FFFFFu ? -INFINITY : dsa::key_f32(tau0);
  for (int b0 = 0; b0 < n; b0 += kRound) {
    float4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int j = b0 + u * (kThreads * 4) + 4 * threadIdx.x;
      v[u] = j < n ? __ldcs(reinterpret_cast<const float4*>(r + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint32_t pass = 0u;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      pass |= v[u].x >= tau0f ? 1u << (4 * u) : 0u;
      pass |= v[u].y >= tau0f ? 1u << (4 * u + 1) : 0u;
      pass |= v[u].z >= tau0f ? 1u << (4 * u + 2) : 0u;
      pass |= v[u].w >= tau0f ? 1u << (4 * u + 3) : 0u;
    }
    if (b0 + kRound > n) {  // the last round: drop the columns past the row
      uint32_t in_row = 0u;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = n - (b0 + u * (kThreads * 4) + 4 * static_cast<int>(threadIdx.x));
        in_row |= (c >= 4 ? 15u : c > 0 ? (1u << c) - 1u : 0u) << (4 * u);
      }
      pass &= in_row;
    }
    const int cnt = __popc(pass);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int wbase = 0;
    if (lane == 31 && incl) wbase = atomicAdd(&S.nc, incl);
    wbase = __shfl_sync(0xffffffffu, wbase, 31);
    if (pass) {
      int slot = wbase + incl - cnt;
      if (slot + cnt > kCap) {
        S.fail = 1;
      } else {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int j = b0 + u * (kThreads * 4) + 4 * threadIdx.x;
          const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (pass & (1u << (4 * u + e))) {
              ckey[slot] = dsa::f32_key(x[e]);
              ccol[slot] = static_cast<uint16_t>(j + e);
              ++slot;
            }
        }
      }
    }
  }
  __syncthreads();
  const int nc = S.nc;
  if (ahead > 0 && static_cast<int64_t>(blockIdx.x) + ahead < T) {
    // The block `ahead` places later (one resident wave) starts on an SM
    // about when this row ends: bring its sampled runs and first round into
    // L2 now, so that its sample phase does not wait on DRAM.
    const int64_t prow = T - 1 - (static_cast<int64_t>(blockIdx.x) + ahead);
    int pn = __ldg(len + prow);
    if (pn > ld) pn = static_cast<int>(ld);
    if (pn > k) {
      const float* pr = scores + prow * ld;
      if (pn > kSample) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int run = 2 * threadIdx.x + h;
          prefetch_l2_line(pr + (static_cast<int>((static_cast<int64_t>(run) * pn) / kRuns) & ~3));
        }
      }
      if (threadIdx.x == 0) {
        const uint32_t b = prefetch_bytes(0, kRound, pn);
        if (b) prefetch_l2_bulk(pr, b);
      }
    }
  }

  // ---- 3. exact k-th key
  if (!S.fail && nc >= k) {
    const CandSrc cand{ckey, ccol, nc};
    uint32_t mx = 0u;
    for (int i = threadIdx.x; i < nc; i += kThreads) mx = max(mx, ckey[i]);
    mx = block_max(mx, S);
    exact_kth(S, cand, nc, tau0, mx, k, par);
    mark(S, cand);
  } else {
    // the sample misjudged this row: exact passes over the row itself
    const dsa::DenseRowSrc<true> src{r, n};
    exact_kth(S, src, n, 0u, 0xFFFFFFFFu, k, par);
    mark(S, src);
  }

  // ---- 4. bitmap -> ascending ids
  const int words = (n + 31) >> 5;
  const int w0 = kWordsPer * threadIdx.x;
  uint32_t bw[kWordsPer];
  const int need = S.need;
  if (S.n_eq != need) {
    // only the `need` tied columns with the smallest indices
    uint32_t tw[kWordsPer];
    int c = 0;
#pragma unroll
    for (int i = 0; i < kWordsPer; ++i) {
      tw[i] = w0 + i < words ? S.tie[w0 + i] : 0u;
      c += __popc(tw[i]);
    }
    int taken = excl_scan(c, S, par, nullptr);
    par ^= 1;
#pragma unroll
    for (int i = 0; i < kWordsPer; ++i) {
      uint32_t t = tw[i], keep = 0u;
      while (t && taken < need) {
        const uint32_t low = t & (0u - t);
        keep |= low;
        t ^= low;
        ++taken;
      }
      if (keep) S.bits[w0 + i] |= keep;
    }
  }
  int c = 0;
#pragma unroll
  for (int i = 0; i < kWordsPer; ++i) {
    bw[i] = w0 + i < words ? S.bits[w0 + i] : 0u;
    c += __popc(bw[i]);
  }
  int pos = excl_scan(c, S, par, nullptr);
  par ^= 1;
  int32_t* staged = reinterpret_cast<int32_t*>(S.cbuf);
#pragma unroll
  for (int i = 0; i < kWordsPer; ++i) {
    uint32_t b = bw[i];
    while (b) {
      const int bit = __ffs(b) - 1;
      b &= b - 1;
      // checked build: at most k ids, staged inside the candidate buffer
      if (dsa::check(pos < k && pos < kCap + kCap / 2, status)) staged[pos] = base + ((w0 + i) << 5) + bit;
      ++pos;
    }
  }
  __syncthreads();
  if ((k & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
    const int4* s4 = reinterpret_cast<const int4*>(staged);
    int4* o4 = reinterpret_cast<int4*>(out);
    for (int i = threadIdx.x; i < (k >> 2); i += kThreads) __stcs(o4 + i, s4[i]);
  } else {
    for (int i = threadIdx.x; i < k; i += kThreads) __stcs(out + i, staged[i]);
  }
  if (vout)
    for (int i = threadIdx.x; i < k; i += kThreads) vout[i] = __ldg(r + (staged[i] - base));
  if (threadIdx.x == 0 && topk_length) topk_length[row] = k;
}
}  // namespace st

// ------------------------------------------------------------ general form
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

int launch_topk_stream(const float* scores, int64_t ld, const int32_t* len, const int32_t* row_start, int T, int k,
                       int32_t* idx, int32_t* topk_length, float* vals, int sm_count, cudaStream_t stream) {
  const size_t smem = sizeof(st::Shared);
  if (cudaFuncSetAttribute(st::topk_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return dsa::launch_error("topk_stream_kernel smem attribute");
  // kCtasPerSm CTAs are resident per SM: the block one wave later is that many SMs' worth ahead
  st::topk_stream_kernel<<<T, st::kThreads, smem, stream>>>(scores, ld, len, row_start, T, k, idx, topk_length, vals,
                                                            st::kCtasPerSm * sm_count, dsa::device_status_ptr());
  return dsa::launch_error("topk_stream_kernel");
}

}  // namespace

extern "C" int dsa_topk(const float* scores, int64_t ld, const int32_t* len, const int32_t* row_start, int T, int k,
                        int32_t* idx, int32_t* topk_length, float* vals, cudaStream_t stream) {
  dsa::clear_error();
  if (T < 0 || ld < 1 || k < 1 || k > DSA_MAX_TOPK)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_topk: need T >= 0, ld >= 1, 1 <= k <= %d", DSA_MAX_TOPK);
  if (ld > INT32_MAX) return dsa::set_error(DSA_ERR_VALUE, "dsa_topk: ld exceeds the int32 column range");
  if (T > 0 && (!scores || !len || !idx)) return dsa::set_error(DSA_ERR_VALUE, "dsa_topk: NULL pointer");
  int sm_count = 0;
  int rc = dsa::check_device(&sm_count);
  if (rc != DSA_OK) return rc;
  if (T == 0) return DSA_OK;
  const bool vec4 = ld % 4 == 0 && dsa::aligned(scores, 16);
  if (vec4 && ld <= st::kMaxLen)
    return launch_topk_stream(scores, ld, len, row_start, T, k, idx, topk_length, vals, sm_count, stream);
  if (vec4) return launch_topk<true>(scores, ld, len, row_start, T, k, idx, topk_length, vals, stream);
  return launch_topk<false>(scores, ld, len, row_start, T, k, idx, topk_length, vals, stream);
}
