// indexer.cu -- lightning-indexer scores on tcgen05 (dense and fused top-k).
//
// score[t, j] = sum_h w[t, h] * ReLU(qi[t, h, :] . ki[start[t] + j, :])
// for j < len[t] (cuDNN Frontend DSA page, section 3 Indexer Forward; THD
// shapes of NeMo glm_moe_dsa cudnn_indexer_topk; head weights arrive
// pre-scaled).  Row geometry (Geom): query segment b holds rows cu_q[b] ..
// cu_q[b+1]-1 and its keys rows cu_k[b] .. cu_k[b+1]-1 of ki; local row q
// sees key columns j < clamp((q_off[b] + q + 1) / ratio, 0, keys of b), the
// section's ratio-causal mask over a compressed key prefix.  The plain causal
// form is cu_k = cu_q, no offsets, ratio 1 (len = q + 1).
//
// Tiling ("swap AB"): one tcgen05.mma computes D[key, (token, head)] for a
// tile of 128 keys (M) against a block of QB tokens x Hi heads = 256 query
// rows (N), contracting over d (K) in steps of 16.  The accumulator lives in
// TMEM (2 x 256 fp32 columns, double-buffered) so that the epilogue of one key
// tile overlaps the MMAs of the next.  Each epilogue thread owns one key (a
// TMEM lane) and reduces over the heads of its tokens with fma(w[h],
// max(D, 0), acc) in four independent chains (head pair i in chain i % 4,
// two heads per packed fma), summed as a tree at the token's last head; its
// 128 columns arrive in four 32-column TMEM loads, each issued before the
// previous chunk is processed.  Both modes run this same instruction
// sequence, so the fused mode sees exactly the scores that the dense mode
// writes.
//
// Warp roles (320 threads; 384 in fused mode): warp 0 issues TMA loads (qi
// block once per block, ki tiles through a multi-stage ring), warp 1
// allocates TMEM and issues the MMAs, warps 2..9 run the epilogue (two warps
// per TMEM lane quarter, each on half of the 256 columns), and in fused mode
// warps 10..11 compact each finished block's candidate segments to the rows'
// final thresholds while the next block runs.  The kernel is persistent: CTA
// c handles query blocks nblocks-1-c, nblocks-1-c-grid, ... (the longest
// causal rows first).
//
// Dense mode writes scores[t, j] for j < len[t] and -inf up to s_max.
// Fused mode (cuDNN DSA section 4: no dense score matrix, caller-owned
// candidate buffer) appends (key(score), j) to row t's candidate list when
// key(score) >= tau[t], a running lower bound of the row's k-th largest key.
// tau is the lower edge of the highest histogram bin at which the emitted
// candidates so far number >= k; since the emitted keys are a subset of the
// keys seen, that edge never exceeds the final k-th largest key, so every
// member of the final top-k (ties included) is emitted.  Stage 2 then
// selects exactly from the candidates (topk.cu).
//
// Rows never overflow their candidate space.  A row's candidates sit in four
// segments, one per key quarter of a tile, each written by one warp in
// ascending key order.  When a segment could overflow on the next tile, its
// warp cuts it down to its own top-k (key descending, column ascending) and
// from then on appends only keys above the k-th key it kept: any key that k
// others of the same row beat cannot be in the row's top-k, and a later key
// that ties the k-th loses the tie to the k earlier columns.  Scores that keep
// rising along the row (every key beats the running threshold) are the case
// this exists for.
#include <climits>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "topk_select.cuh"

namespace {

constexpr int kKeyTile = 128;
constexpr int kNRows = 256;
constexpr int kEpiWarps = 8;                   // two per TMEM lane quarter
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;     // TMA warp, MMA warp, epilogue
constexpr int kCmpWarps = 2;                   // fused mode: warps compacting the previous block's candidates
constexpr int kCmpWarp0 = 2 + kEpiWarps;
constexpr int kCompactU = 8;                   // 16-byte loads per lane per compaction round
__host__ __device__ constexpr int indexer_threads(int fused) { return kThreads + (fused ? kCmpWarps * 32 : 0); }
constexpr int kSlices = kEpiWarps / 4;          // column slices of the 256 accumulator columns
constexpr int kSliceCols = kNRows / kSlices;    // columns one epilogue warp reduces per tile
constexpr int kSliceChunks = kSliceCols / 32;   // 32-column TMEM loads per tile
static_assert(kSliceChunks == 2 || kSliceChunks == 4, "a slice is 64 or 128 columns");
constexpr uint32_t kTmemCols = 512;
constexpr int kHistWords = 8192;   // 32-bit bin counters shared by the block's rows
constexpr int kTauUpdateEvery = 512;

// Which keys each query row sees (see the file comment).  Row lengths are
// also clamped to s_max, the caller's bound on the longest row.
struct Geom {
  const int32_t* cu_q;
  const int32_t* cu_k;
  const int32_t* q_off;  // or nullptr: all offsets 0
  int n_docs;
  int ratio;
  int s_max;
};

struct IndexerParams {
  const float* w;
  const float* q_scale;  // fp8 inputs: descale per (token, head) [T, Hi]
  const float* k_scale;  // fp8 inputs: descale per key row [Tk]
  const uint32_t* q_sf;  // mxfp8 inputs: E8M0 scales [T * Hi] rows of 4 bytes (one per 32 elements of d)
  const uint32_t* k_sf;  // mxfp8 inputs: E8M0 scales [Tk] rows of 4 bytes
  Geom g;
  int T;
  int Tk;
  int Hi;
  int d;
  int nch;  // 128-byte chunks per row of qi / ki (d * element bytes / 128)
  int qb;        // tokens per block = 256 / Hi
  int nblocks;
  int stages;
  // dense
  float* scores;
  int64_t ld;
  int s_max;
  // fused
  uint2* cand;        // [T][4 segments][cap/4] (key, column) pairs
  int32_t* cand_cnt;  // [T][4] candidates written per segment
  uint2* cand_tau;    // [T] the row's final threshold bin [x, y): at least k stored candidates reach x,
                      // fewer than k reach y (y = 0: x's bin is the top one)
  int cap;            // per row, a multiple of 16
  int compact;        // segments may fill up (cap below the longest row's keys per segment)
  int k;
  int hist_bits;  // log2(bins per row)
  uint32_t* status;
};

struct SmemLayout {
  uint32_t q_off, k_off, sf_off, w_off, tok_off, hist_off, row_off, cmp_off, bar_off, misc_off, total;
};

// MXFP8 block scales staged for tcgen05.cp: 512 bytes per 128-row block
// ([row % 32][row / 32][4 scale bytes]), one block per key tile of each ring
// stage, then the query block's two.
constexpr uint32_t kSfBlockBytes = 512;

__host__ __device__ inline SmemLayout smem_layout(int nch, int stages, int qb, int fused, int mx = 0) {
  SmemLayout L;
  uint32_t o = 0;
  L.q_off = o;
  o += nch * kNRows * 128;
  L.k_off = o;
  o += stages * nch * kKeyTile * 128;
  L.sf_off = o;
  if (mx) o += (stages + kNRows / 128) * kSfBlockBytes;
  L.w_off = o;
  o += kNRows * 4;
  L.tok_off = o;
  o += 2 * 32 * 4;
  L.hist_off = o;
  if (fused) o += kHistWords * 4;
  L.row_off = o;
  o += (32 + 128 + 32 + 128 + 128) * 4;  // tau, segment counts, since, segment floors, segment drops
  o += 2 * (32 + 128) * 4;               // two slots of a block's final thresholds and segment counts
  L.cmp_off = o;
  if (fused) o += kEpiWarps * 256 * 4;  // one 256-bin histogram per epilogue warp (segment compaction)
  L.bar_off = o;
  o += (2 * 8 + 9 + 4) * 8;
  L.misc_off = o;
  o += 16;
  L.total = o;
  return L;
}

__device__ __forceinline__ int doc_index(const int32_t* __restrict__ cu, int n_docs, int t) {
  int lo = 0, hi = n_docs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Drops the 128-byte L2 line at `a` (128-byte aligned) without writing it
// back; its contents become undefined.
__device__ __forceinline__ void l2_discard_line(uintptr_t a) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(a) : "memory");
}

// Keys that local row q of segment b sees in the general form (kept out of
// line: inlined into every warp role it slowed the plain form measurably).
// Returns (first key row, number of keys).
__device__ __noinline__ int2 row_len_general(const int32_t* cu_q, const int32_t* cu_k, const int32_t* q_off, int ratio,
                                             int s_max, int b, int t) {
  const int k0 = __ldg(cu_k + b);
  const int64_t nk = __ldg(cu_k + b + 1) - k0;
  const int64_t num = (q_off ? static_cast<int64_t>(__ldg(q_off + b)) : 0) + (t - __ldg(cu_q + b)) + 1;
  int64_t len = num > 0 ? num / ratio : 0;  // a non-positive bound clamps to 0 either way
  len = len < nk ? len : nk;
  len = len < s_max ? len : s_max;
  return make_int2(k0, len > 0 ? static_cast<int>(len) : 0);
}

// Number of keys query row t sees; *start receives the row of its first key.
// GEN = 0: the plain causal form (cu_k = cu_q, ratio 1, no offsets), with the
// general form compiled out: kernels that only need the plain form keep the
// plain form's code (measured: the general form compiled into the plain
// kernels slowed the dense indexer by 4-8%).
template <int GEN>
__device__ __forceinline__ int row_geom(const Geom& g, int t, int* start) {
  const int b = doc_index(g.cu_q, g.n_docs, t);
  if (!GEN) {
    // the plain causal form: one load, len = q + 1 (at most the segment, so
    // s_max only cuts rows a caller under-declared)
    const int s = __ldg(g.cu_q + b);
    *start = s;
    return min(t - s + 1, g.s_max);
  }
  const int2 r = row_len_general(g.cu_q, g.cu_k, g.q_off, g.ratio, g.s_max, b, t);
  *start = r.x;
  return r.y;
}

struct BlockRange {
  int t0, t1, kt0, kt1;
};

// Key tiles of a block of query rows: from the first row's first key to the
// last row's last key (both ends grow with the row, within and across
// segments); kt1 < kt0 when no row of the block sees a key.
template <int GEN>
__device__ __forceinline__ BlockRange block_range(const IndexerParams& p, int blk) {
  BlockRange r;
  r.t0 = blk * p.qb;
  r.t1 = min(r.t0 + p.qb, p.T);
  int s0, s1;
  row_geom<GEN>(p.g, r.t0, &s0);
  r.kt0 = s0 / kKeyTile;
  if (!GEN) {
    r.kt1 = (r.t1 - 1) / kKeyTile;  // keys stored like the queries: the last row's own key
    return r;
  }
  const int l1 = row_geom<GEN>(p.g, r.t1 - 1, &s1);
  const int end = s1 + l1;  // one past the block's last key
  r.kt1 = end > r.kt0 * kKeyTile ? (end - 1) / kKeyTile : r.kt0 - 1;
  return r;
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Cut one candidate segment (n > k pairs in ascending column order, in
// global memory) down to its top-k by (key descending, column ascending),
// keeping the column order, and return the smallest key a later (larger)
// column must reach to enter it: one above the k-th key kept.  One warp;
// hist is a 256-word scratch of this warp.  The k-th key comes from a
// four-pass radix select on 8-bit digits, the ties at it from the front.
__device__ __noinline__ uint32_t compact_segment(uint2* seg, int n, int k, uint32_t* hist) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0u, mask = 0u;
  int need = k;  // rank of the k-th key among the keys matching prefix
  __syncwarp();
  for (int shift = 24; shift >= 0; shift -= 8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) hist[lane * 8 + i] = 0u;
    __syncwarp();
    for (int b = 0; b < n; b += 32) {
      const int i = b + lane;
      const uint32_t key = i < n ? __ldcg(&seg[i].x) : 0u;
      const bool in = i < n && (key & mask) == prefix;
      const uint32_t digit = in ? (key >> shift) & 255u : 256u + lane;
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], static_cast<uint32_t>(__popc(peers)));
    }
    __syncwarp();
    // lane l sums bins 255-8l down to 248-8l; the first lane whose running
    // total from the top reaches need holds the digit
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += static_cast<int>(hist[255 - lane * 8 - i]);
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int g = __ffs(__ballot_sync(0xffffffffu, incl >= need)) - 1;
    int digit = 0, above = 0;
    if (lane == g) {
      int run = incl - s;
      for (int i = 0; i < 8; ++i) {
        const int c = static_cast<int>(hist[255 - lane * 8 - i]);
        if (run + c >= need) {
          digit = 255 - lane * 8 - i;
          above = run;
          break;
        }
        run += c;
      }
    }
    digit = __shfl_sync(0xffffffffu, digit, g);
    need -= __shfl_sync(0xffffffffu, above, g);
    prefix |= static_cast<uint32_t>(digit) << shift;
    mask |= 255u << shift;
    __syncwarp();
  }
  // keep keys above the k-th, and the first `need` keys equal to it
  int out = 0, eq_seen = 0;
  for (int b = 0; b < n; b += 32) {
    const int i = b + lane;
    const uint2 e = i < n ? __ldcg(&seg[i]) : make_uint2(0u, 0u);
    const bool eq = i < n && e.x == prefix;
    const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
    const bool keep = (i < n && e.x > prefix) || (eq && eq_seen + __popc(eqm & dsa::lanemask_lt()) < need);
    const uint32_t km = __ballot_sync(0xffffffffu, keep);
    __syncwarp();  // every lane has read this round before any lane writes
    if (keep) seg[out + __popc(km & dsa::lanemask_lt())] = e;
    out += __popc(km);
    eq_seen += __popc(eqm);
  }
  __syncwarp();
  return prefix == 0xFFFFFFFFu ? prefix : prefix + 1u;
}

// Row histogram bins: a window of 64 octaves of positive scores, [2^-32,
// 2^32), at 2^(bits-6) bins per octave (32 for 2048 bins); keys below the
// window (negative, zero and tiny scores) share bin 0 and keys above it the
// top bin.  The map is monotone in the key and hist_edge(b) is the smallest
// key that bin b holds, so the edge of a bin is a lower bound of every key
// counted at or above it.  (The leading key bits alone would give 8 bins per
// octave, and index scores typically span an octave or two.)
constexpr uint32_t kHistWindowLo = 0xAF800000u;  // the key of 2^-32
__device__ __forceinline__ uint32_t hist_bin(uint32_t key, int bits) {
  const int shift = 29 - bits;  // keeps bits - 6 mantissa bits
  const int b = static_cast<int>(key >> shift) - static_cast<int>(kHistWindowLo >> shift);
  return static_cast<uint32_t>(min(max(b, 0), (1 << bits) - 1));
}
__device__ __forceinline__ uint32_t hist_edge(int bin, int bits) {
  const int shift = 29 - bits;
  return bin == 0 ? 0u : (static_cast<uint32_t>(bin) + (kHistWindowLo >> shift)) << shift;
}

// Raise tau of one row from its histogram (one warp, one 32-bit counter per
// bin): find the highest bin b at which the counts of bins >= b reach k and
// set tau to b's lower edge (only ever raised).  Bins below the current
// tau's bin cannot give a higher edge, so only bins from that one up are
// read.  Two warp scans: first over 32 contiguous groups of those bins
// (lane 0 = highest), then over the bins of the crossing group spread across
// the lanes.
__device__ __forceinline__ void update_tau(const uint32_t* hist_row, int bins, int hist_bits, int k, uint32_t* tau) {
  const int lane = threadIdx.x & 31;
  const int b_lo = static_cast<int>(hist_bin(*reinterpret_cast<volatile uint32_t*>(tau), hist_bits));
  int per = 1;  // bins per group, a power of two; group 0 holds the highest bins
  while (per * 32 < bins - b_lo) per <<= 1;
  const int b_hi = bins - lane * per;
  int s = 0;
  // the sum does not depend on order: start each lane at a different offset so
  // that the lanes spread over the banks
  for (int j = 0; j < per; ++j) {
    const int bi = b_hi - 1 - ((j + lane) & (per - 1));
    if (bi >= b_lo) s += static_cast<int>(hist_row[bi]);
  }
  int incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t hit = __ballot_sync(0xffffffffu, incl >= k);
  if (hit == 0u) return;               // fewer than k candidates at or above tau's bin so far
  const int g = __ffs(hit) - 1;        // crossing group
  int before = __shfl_sync(0xffffffffu, incl - s, g);
  // bins of group g, top down, spread over the lanes in rounds of 32
  const int g_hi = bins - g * per;
  for (int r0 = 0; r0 < per; r0 += 32) {
    const int bi = g_hi - 1 - r0 - lane;  // lane 0 takes the highest bin of the round
    const int c = (r0 + lane < per && bi >= b_lo) ? static_cast<int>(hist_row[bi]) : 0;  // groups narrower than 32
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const uint32_t h2 = __ballot_sync(0xffffffffu, before + inc >= k);
    if (h2 != 0u) {
      if (lane == __ffs(h2) - 1) {
        const uint32_t t = hist_edge(bi, hist_bits);
        volatile uint32_t* vt = tau;
        if (t > *vt) *vt = t;
      }
      break;
    }
    before += __shfl_sync(0xffffffffu, inc, 31);
  }
  __syncwarp();
}

// F8 = 1: qi / ki are E4M3 with fp32 descales (kind::f8f6f4 MMAs, K = 32
// per instruction, so a 128-byte chunk is still four instructions); the
// epilogue folds q_scale into the head weights and multiplies the head sum
// by k_scale: w * ReLU(qs * ks * D) = ks * (w * qs) * ReLU(D) for positive
// descales.
// F8 = 2: qi / ki are E4M3 with E8M0 scales per 32 elements of d (MXFP8).
// The block-scaled MMA (kind::mxf8f6f4, one instruction per 32-element block)
// applies them: the whole TMA warp stages each key tile's and query block's
// scale bytes in shared memory in the layout tcgen05.cp expects, the MMA
// thread copies them to TMEM before the tile's MMAs (in issue order), and the
// epilogue is the bf16 one.  The scale columns take the TMEM room of the second
// accumulator, so the accumulator is single-buffered.
template <int FUSED, int HI, int GEN, int F8>
__global__ void __launch_bounds__(indexer_threads(FUSED), 1)
    indexer_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const IndexerParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dsa::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  constexpr bool MX = F8 == 2;
  // MX: the accumulator is a ring of three 128-column half-tiles (half s of
  // tile g is half-tile j = 2g + s, slot j % 3, read by the epilogue warps of
  // column slice s), and the block scales take the columns after it, two
  // buffers each (key tile by tile parity, query block by block parity).
  constexpr int kMxSlots = 3;
  constexpr uint32_t kSfaCol = 3 * 128, kSfbCol = kSfaCol + 8;  // MX: A 2 x 4, B 2 x 8 columns
  const SmemLayout L = smem_layout(p.nch, p.stages, p.qb, FUSED, MX);
  uint8_t* qbuf = smem + L.q_off;
  uint8_t* kbuf = smem + L.k_off;
  uint8_t* sfbuf = smem + L.sf_off;  // MX: [stage] key-tile scales, then the query block's
  float* w_s = reinterpret_cast<float*>(smem + L.w_off);
  int32_t* tok_start = reinterpret_cast<int32_t*>(smem + L.tok_off);
  int32_t* tok_len = tok_start + 32;
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + L.hist_off);
  uint32_t* row_tau = reinterpret_cast<uint32_t*>(smem + L.row_off);
  int32_t* seg_cnt = reinterpret_cast<int32_t*>(row_tau + 32);  // [32 rows][4 segments], one writer each
  int32_t* row_since = seg_cnt + 128;  // candidate count at the row's last tau update (owner warp only)
  uint32_t* seg_floor = reinterpret_cast<uint32_t*>(row_since + 32);  // [32][4] entry floor after a compaction
  int32_t* seg_drop = reinterpret_cast<int32_t*>(seg_floor + 128);    // [32][4] candidates dropped by compactions
  // [2 slots]: a finished block's final threshold per row [32] and stored
  // candidates per (row, segment) [32][4], handed from the epilogue to the
  // compaction warps (slot = the block's parity within this CTA)
  uint32_t* pend_x = reinterpret_cast<uint32_t*>(seg_drop + 128);
  int32_t* pend_n = reinterpret_cast<int32_t*>(pend_x + 2 * 32);
  uint32_t* cmp_hist = reinterpret_cast<uint32_t*>(smem + L.cmp_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* full = bars;
  uint64_t* empty = bars + 8;
  uint64_t* qfull = bars + 16;
  uint64_t* qempty = bars + 17;
  uint64_t* tfull = bars + 18;   // [2] ([3] for MX)
  uint64_t* tempty = bars + 21;  // [2] ([3] for MX)
  uint64_t* drain = bars + 24;   // the MMA issuer's exit commit
  uint64_t* pend_full = bars + 25;   // [2] a slot holds a finished block (all epilogue warps)
  uint64_t* pend_empty = bars + 27;  // [2] the compaction warps are done with a slot
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = p.nch;
  constexpr int kChunkElems = F8 ? 128 : 64;  // elements per 128-byte chunk
  const int S = p.stages;

  if (threadIdx.x == 0) {
    // MX: a tile (query block) is ready when its TMA bytes landed and the
    // producer warp staged its scales: two arrivals
    for (int s = 0; s < S; ++s) {
      dsa::mbar_init(&full[s], MX ? 2 : 1);
      dsa::mbar_init(&empty[s], 1);
    }
    dsa::mbar_init(qfull, MX ? 2 : 1);
    dsa::mbar_init(qempty, 1);
    // an accumulator is drained by every epilogue warp; an MX half-tile slot
    // by the four warps of its column slice
    for (int b = 0; b < (MX ? kMxSlots : 2); ++b) {
      dsa::mbar_init(&tfull[b], 1);
      dsa::mbar_init(&tempty[b], MX ? kEpiWarps / kSlices : kEpiWarps);
    }
    dsa::mbar_init(drain, 1);
    for (int b = 0; b < 2; ++b) {
      dsa::mbar_init(&pend_full[b], kEpiWarps);
      dsa::mbar_init(&pend_empty[b], kCmpWarps);
    }
    *abort_flag = 0;
    dsa::fence_barrier_init();
  }
  if (warp == 1) dsa::tmem_alloc(tmem_slot, kTmemCols);
  dsa::tc_fence_before();
  __syncthreads();
  dsa::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const dsa::Waiter wt = dsa::make_waiter(abort_flag, p.status);

  if (warp == 0) {
    if constexpr (MX) {
      // ------------------------------------------ TMA producer (MX: whole warp)
      // Lane 0 issues the TMA loads; all 32 lanes stage the scale bytes of
      // each query block and key tile, and lane 0 then arrives a second time.
      if (lane == 0) {
        dsa::tma_prefetch_desc(&map_q);
        dsa::tma_prefetch_desc(&map_k);
      }
      const uint64_t keep = dsa::l2_policy_evict_last();
      const uint64_t stream = dsa::l2_policy_evict_first();
      // scale rows [row0, row0 + 128 nblk) -> nblk staged blocks at dst: lane r
      // writes the 16 bytes of rows r, r + 32, r + 64, r + 96 of each block
      auto stage_scales = [&](uint8_t* dst, const uint32_t* src, int64_t row0, int nblk, int64_t rows) {
        dsa::fence_proxy_async_smem();  // the slot's last reader was tcgen05.cp (async proxy)
        for (int h = 0; h < nblk; ++h) {
          uint32_t v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int64_t r = row0 + 128 * h + 32 * q + lane;
            v[q] = r < rows ? __ldg(src + r) : 0x7F7F7F7Fu;  // past the end: scale 1 on zero-filled codes
          }
          *reinterpret_cast<uint4*>(dst + h * kSfBlockBytes + lane * 16) = make_uint4(v[0], v[1], v[2], v[3]);
        }
        dsa::fence_proxy_async_smem();  // generic writes -> tcgen05.cp (async proxy)
        __syncwarp();
      };
      int stage = 0;
      uint32_t phase = 0;
      int iter = 0;
      bool ok = true;
      int n_issued = 0;  // key-tile loads issued: load i went to stage i % S, phase (i / S) & 1
      int q_issued = 0;  // query-block loads issued: load m completes phase m of qfull
      for (int blk = p.nblocks - 1 - blockIdx.x; blk >= 0 && ok; blk -= gridDim.x, ++iter) {
        const BlockRange br = block_range<GEN>(p, blk);
        if (iter > 0 && !dsa::mbar_wait_warp(qempty, (iter - 1) & 1, wt)) { ok = false; break; }
        if (lane == 0) {
          dsa::mbar_expect_tx(qfull, nch * kNRows * 128);
          for (int c = 0; c < nch; ++c)
            dsa::tma_load_2d_hint(qbuf + c * kNRows * 128, &map_q, c * kChunkElems, br.t0 * p.Hi, qfull, stream);
        }
        ++q_issued;
        stage_scales(sfbuf + S * kSfBlockBytes, p.q_sf, static_cast<int64_t>(br.t0) * p.Hi, kNRows / 128,
                     static_cast<int64_t>(p.T) * p.Hi);
        if (lane == 0) dsa::mbar_arrive(qfull);
        for (int kt = br.kt0; kt <= br.kt1; ++kt) {
          if (!dsa::mbar_wait_warp(&empty[stage], phase ^ 1, wt)) { ok = false; break; }
          if (lane == 0) {
            dsa::mbar_expect_tx(&full[stage], nch * kKeyTile * 128);
            uint8_t* dst = kbuf + stage * nch * kKeyTile * 128;
            for (int c = 0; c < nch; ++c)
              dsa::tma_load_2d_hint(dst + c * kKeyTile * 128, &map_k, c * kChunkElems, kt * kKeyTile, &full[stage],
                                    keep);
          }
          stage_scales(sfbuf + stage * kSfBlockBytes, p.k_sf, static_cast<int64_t>(kt) * kKeyTile, 1, p.Tk);
          if (lane == 0) dsa::mbar_arrive(&full[stage]);
          ++n_issued;
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
      if (lane == 0) {  // drain, as below
        if (q_issued > 0) dsa::mbar_drain(qfull, (q_issued - 1) & 1, p.status);
        for (int j = 1; j <= n_issued && j <= S; ++j) {
          const int i = n_issued - j;
          dsa::mbar_drain(&full[i % S], (i / S) & 1, p.status);
        }
      }
      __syncwarp();
    } else if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      dsa::tma_prefetch_desc(&map_q);
      dsa::tma_prefetch_desc(&map_k);
      // key tiles are re-read by every query block; query blocks are read once
      const uint64_t keep = dsa::l2_policy_evict_last();
      const uint64_t stream = dsa::l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      int iter = 0;
      bool ok = true;
      int n_issued = 0;  // key-tile loads issued: load i went to stage i % S, phase (i / S) & 1
      int q_issued = 0;  // query-block loads issued: load m completes phase m of qfull
      for (int blk = p.nblocks - 1 - blockIdx.x; blk >= 0 && ok; blk -= gridDim.x, ++iter) {
        const BlockRange br = block_range<GEN>(p, blk);
        if (iter > 0 && !dsa::mbar_wait(qempty, (iter - 1) & 1, wt)) { ok = false; break; }
        dsa::mbar_expect_tx(qfull, nch * kNRows * 128);
        for (int c = 0; c < nch; ++c)
          dsa::tma_load_2d_hint(qbuf + c * kNRows * 128, &map_q, c * kChunkElems, br.t0 * p.Hi, qfull, stream);
        ++q_issued;
        for (int kt = br.kt0; kt <= br.kt1; ++kt) {
          if (!dsa::mbar_wait(&empty[stage], phase ^ 1, wt)) { ok = false; break; }
          dsa::mbar_expect_tx(&full[stage], nch * kKeyTile * 128);
          uint8_t* dst = kbuf + stage * nch * kKeyTile * 128;
          for (int c = 0; c < nch; ++c)
            dsa::tma_load_2d_hint(dst + c * kKeyTile * 128, &map_k, c * kChunkElems, kt * kKeyTile, &full[stage], keep);
          ++n_issued;
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
      // Every copy this thread issued has landed before the CTA leaves (all of
      // them were consumed unless the kernel aborted): the newest query block
      // and the newest load of each ring stage (a stage or the query buffer is
      // reloaded only after its previous load was consumed).
      if (q_issued > 0) dsa::mbar_drain(qfull, (q_issued - 1) & 1, p.status);
      for (int j = 1; j <= n_issued && j <= S; ++j) {
        const int i = n_issued - j;
        dsa::mbar_drain(&full[i % S], (i / S) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    if (MX && lane == 0) {
      // ------------------------------------------- MMA issuer (MX: block scales)
      const uint32_t q_addr = dsa::smem_u32(qbuf), k_addr = dsa::smem_u32(kbuf), sf_addr = dsa::smem_u32(sfbuf);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t j = 0;  // half-tiles issued
      uint32_t g = 0;  // tiles issued
      int iter = 0;
      bool ok = true;
      for (int blk = p.nblocks - 1 - blockIdx.x; blk >= 0 && ok; blk -= gridDim.x, ++iter) {
        const BlockRange br = block_range<GEN>(p, blk);
        if (!dsa::mbar_wait(qfull, iter & 1, wt)) break;
        dsa::tc_fence_after();
        const uint32_t sfb = kSfbCol + 8 * (iter & 1);
        for (int kt = br.kt0; kt <= br.kt1 && ok; ++kt, ++g) {
          if (!dsa::mbar_wait(&full[stage], phase, wt)) { ok = false; break; }
          const uint32_t sfa = kSfaCol + 4 * (g & 1);
          const uint32_t a0 = k_addr + stage * nch * kKeyTile * 128;
          for (int h = 0; h < kSlices; ++h, ++j) {
            const uint32_t slot = j % kMxSlots;
            // the slot's last reader (three half-tiles back) is done: so is every
            // MMA before it, hence the scale buffers two tiles / one block back
            if (!dsa::mbar_wait(&tempty[slot], ((j / kMxSlots) & 1) ^ 1, wt)) { ok = false; break; }
            dsa::tc_fence_after();
            if (h == 0) {
              if (kt == br.kt0) {  // the query block's scales, 2 x 128 rows
                dsa::tmem_cp_32x128b_x4(tmem_base + sfb, dsa::smem_desc(sf_addr + S * kSfBlockBytes, 128, 128, 0));
                dsa::tmem_cp_32x128b_x4(tmem_base + sfb + 4,
                                        dsa::smem_desc(sf_addr + (S + 1) * kSfBlockBytes, 128, 128, 0));
              }
              dsa::tmem_cp_32x128b_x4(tmem_base + sfa, dsa::smem_desc(sf_addr + stage * kSfBlockBytes, 128, 128, 0));
            }
            // half h: the 128 query rows of column slice h against the 128 keys
            const uint32_t b0 = q_addr + h * (kNRows / kSlices) * 128;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {  // one instruction per 32-element scale block of d = 128
              const uint64_t ad = dsa::smem_desc(a0 + kk * 32, 16, 1024, dsa::kSwizzle128B);
              const uint64_t bd = dsa::smem_desc(b0 + kk * 32, 16, 1024, dsa::kSwizzle128B);
              dsa::umma_mxf8(tmem_base + slot * 128, ad, bd, dsa::idesc_mxf8(kKeyTile, kNRows / kSlices, kk, kk),
                             tmem_base + sfa, tmem_base + sfb + 4 * h, kk != 0);
            }
            dsa::umma_commit(&tfull[slot]);
          }
          if (!ok) break;
          dsa::umma_commit(&empty[stage]);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        dsa::umma_commit(qempty);
      }
      dsa::umma_drain(drain, p.status);  // every MMA and copy issued has completed
    } else if (lane == 0) {
      // ------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = F8 ? dsa::idesc_e4m3(kKeyTile, kNRows) : dsa::idesc_bf16(kKeyTile, kNRows, 0, 0);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int iter = 0;
      bool ok = true;
      const uint32_t q_addr = dsa::smem_u32(qbuf), k_addr = dsa::smem_u32(kbuf);
      for (int blk = p.nblocks - 1 - blockIdx.x; blk >= 0 && ok; blk -= gridDim.x, ++iter) {
        const BlockRange br = block_range<GEN>(p, blk);
        if (!dsa::mbar_wait(qfull, iter & 1, wt)) break;
        dsa::tc_fence_after();
        for (int kt = br.kt0; kt <= br.kt1; ++kt) {
          if (!dsa::mbar_wait(&tempty[acc], acc_phase ^ 1, wt)) { ok = false; break; }
          if (!dsa::mbar_wait(&full[stage], phase, wt)) { ok = false; break; }
          dsa::tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * kNRows;
          const uint32_t a0 = k_addr + stage * nch * kKeyTile * 128;
          for (int c = 0; c < nch; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = dsa::smem_desc(a0 + c * kKeyTile * 128 + kk * 32, 16, 1024, dsa::kSwizzle128B);
              const uint64_t bd = dsa::smem_desc(q_addr + c * kNRows * 128 + kk * 32, 16, 1024, dsa::kSwizzle128B);
              if (F8) dsa::umma_f8(d_tmem, ad, bd, idesc, (c | kk) != 0);
              else dsa::umma_bf16(d_tmem, ad, bd, idesc, (c | kk) != 0);
            }
          }
          dsa::umma_commit(&empty[stage]);
          dsa::umma_commit(&tfull[acc]);
          if (++stage == S) { stage = 0; phase ^= 1; }
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
        dsa::umma_commit(qempty);
      }
      dsa::umma_drain(drain, p.status);  // every MMA issued has completed
    }
  } else if (warp < kCmpWarp0) {
    // -------------------------------------------------------- epilogue
    const int ew = warp - 2;                  // 0 .. kEpiWarps-1
    const int quarter = warp & 3;             // TMEM lane quarter of this warp
    const int slice = ew >> 2;                // column slice: 0 .. kSlices-1
    const int et = threadIdx.x - 64;          // 0..255
    const int key_lane = quarter * 32 + lane; // key within the tile
    constexpr int QB = kNRows / HI;
    constexpr int tok_per_slice = QB / kSlices;  // tokens of one column slice
    const int Hi = HI;
    const int hist_words_row = FUSED ? (kHistWords / QB) : 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t jh = static_cast<uint32_t>(slice);  // MX: this warp's half-tiles are 2g + slice
    bool ok = true;
    // A wait of this thread gave up.  The thread carries on through the
    // block's tiles (its TMEM loads stay in the allocation, its stores in the
    // outputs and candidate segments, so the garbage it may compute is
    // harmless in a kernel that is aborting, and no collective instruction
    // sees a diverged warp); the eight warps leave together at the block's
    // last barrier, which reduces the flag over the group.
    bool failed = false;
    const int seg = quarter;              // this warp writes segment `quarter` of its rows
    const int cap_seg = FUSED ? p.cap / 4 : 0;
    uint32_t blk_i = 0;                   // blocks finished by this CTA (slot of the hand-over)
    for (int blk = p.nblocks - 1 - blockIdx.x; blk >= 0 && ok; blk -= gridDim.x) {
      const BlockRange br = block_range<GEN>(p, blk);
      uint32_t cmask = 0u;                 // bit q: this warp's segment of row q was compacted
      int wcnt[tok_per_slice];              // candidates this warp wrote per row (warp-uniform)
#pragma unroll
      for (int q = 0; q < tok_per_slice; ++q) wcnt[q] = 0;
      named_bar(1, kEpiThreads);  // previous block's readers of w_s / tok_* are done
      for (int i = et; i < kNRows; i += kEpiThreads) {
        const int r = i / HI, h = i - r * HI;
        const int t = br.t0 + r;
        float wv = t < p.T ? __ldg(p.w + static_cast<int64_t>(t) * Hi + h) : 0.f;
        if (F8 == 1 && t < p.T) wv *= __ldg(p.q_scale + static_cast<int64_t>(t) * Hi + h);
        w_s[i] = wv;
      }
      if (et < p.qb) {
        const int t = br.t0 + et;
        if (t < p.T) {
          int s;
          tok_len[et] = row_geom<GEN>(p.g, t, &s);
          tok_start[et] = s;
        } else {
          tok_start[et] = INT_MAX;
          tok_len[et] = 0;
        }
        if (FUSED) {
          row_tau[et] = 0u;
          row_since[et] = 0;
#pragma unroll
          for (int sg = 0; sg < 4; ++sg) {
            seg_cnt[et * 4 + sg] = 0;
            seg_floor[et * 4 + sg] = 0u;
            seg_drop[et * 4 + sg] = 0;
          }
        }
      }
      if (FUSED)
        for (int i = et; i < kHistWords; i += kEpiThreads) hist[i] = 0u;
      named_bar(1, kEpiThreads);
      // this thread's rows (tokens slice*tok_per_slice + q): key window
      // [rs, rs + rl) in registers, so the per-token check needs no load
      int rs[tok_per_slice], rl[tok_per_slice];
#pragma unroll
      for (int q = 0; q < tok_per_slice; ++q) {
        rs[q] = tok_start[slice * tok_per_slice + q];
        rl[q] = tok_len[slice * tok_per_slice + q];
      }

      // fp8: this thread's key descale, loaded one tile ahead
      float ks_next = 1.f;
      if (F8 == 1) {
        const int s0 = br.kt0 * kKeyTile + key_lane;
        ks_next = s0 < p.Tk ? __ldg(p.k_scale + s0) : 0.f;
      }
      for (int kt = br.kt0; kt <= br.kt1; ++kt) {
        const float ks = ks_next;
        if (F8 == 1) {
          const int s1 = (kt + 1) * kKeyTile + key_lane;
          ks_next = (kt < br.kt1 && s1 < p.Tk) ? __ldg(p.k_scale + s1) : 0.f;
        }
        // the accumulator (or, MX, this slice's half-tile slot) of this tile
        uint32_t slot = static_cast<uint32_t>(acc), slot_phase = acc_phase;
        if constexpr (MX) {
          slot = jh % kMxSlots;
          slot_phase = (jh / kMxSlots) & 1;
        }
        if (!failed) failed = !dsa::mbar_wait(&tfull[slot], slot_phase, wt);
        dsa::tc_fence_after();
        const int s_key = kt * kKeyTile + key_lane;  // absolute key row
        // this warp's columns [slice*kSliceCols, (slice+1)*kSliceCols) = tokens [slice*tok_per_slice, ...)
        const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                (MX ? slot * 128 : acc * kNRows + slice * kSliceCols);
        dsa::check((MX ? (slot + 1) * 128 : acc * kNRows + (slice + 1) * kSliceCols) <= kSfaCol || !MX, p.status);
        dsa::check(acc * kNRows + (slice + 1) * kSliceCols <= static_cast<int>(kTmemCols), p.status);
        // fused: a row's entry bound for this tile, read once (tau only rises
        // and a compacted segment's floor only rises, so a value read early
        // can only admit more candidates)
        uint32_t thr[tok_per_slice];
        if (FUSED) {
#pragma unroll
          for (int q = 0; q < tok_per_slice; ++q) {
            const int r = slice * tok_per_slice + q;
            const uint32_t tau = reinterpret_cast<volatile uint32_t*>(row_tau)[r];
            const uint32_t fl =
                ((cmask >> q) & 1u) ? reinterpret_cast<volatile uint32_t*>(seg_floor)[r * 4 + seg] : 0u;
            thr[q] = max(tau, fl);
          }
        }
        // score = sum_h w[h] * max(D[h], 0).  Head pair (2i, 2i+1) goes to
        // chain i % 4 (one packed fma per pair), and the four chains are
        // summed as a tree at the token's last head: four independent
        // dependency chains instead of one.  Fused and dense modes run this
        // same sequence, so their scores are identical.
        float ch[8];
        auto process = [&](const uint32_t(&v)[32], auto chunk) {
          constexpr int c = decltype(chunk)::value;  // 32-column chunk of this slice
          const float4* w4 = reinterpret_cast<const float4*>(w_s + slice * kSliceCols + c * 32);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const int cl = c * 32 + 4 * g;  // first of four columns (compile-time)
            const int h = cl % HI;          // a multiple of 4 (kSliceCols % HI == 0, HI % 8 == 0)
            if (h == 0) {
#pragma unroll
              for (int j = 0; j < 8; ++j) ch[j] = 0.f;
            }
            const float4 wv = w4[g];
            const int j0 = (h >> 1) & 3;  // 0 or 2; the next pair takes j0 + 1
            dsa::fma2(ch[2 * j0], ch[2 * j0 + 1], wv.x, wv.y, fmaxf(__uint_as_float(v[4 * g]), 0.f),
                      fmaxf(__uint_as_float(v[4 * g + 1]), 0.f));
            dsa::fma2(ch[2 * j0 + 2], ch[2 * j0 + 3], wv.z, wv.w, fmaxf(__uint_as_float(v[4 * g + 2]), 0.f),
                      fmaxf(__uint_as_float(v[4 * g + 3]), 0.f));
            if (h + 3 == HI - 1) {
              const float sum = ((ch[0] + ch[1]) + (ch[2] + ch[3])) + ((ch[4] + ch[5]) + (ch[6] + ch[7]));
              const float score = F8 == 1 ? sum * ks : sum;
              const int q = cl / HI;  // token within this slice (compile-time)
              const int r = slice * tok_per_slice + q;
              const int t = br.t0 + r;
              const int st = rs[q];
              const bool valid = static_cast<uint32_t>(s_key - st) < static_cast<uint32_t>(rl[q]);
              if (!FUSED) {
                // checked build: row and column inside scores [T, ld]
                if (valid && dsa::check(t < p.T && s_key - st < p.ld, p.status))
                  __stcs(p.scores + static_cast<int64_t>(t) * p.ld + (s_key - st), score);
              } else {
                const uint32_t key = dsa::f32_key(score);
                const bool emit = valid && key >= thr[q];
                // append to this warp's own segment of row t: no atomics, the
                // warp-uniform counter lives in a register; the segment has
                // room for a whole tile (compaction below)
                const uint32_t em = __ballot_sync(0xffffffffu, emit);
                const int slot = wcnt[q] + __popc(em & dsa::lanemask_lt());
                if (emit && dsa::check(slot < cap_seg && t < p.T, p.status)) {
                  // default L2 policy: the compaction warps read the segment back one block later
                  p.cand[(static_cast<int64_t>(t) * 4 + seg) * cap_seg + slot] = make_uint2(key, s_key - st);
                  // histogram of stored keys, one 32-bit counter per bin; the
                  // result is unused, so this is a fire-and-forget reduction
                  atomicAdd(&hist[r * hist_words_row + hist_bin(key, p.hist_bits)], 1u);
                }
                wcnt[q] += __popc(em);
              }
            }
          }
        };
        // four 32-column TMEM loads, each issued before the previous chunk is
        // processed, so only the first load's latency is exposed
        uint32_t va[32], vb[32];
        dsa::tmem_ld32(t_addr, va);
        dsa::tmem_wait_ld_pin(va);
        dsa::tmem_ld32(t_addr + 32, vb);
        process(va, std::integral_constant<int, 0>{});
        dsa::tmem_wait_ld_pin(vb);
        if constexpr (kSliceChunks == 4) {
          dsa::tmem_ld32(t_addr + 64, va);
          process(vb, std::integral_constant<int, 1>{});
          dsa::tmem_wait_ld_pin(va);
          dsa::tmem_ld32(t_addr + 96, vb);
          process(va, std::integral_constant<int, 2>{});
          dsa::tmem_wait_ld_pin(vb);
          process(vb, std::integral_constant<int, 3>{});
        } else {
          process(vb, std::integral_constant<int, 1>{});
        }
        dsa::tc_fence_before();
        __syncwarp();
        if (lane == 0) dsa::mbar_arrive(&tempty[slot]);
        if constexpr (MX) {
          jh += kSlices;
        } else {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
        if (FUSED && p.compact) {
          // a segment that might not hold the next tile's 32 keys is cut to its top-k
#pragma unroll
          for (int q = 0; q < tok_per_slice; ++q) {
            if (wcnt[q] > cap_seg - 32) {
              const int r = slice * tok_per_slice + q;
              const int64_t t = br.t0 + r;
              const uint32_t fl = compact_segment(p.cand + (t * 4 + seg) * cap_seg, wcnt[q], p.k, cmp_hist + ew * 256);
              if (lane == 0) {
                seg_floor[r * 4 + seg] = fl;
                seg_drop[r * 4 + seg] += wcnt[q] - p.k;
              }
              wcnt[q] = p.k;
              cmask |= 1u << q;
              __syncwarp();
            }
          }
        }
        if (FUSED && ((kt - br.kt0) & 3) == 3) {
          // Every fourth tile, raise tau of the rows this warp owns once enough
          // new candidates arrived.  No barrier: tau only has to stay a lower
          // bound of the row's k-th largest key, and a histogram read while
          // other warps still add to it can only undercount, which lowers it.
          const int r0 = slice * tok_per_slice;
          if (lane == 0) {
#pragma unroll
            for (int q = 0; q < tok_per_slice; ++q)
              reinterpret_cast<volatile int32_t*>(seg_cnt)[(r0 + q) * 4 + seg] = wcnt[q] + seg_drop[(r0 + q) * 4 + seg];
          }
          for (int r = r0 + (ew & 3); r < r0 + tok_per_slice; r += 4) {
            int cnt = 0;  // candidates emitted so far (stored or since dropped)
            if (lane == 0) {
              const volatile int32_t* sc = reinterpret_cast<volatile int32_t*>(seg_cnt) + r * 4;
              for (int sg = 0; sg < 4; ++sg) cnt += sc[sg];
            }
            cnt = __shfl_sync(0xffffffffu, cnt, 0);
            if (cnt - row_since[r] >= kTauUpdateEvery) {
              update_tau(hist + r * hist_words_row, hist_words_row, p.hist_bits, p.k, &row_tau[r]);
              if (lane == 0) row_since[r] = cnt;  // row_since: candidate count at the last update
              __syncwarp();
            }
          }
        }
      }
      if (dsa::named_bar_any(1, kEpiThreads, failed)) {
        ok = false;
        break;
      }
      if (!FUSED) {
        // columns len[t] .. s_max-1 of the block's rows are -inf
        for (int r = 0; r < p.qb; ++r) {
          const int t = br.t0 + r;
          if (t >= p.T) break;
          float* row = p.scores + static_cast<int64_t>(t) * p.ld;
          for (int j = tok_len[r] + et; j < p.s_max; j += kEpiThreads) row[j] = -INFINITY;
        }
      } else {
        // this block goes to slot blk_i & 1 once the compaction warps are done
        // with the block that used it before
        const int slot = static_cast<int>(blk_i & 1u);
        if (!failed) failed = !dsa::mbar_wait(&pend_empty[slot], ((blk_i >> 1) & 1u) ^ 1u, wt);
        if (lane == 0) {
#pragma unroll
          for (int q = 0; q < tok_per_slice; ++q) {
            const int r = slice * tok_per_slice + q;
            pend_n[slot * 128 + r * 4 + seg] = wcnt[q];
          }
        }
        // Each row's threshold bin from its complete histogram (the running
        // threshold lags by up to kTauUpdateEvery candidates): b = the highest
        // bin at which the row's emitted candidates number >= k, [x, y) its
        // key range.  A candidate that a compacted segment dropped (or never
        // admitted, below its floor) is beaten by k stored keys of its
        // segment, so at least k stored candidates reach x; fewer than k keys
        // of the row reach y, all of them stored, so all of them are in the
        // row's top-k.  Stage 2 takes those outright and ranks only the
        // stored keys in [x, y).  (The block's last barrier above ordered
        // every histogram update before these reads; the next block clears
        // the histograms only after its first barrier.)
        for (int r = ew; r < p.qb; r += kEpiWarps) {
          update_tau(hist + r * hist_words_row, hist_words_row, p.hist_bits, p.k, &row_tau[r]);
          __syncwarp();
          const int t = br.t0 + r;
          const uint32_t x = reinterpret_cast<volatile uint32_t*>(row_tau)[r];
          if (lane == 0) pend_x[slot * 32 + r] = x;
          if (lane == 0 && t < p.T) {
            const int b = static_cast<int>(hist_bin(x, p.hist_bits));
            const uint32_t y = b + 1 < (1 << p.hist_bits) ? hist_edge(b + 1, p.hist_bits) : 0u;
            p.cand_tau[t] = make_uint2(x, y);
          }
        }
        __syncwarp();
        if (lane == 0) dsa::mbar_arrive(&pend_full[slot]);
      }
      ++blk_i;
    }
  } else if (FUSED) {
    // -------------------------------------------------- segment compaction
    // One block behind the epilogue: each finished block's candidate
    // segments are compacted in place to the candidates at or above the
    // row's final threshold x (nothing below it can be selected), so that
    // stage 2 reads about k candidates per row instead of all that were
    // emitted.  A kept candidate moves to index kept + (kept ones before it
    // in the round), never past its own index, and a round's stores follow
    // all its loads, so nothing is read after it was overwritten.  These
    // warps only touch global memory and the handed-over slot.
    const int cw = warp - kCmpWarp0;  // 0 .. kCmpWarps-1
    const int cap_seg = p.cap / 4;
    uint32_t i = 0;
    for (int blk = p.nblocks - 1 - blockIdx.x; blk >= 0; blk -= gridDim.x, ++i) {
      const BlockRange br = block_range<GEN>(p, blk);
      const int slot = static_cast<int>(i & 1u);
      if (!dsa::mbar_wait_warp(&pend_full[slot], (i >> 1) & 1u, wt)) break;
      for (int pr = cw; pr < p.qb * 4; pr += kCmpWarps) {
        const int r = pr >> 2, sg = pr & 3;
        const int t = br.t0 + r;
        if (t >= p.T) break;
        const uint32_t x = pend_x[slot * 32 + r];
        const int n = pend_n[slot * 128 + pr];
        int kept = n;
        if (x != 0u) {  // x == 0: every candidate stays
          uint2* segp = p.cand + (static_cast<int64_t>(t) * 4 + sg) * cap_seg;  // 16-byte aligned: cap_seg % 4 == 0
          const uint4* seg4 = reinterpret_cast<const uint4*>(segp);
          const uint32_t below = (1u << lane) - 1u;
          kept = 0;
          for (int i0 = 0; i0 < n; i0 += 64 * kCompactU) {
            uint4 v[kCompactU];
#pragma unroll
            for (int u = 0; u < kCompactU; ++u) {
              const int e = i0 + 64 * u + 2 * lane;  // the pair's first candidate
              v[u] = e < n ? seg4[e >> 1] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < kCompactU; ++u) {
              const int e = i0 + 64 * u + 2 * lane;
              const uint32_t m0 = __ballot_sync(0xffffffffu, e < n && v[u].x >= x);
              const uint32_t m1 = __ballot_sync(0xffffffffu, e + 1 < n && v[u].z >= x);
              const bool k0 = (m0 >> lane) & 1u, k1 = (m1 >> lane) & 1u;
              const int at = kept + __popc(m0 & below) + __popc(m1 & below);
              if (k0) segp[at] = make_uint2(v[u].x, v[u].y);
              if (k1) segp[at + (k0 ? 1 : 0)] = make_uint2(v[u].z, v[u].w);
              kept += __popc(m0) + __popc(m1);
            }
          }
        }
        if (lane == 0) p.cand_cnt[static_cast<int64_t>(t) * 4 + sg] = kept;
        if (kept < n) {
          // The candidates past `kept` are dead: drop their L2 lines without
          // writing them back (only lines wholly inside the dead range of
          // this segment; the line holding the last live or the last emitted
          // candidate stays)
          const uintptr_t seg0 = reinterpret_cast<uintptr_t>(p.cand + (static_cast<int64_t>(t) * 4 + sg) * cap_seg);
          const uintptr_t lo = (seg0 + static_cast<uintptr_t>(kept) * 8u + 127u) & ~static_cast<uintptr_t>(127);
          const uintptr_t hi = (seg0 + static_cast<uintptr_t>(n) * 8u) & ~static_cast<uintptr_t>(127);
          for (uintptr_t a = lo + 128u * lane; a < hi; a += 128u * 32u) l2_discard_line(a);
        }
      }
      __syncwarp();
      if (lane == 0) dsa::mbar_arrive(&pend_empty[slot]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    dsa::tc_fence_after();
    dsa::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Candidates of one row: four segments of (key, column) pairs.
struct SegmentedPairSrc {
  const uint2* base;  // row's first segment
  int cap_seg;
  int n0, n1, n2, n3;  // valid pairs per segment
  int n;
  __device__ __forceinline__ uint32_t key_at(int i) const {
    const int e1 = n0, e2 = n0 + n1, e3 = n0 + n1 + n2;
    const int sg = (i >= e1) + (i >= e2) + (i >= e3);
    const int off = i - (sg == 0 ? 0 : sg == 1 ? e1 : sg == 2 ? e2 : e3);
    return __ldg(&base[sg * cap_seg + off].x);
  }
  template <class F>
  __device__ __forceinline__ void for_each(F&& f) const {
    const int e1 = n0, e2 = n0 + n1, e3 = n0 + n1 + n2;
    constexpr int U = 4;  // loads in flight per thread before processing
    for (int b = 0; b < n; b += blockDim.x * U) {
      uint2 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = b + u * blockDim.x + threadIdx.x;
        v[u] = make_uint2(0u, 0u);
        if (i < n) {
          const int sg = (i >= e1) + (i >= e2) + (i >= e3);
          const int off = i - (sg == 0 ? 0 : sg == 1 ? e1 : sg == 2 ? e2 : e3);
          v[u] = __ldcs(base + sg * cap_seg + off);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = b + u * blockDim.x + threadIdx.x;
        f(v[u].x, static_cast<int32_t>(v[u].y), i < n);
      }
    }
  }
};

// Stage 2 of the fused path: exact top-k of each row's candidates.
template <int GEN>
__global__ void __launch_bounds__(dsa::kTopkThreads)
    fused_select_kernel(const __grid_constant__ Geom g, int T, int k, const uint2* cand,
                        const int32_t* __restrict__ cand_cnt, int cap, int32_t* idx, int32_t* topk_length,
                        uint32_t* status) {
  extern __shared__ __align__(16) uint8_t smem_raw2[];
  dsa::TopkShared& S = *reinterpret_cast<dsa::TopkShared*>(smem_raw2);
  const int t = blockIdx.x;
  int st;
  const int len = row_geom<GEN>(g, t, &st);
  int32_t* out = idx + static_cast<int64_t>(t) * k;
  if (len <= k) {
    for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = j < len ? st + j : -1;
    if (threadIdx.x == 0 && topk_length) topk_length[t] = len;
    return;
  }
  const int cap_seg = cap / 4;
  int c[4];
  bool overflow = false;
#pragma unroll
  for (int sg = 0; sg < 4; ++sg) {
    c[sg] = __ldg(cand_cnt + static_cast<int64_t>(t) * 4 + sg);
    if (c[sg] > cap_seg) {
      overflow = true;
      c[sg] = cap_seg;
    }
  }
  if (overflow && threadIdx.x == 0) atomicOr(status, DSA_STATUS_CAND_OVERFLOW);
  const int n = c[0] + c[1] + c[2] + c[3];
  if (n < k) {  // only reachable after an overflow: keep the output well-formed
    for (int j = threadIdx.x; j < k; j += blockDim.x) out[j] = -1;
    if (threadIdx.x == 0 && topk_length) topk_length[t] = 0;
    return;
  }
  const SegmentedPairSrc src{cand + static_cast<int64_t>(t) * cap, cap_seg, c[0], c[1], c[2], c[3], n};
  if (len <= 32 * dsa::kBitmapWords && dsa::select_topk_sampled(S, src, n, k, len)) {
    dsa::emit_bits_ascending(S, len, [&](int pos, int j) { out[pos] = st + j; });
  } else {
    dsa::select_topk(S, src, k);
    for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = st + S.sel[i];
  }
  if (threadIdx.x == 0 && topk_length) topk_length[t] = k;
}

// Stage 2's multi-row form (below) serves rows of up to kSelMaxLen columns
// (its column bitmaps); longer rows use fused_select_kernel.
constexpr int kSelMaxLen = 65536;

// Stage 2, multi-row form: four persistent 256-thread CTAs per SM, one row
// each at a time, so that the rows' phases overlap.  Stage 1 hands over each
// row's final threshold bin [x, y) (see the fused epilogue): fewer than k of
// the row's keys reach y and all of them are stored, so all of them are
// selected; at least k stored keys reach x, so nothing below x is (stage 1's
// compaction warps have already removed those).  Per row:
//  1. one streaming pass over the candidate segments (16-byte loads, the
//     segments prefetched into L2 one row ahead) sets the columns of keys
//     >= y in the selection bitmap and keeps the keys in [x, y) -- typically
//     a few hundred -- in a shared-memory list (a row with more than the list
//     holds is ranked from the segments themselves, the same steps as passes
//     over global memory);
//  2. radix passes (11 bits at most) over v = key - lo of the kept keys, with
//     lo / hi their smallest / largest key, find the exact key tau of rank
//     need = k - (keys >= y) among them and how many keys equal to tau are
//     still needed;
//  3. kept keys above tau go to the selection bitmap and keys equal to it to
//     a tie bitmap; the block takes the needed tied columns from the smallest
//     up, and one scan of the bitmap turns it into ascending ids, staged in
//     shared memory and stored with 16-byte writes (and, when asked for, the
//     logits of the selected candidates at their slots).
constexpr int kMThreads = 256;
constexpr int kMWarps = kMThreads / 32;
constexpr int kMKeep = 1024;                  // kept keys ([x, y)) held in shared memory
constexpr int kMBits = 10;                     // radix digit
constexpr int kMBins = 1 << kMBits;
constexpr int kMBinsPer = kMBins / kMThreads;  // histogram bins one thread scans
constexpr int kMStageU = 6;                    // 16-byte loads in flight per thread
constexpr int kMStage = kMStageU * kMThreads;  // staged 16-byte slots of one batch
constexpr int kMWords = kSelMaxLen / 32;       // column bitmaps for rows of up to 65536 columns
constexpr int kMWordsPer = kMWords / kMThreads;  // bitmap words owned by one thread
constexpr int kMCtasPerSm = 4;
static_assert(kMStage * 4 >= DSA_MAX_TOPK, "the id staging buffer aliases the load staging buffer");

// 16-byte global -> shared copy that the L2 may evict first (read once).
__device__ __forceinline__ void cp_async16_cs(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "l"(dsa::l2_policy_evict_first())
               : "memory");
}

struct MultiShared {
  uint4 stage[kMStage];   // each thread's in-flight 16-byte loads; after step 2, the row's ids
  uint32_t skey[kMKeep];  // kept keys
  uint32_t scol[kMKeep];
  uint32_t hist[kMBins];
  uint32_t sel[kMWords];
  uint32_t tie[kMWords];
  int wsum[2][kMWarps];
  uint32_t wlo[kMWarps], whi[kMWarps];
  int wtop[kMWarps];
  int ns;  // kept keys of the row (may exceed kMKeep)
  int bin, above, n_eq;
};

// Exclusive prefix of v over the block (one barrier); wsum buffer `par`
// must not be in use by another scan between two barriers.
__device__ __forceinline__ int multi_scan(int v, int (*wsum)[kMWarps], int par) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[par][warp] = incl;
  __syncthreads();
  int before = 0;
#pragma unroll
  for (int w = 0; w < kMWarps; ++w)
    if (w < warp) before += wsum[par][w];
  return before + incl - v;
}

template <int GEN>
__global__ void __launch_bounds__(kMThreads, kMCtasPerSm)
    fused_select_multi_kernel(const __grid_constant__ Geom g, int T, int k, const uint2* cand,
                              const int32_t* __restrict__ cand_cnt, const uint2* __restrict__ cand_tau, int cap,
                              int32_t* idx, int32_t* topk_length, float* logits, uint32_t* status) {
  extern __shared__ __align__(16) uint8_t smem_multi[];
  MultiShared& S = *reinterpret_cast<MultiShared*>(smem_multi);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cap_seg = cap / 4;
  for (int i = threadIdx.x; i < kMBins; i += kMThreads) S.hist[i] = 0u;
  for (int i = threadIdx.x; i < kMWords; i += kMThreads) {
    S.sel[i] = 0u;
    S.tie[i] = 0u;
  }
  __syncthreads();
  // A row's segment counts and threshold bin are loaded one row ahead (their
  // latency hides behind the row before), and its candidate segments are
  // prefetched into L2 then.
  int4 cnt_next = make_int4(0, 0, 0, 0);
  uint2 xy_next = make_uint2(0u, 0u);
  auto load_meta = [&](int r) {
    if (r >= T) return;
    const int t = T - 1 - r;
    cnt_next = __ldg(reinterpret_cast<const int4*>(cand_cnt) + t);  // [T][4] int32: 16-byte rows
    xy_next = __ldg(cand_tau + t);
  };
  auto prefetch_row = [&](int r, const int4& cn) {
    if (r >= T) return;
    const int t = T - 1 - r;
    const int cs[4] = {cn.x, cn.y, cn.z, cn.w};
#pragma unroll
    for (int sg = 0; sg < 4; ++sg) {
      const int cnt = min(cs[sg], cap_seg);
      const uint32_t bytes = static_cast<uint32_t>((cnt + 1) & ~1) * 8u;  // whole 16-byte pairs
      if (bytes) dsa::l2_prefetch_bulk(cand + static_cast<int64_t>(t) * cap + sg * cap_seg, bytes);
    }
  };
  load_meta(blockIdx.x);
  const int w0 = kMWordsPer * static_cast<int>(threadIdx.x);  // this thread's bitmap words, in column order
  // longest rows first
  for (int r = blockIdx.x; r < T; r += gridDim.x) {
    const int4 cn = cnt_next;
    const uint2 xy = xy_next;
    load_meta(r + gridDim.x);
    if (threadIdx.x == 0) prefetch_row(r + gridDim.x, cnt_next);
    const int t = T - 1 - r;
    int st = 0;
    const int len = row_geom<GEN>(g, t, &st);
    int32_t* out = idx + static_cast<int64_t>(t) * k;
    float* lout = logits ? logits + static_cast<int64_t>(t) * k : nullptr;
    int c[4] = {cn.x, cn.y, cn.z, cn.w};
    bool overflow = false;
#pragma unroll
    for (int sg = 0; sg < 4; ++sg) {
      if (c[sg] > cap_seg) {
        overflow = true;
        c[sg] = cap_seg;
      }
    }
    const uint2* seg0 = cand + static_cast<int64_t>(t) * cap;
    if (len <= k) {
      for (int j = threadIdx.x; j < k; j += kMThreads) out[j] = j < len ? st + j : -1;
      if (threadIdx.x == 0 && topk_length) topk_length[t] = len;
      if (lout) {
        // every key of a row this short is a candidate: its value goes to the
        // slot of its column
        for (int j = len + threadIdx.x; j < k; j += kMThreads) lout[j] = -INFINITY;
#pragma unroll
        for (int sg = 0; sg < 4; ++sg)
          for (int i = threadIdx.x; i < c[sg]; i += kMThreads) {
            const uint2 v = seg0[sg * cap_seg + i];
            if (static_cast<int>(v.y) < len) lout[v.y] = dsa::key_f32(v.x);
          }
      }
      continue;
    }
    if (overflow && threadIdx.x == 0) atomicOr(status, DSA_STATUS_CAND_OVERFLOW);
    const int n = c[0] + c[1] + c[2] + c[3];
    if (n < k) {  // only reachable after an overflow: keep the output well-formed
      for (int j = threadIdx.x; j < k; j += kMThreads) {
        out[j] = -1;
        if (lout) lout[j] = -INFINITY;
      }
      if (threadIdx.x == 0 && topk_length) topk_length[t] = 0;
      continue;
    }
    // ---- 1. keys >= y into the bitmap, keys in [x, y) into the kept list
    uint32_t tx = overflow ? 0u : xy.x, ty = overflow ? 0u : xy.y;  // ty == 0: no outright keys
    uint32_t lo, hi;
    int n_keep, n_top;
    for (;;) {
      if (threadIdx.x == 0) S.ns = 0;
      __syncthreads();
      lo = 0xFFFFFFFFu;
      hi = 0u;
      int top = 0;
      // the row's 16-byte slots (two pairs each) as one flat range over the
      // four segments: segment sg holds slots [o[sg], o[sg + 1])
      const int o1 = (c[0] + 1) >> 1, o2 = o1 + ((c[1] + 1) >> 1), o3 = o2 + ((c[2] + 1) >> 1);
      const int n4 = o3 + ((c[3] + 1) >> 1);
      for (int j0 = 0; j0 < n4; j0 += kMStage) {
        // kMStageU copies per thread into its own staging slots (read back
        // only by this thread, after its own wait: no barrier needed)
#pragma unroll
        for (int u = 0; u < kMStageU; ++u) {
          const int f = j0 + u * kMThreads + static_cast<int>(threadIdx.x);
          if (f < n4) {
            const int sg = (f >= o1) + (f >= o2) + (f >= o3);
            const int local = f - (sg == 0 ? 0 : sg == 1 ? o1 : sg == 2 ? o2 : o3);
            cp_async16_cs(dsa::smem_u32(&S.stage[u * kMThreads + threadIdx.x]),
                          reinterpret_cast<const uint4*>(seg0 + sg * cap_seg) + local);
          }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        // this thread's kept keys of its pairs, then one shared-counter add per warp
        uint32_t kmask = 0u;
        uint4 v[kMStageU];
#pragma unroll
        for (int u = 0; u < kMStageU; ++u) {
          const int f = j0 + u * kMThreads + static_cast<int>(threadIdx.x);
          v[u] = S.stage[u * kMThreads + threadIdx.x];
          const int sg = (f >= o1) + (f >= o2) + (f >= o3);
          const int local = f - (sg == 0 ? 0 : sg == 1 ? o1 : sg == 2 ? o2 : o3);
          const int cnt = f < n4 ? (sg == 0 ? c[0] : sg == 1 ? c[1] : sg == 2 ? c[2] : c[3]) : 0;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
              const int e = 2 * local + h;
              const uint32_t key = h ? v[u].z : v[u].x, col = h ? v[u].w : v[u].y;
              if (e < cnt && key >= tx) {
                if (ty != 0u && key >= ty) {
                  if (dsa::check(static_cast<int>(col) < len, status)) {  // checked build: the column lies in the row
                    atomicOr(&S.sel[col >> 5], 1u << (col & 31));
                    ++top;
                  }
                } else {
                  lo = min(lo, key);
                  hi = max(hi, key);
                  kmask |= 1u << (2 * u + h);
                }
              }
          }
        }
          const int mine = __popc(kmask);
          int incl = mine;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          int base = 0;
          if (lane == 31 && incl > 0) base = atomicAdd(&S.ns, incl);
          base = __shfl_sync(0xffffffffu, base, 31) + incl - mine;
#pragma unroll
          for (int u = 0; u < kMStageU; ++u) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if ((kmask >> (2 * u + h)) & 1u) {
                if (base < kMKeep) {
                  S.skey[base] = h ? v[u].z : v[u].x;
                  S.scol[base] = h ? v[u].w : v[u].y;
                }
                ++base;
              }
            }
          }
      }
      lo = __reduce_min_sync(0xffffffffu, lo);
      hi = __reduce_max_sync(0xffffffffu, hi);
      top = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(top)));
      if (lane == 0) {
        S.wlo[warp] = lo;
        S.whi[warp] = hi;
        S.wtop[warp] = top;
      }
      __syncthreads();
      n_keep = S.ns;
      lo = 0xFFFFFFFFu;
      hi = 0u;
      n_top = 0;
#pragma unroll
      for (int w = 0; w < kMWarps; ++w) {
        lo = min(lo, S.wlo[w]);
        hi = max(hi, S.whi[w]);
        n_top += S.wtop[w];
      }
      // not reachable (see the stage 1 epilogue): fewer than k keys reach y and
      // at least k reach x; kept so that a row is never selected wrongly
      if ((n_top < k && n_top + n_keep >= k) || (tx == 0u && ty == 0u)) break;
      tx = 0u;
      ty = 0u;
#pragma unroll
      for (int j = 0; j < kMWordsPer; ++j) S.sel[w0 + j] = 0u;
      __syncthreads();  // every thread has read S.ns and the per-warp words
    }
    const bool in_smem = n_keep <= kMKeep;
    // f(key, column) for every kept key: from the shared list, or from the
    // segments when the list overflowed (no warp-collective inside f)
    auto for_each = [&](auto&& f) {
      if (in_smem) {
        for (int i = threadIdx.x; i < n_keep; i += kMThreads) f(S.skey[i], S.scol[i]);
      } else {
#pragma unroll 1
        for (int sg = 0; sg < 4; ++sg)
          for (int i = threadIdx.x; i < c[sg]; i += kMThreads) {
            const uint2 v = seg0[sg * cap_seg + i];
            if (v.x >= tx && (ty == 0u || v.x < ty)) f(v.x, v.y);
          }
      }
    };
    // ---- 2. radix passes over v = key - lo, at most 11 bits each, top down
    const int nbits = hi > lo ? 32 - __clz(hi - lo) : 0;
    uint32_t prefix = 0u, mask = 0u;
    int k_rem = k - n_top, n_eq = n_keep, shift = nbits, par = 0;
    while (shift > 0) {
      const int db = shift < kMBits ? shift : kMBits;
      shift -= db;
      const int nb = 1 << db;
      for_each([&](uint32_t key, uint32_t) {
        const uint32_t v = key - lo;
        if ((v & mask) == prefix) atomicAdd(&S.hist[(v >> shift) & (nb - 1)], 1u);
      });
      __syncthreads();
      // thread i holds bins nb-1-kMBinsPer*i .. (the top bins first)
      int cb[kMBinsPer];
      int sum = 0;
#pragma unroll
      for (int j = 0; j < kMBinsPer; ++j) {
        const int b = nb - 1 - kMBinsPer * static_cast<int>(threadIdx.x) - j;
        cb[j] = b >= 0 ? static_cast<int>(S.hist[b]) : 0;
        if (b >= 0) S.hist[b] = 0u;  // ready for the next pass
        sum += cb[j];
      }
      const int excl = multi_scan(sum, S.wsum, par);
      par ^= 1;
      if (excl < k_rem && excl + sum >= k_rem) {
        int acc = excl;
#pragma unroll
        for (int j = 0; j < kMBinsPer; ++j) {
          if (acc + cb[j] >= k_rem) {
            S.bin = nb - 1 - kMBinsPer * static_cast<int>(threadIdx.x) - j;
            S.above = acc;
            S.n_eq = cb[j];
            break;
          }
          acc += cb[j];
        }
      }
      __syncthreads();
      prefix |= static_cast<uint32_t>(S.bin) << shift;
      mask |= static_cast<uint32_t>(nb - 1) << shift;
      k_rem -= S.above;
      n_eq = S.n_eq;
    }
    const uint32_t tau = lo + prefix;
    const int need = k_rem;
    // ---- 3. bitmaps of the selected and the tied columns
    for_each([&](uint32_t key, uint32_t col) {
      if (!dsa::check(static_cast<int>(col) < len, status)) return;  // checked build: the column lies in the row
      if (key > tau) atomicOr(&S.sel[col >> 5], 1u << (col & 31));
      else if (key == tau) atomicOr(&S.tie[col >> 5], 1u << (col & 31));
    });
    __syncthreads();
    uint32_t m[kMWordsPer], tb[kMWordsPer];
    int pm = 0, pt = 0;
#pragma unroll
    for (int j = 0; j < kMWordsPer; ++j) {
      m[j] = S.sel[w0 + j];
      tb[j] = S.tie[w0 + j];
      S.sel[w0 + j] = 0u;  // ready for the next row
      S.tie[w0 + j] = 0u;
      pt += __popc(tb[j]);
    }
    if (n_eq != need) {
      // only the `need` tied columns with the smallest indices
      int taken = multi_scan(pt, S.wsum, par);
      par ^= 1;
#pragma unroll
      for (int j = 0; j < kMWordsPer; ++j) {
        uint32_t keep = 0u, rest = tb[j];
        while (rest && taken < need) {
          const uint32_t low = rest & (0u - rest);
          keep |= low;
          rest ^= low;
          ++taken;
        }
        tb[j] = keep;
      }
    }
#pragma unroll
    for (int j = 0; j < kMWordsPer; ++j) {
      m[j] |= tb[j];
      pm += __popc(m[j]);
    }
    // the ids in ascending order, staged in shared memory (in the load
    // staging buffer, free since step 1), then stored with 16-byte writes
    // where the row allows (with logits asked for they go to global memory
    // directly)
    const int pos0 = multi_scan(pm, S.wsum, par);
    par ^= 1;
    const bool stage_ids = lout == nullptr && (reinterpret_cast<uintptr_t>(out) & 15u) == 0u;
    int pos = pos0;
#pragma unroll
    for (int j = 0; j < kMWordsPer; ++j) {
      uint32_t w = m[j];
      while (w) {
        const int b = __ffs(w) - 1;
        w &= w - 1;
        if (dsa::check(pos < k, status)) {  // checked build: k ids at most
          const int id = st + ((w0 + j) << 5) + b;
          if (stage_ids) reinterpret_cast<int32_t*>(S.stage)[pos] = id;
          else out[pos] = id;
        }
        ++pos;
      }
    }
    if (threadIdx.x == 0 && topk_length) topk_length[t] = k;
    if (stage_ids) {
      __syncthreads();
      for (int i = threadIdx.x; i < k / 4; i += kMThreads)
        reinterpret_cast<int4*>(out)[i] = reinterpret_cast<const int4*>(S.stage)[i];
      for (int i = (k & ~3) + static_cast<int>(threadIdx.x); i < k; i += kMThreads)
        out[i] = reinterpret_cast<const int32_t*>(S.stage)[i];
    }
    if (lout) {
      // each selected candidate's value at the slot of its column: the slot is
      // its word's first slot plus the selected columns below it in the word
      int p2 = pos0;
#pragma unroll
      for (int j = 0; j < kMWordsPer; ++j) {
        S.sel[w0 + j] = m[j];
        S.tie[w0 + j] = static_cast<uint32_t>(p2);
        p2 += __popc(m[j]);
      }
      __syncthreads();
#pragma unroll 1
      for (int sg = 0; sg < 4; ++sg)
        for (int i = threadIdx.x; i < c[sg]; i += kMThreads) {
          const uint2 v = seg0[sg * cap_seg + i];
          const int col = static_cast<int>(v.y);
          if (v.x < tx || col >= len) continue;
          const uint32_t word = S.sel[col >> 5], below = (1u << (col & 31)) - 1u;
          if ((word >> (col & 31)) & 1u) lout[S.tie[col >> 5] + __popc(word & below)] = dsa::key_f32(v.x);
        }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kMWordsPer; ++j) {
        S.sel[w0 + j] = 0u;
        S.tie[w0 + j] = 0u;
      }
    }
    __syncthreads();  // the next row reuses the shared words above
  }
}

int validate_common(const void* qi, const void* ki, const float* w, int n_docs, int Tq, int Hi, int d,
                    const char* fn) {
  if (!qi || !ki || !w) return dsa::set_error(DSA_ERR_VALUE, "%s: NULL input pointer", fn);
  if (n_docs < 1 || Tq < 1) return dsa::set_error(DSA_ERR_VALUE, "%s: need n_docs >= 1 and T >= 1", fn);
  if (d != 64 && d != 128) return dsa::set_error(DSA_ERR_VALUE, "%s: d must be 64 or 128 (got %d)", fn, d);
  if (Hi != 8 && Hi != 16 && Hi != 32 && Hi != 64)
    return dsa::set_error(DSA_ERR_VALUE, "%s: Hi must be 8, 16, 32 or 64 (got %d)", fn, Hi);
  if (!dsa::aligned(qi, 16) || !dsa::aligned(ki, 16))
    return dsa::set_error(DSA_ERR_VALUE, "%s: qi and ki must be 16-byte aligned", fn);
  if (static_cast<int64_t>(Tq) * Hi > INT_MAX) return dsa::set_error(DSA_ERR_VALUE, "%s: T*Hi too large", fn);
  return DSA_OK;
}

// The plain causal THD form: keys stored like the queries, ratio 1.
int validate_indexer(const void* qi, const void* ki, const float* w, const int32_t* cu, int n_docs, int T, int Hi,
                     int d, int s_max, const char* fn) {
  int rc = validate_common(qi, ki, w, n_docs, T, Hi, d, fn);
  if (rc != DSA_OK) return rc;
  if (!cu) return dsa::set_error(DSA_ERR_VALUE, "%s: NULL cu_seqlens", fn);
  if (s_max < 1 || s_max > T) return dsa::set_error(DSA_ERR_VALUE, "%s: need 1 <= s_max <= T", fn);
  return DSA_OK;
}

// The ratio-causal form over a compressed key prefix.
int validate_ratio(const void* qi, const void* ki, const float* w, const int32_t* cu_q, const int32_t* cu_k,
                   int n_docs, int Tq, int Tk, int Hi, int d, int ratio, int s_max, const char* fn) {
  int rc = validate_common(qi, ki, w, n_docs, Tq, Hi, d, fn);
  if (rc != DSA_OK) return rc;
  if (!cu_q || !cu_k) return dsa::set_error(DSA_ERR_VALUE, "%s: NULL cu_seqlens_q or cu_seqlens_k", fn);
  if (Tk < 1 || ratio < 1) return dsa::set_error(DSA_ERR_VALUE, "%s: need Tk >= 1 and ratio >= 1", fn);
  if (s_max < 1 || s_max > Tk) return dsa::set_error(DSA_ERR_VALUE, "%s: need 1 <= s_max <= Tk", fn);
  return DSA_OK;
}

Geom plain_geom(const int32_t* cu, int n_docs, int s_max) { return Geom{cu, cu, nullptr, n_docs, 1, s_max}; }

// The indexer's tensor inputs: bf16 qi / ki, or E4M3 with fp32 descales.
struct Inputs {
  const void* qi;
  const void* ki;
  const float* w;
  const float* q_scale;  // non-NULL: qi / ki are E4M3 (one byte per element)
  const float* k_scale;
  int Tq, Tk, Hi, d;
  const uint32_t* q_sf = nullptr;  // non-NULL: qi / ki are E4M3 with E8M0 block scales (MXFP8)
  const uint32_t* k_sf = nullptr;
  int elem_bytes() const { return (q_scale || q_sf) ? 1 : 2; }
};

int make_maps(const Inputs& in, CUtensorMap* mq, CUtensorMap* mk) {
  const CUtensorMapDataType dt = in.elem_bytes() == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t box = 128 / in.elem_bytes();  // one 128-byte swizzled chunk
  const uint64_t row = static_cast<uint64_t>(in.d) * in.elem_bytes();
  int rc = dsa::encode_tensor_map_2d(mq, in.qi, dt, in.d, static_cast<uint64_t>(in.Tq) * in.Hi, row, box, kNRows,
                                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != DSA_OK) return rc;
  return dsa::encode_tensor_map_2d(mk, in.ki, dt, in.d, in.Tk, row, box, kKeyTile, CU_TENSOR_MAP_SWIZZLE_128B);
}

void fill_params(IndexerParams& p, const Inputs& in, const Geom& g) {
  p.w = in.w;
  p.q_scale = in.q_scale;
  p.k_scale = in.k_scale;
  p.q_sf = in.q_sf;
  p.k_sf = in.k_sf;
  p.g = g;
  p.T = in.Tq;
  p.Tk = in.Tk;
  p.Hi = in.Hi;
  p.d = in.d;
  p.nch = in.d * in.elem_bytes() / 128;
  p.qb = kNRows / in.Hi;
  p.nblocks = (in.Tq + p.qb - 1) / p.qb;
  p.s_max = g.s_max;
  p.status = dsa::device_status_ptr();
}

bool is_plain(const Geom& g) { return g.cu_k == g.cu_q && g.ratio == 1 && !g.q_off; }

template <int FUSED, int HI, int GEN, int F8>
int launch_indexer_hi(const CUtensorMap& mq, const CUtensorMap& mk, IndexerParams& p, int sm_count,
                      cudaStream_t stream) {
  const int max_stages = FUSED ? 3 : 4;
  p.stages = p.nch == 1 ? 6 : max_stages;
  const SmemLayout L = smem_layout(p.nch, p.stages, p.qb, FUSED, F8 == 2);
  const size_t smem = L.total + 1024;
  if (cudaFuncSetAttribute(indexer_kernel<FUSED, HI, GEN, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return dsa::launch_error("indexer_kernel smem attribute");
  const int grid = p.nblocks < sm_count ? p.nblocks : sm_count;
  indexer_kernel<FUSED, HI, GEN, F8><<<grid, indexer_threads(FUSED), smem, stream>>>(mq, mk, p);
  return dsa::launch_error("indexer_kernel");
}

template <int FUSED, int GEN>
int launch_indexer_gen(const CUtensorMap& mq, const CUtensorMap& mk, IndexerParams& p, int sm_count,
                       cudaStream_t stream) {
  if (p.q_scale) {  // fp8 inputs: 32 or 64 heads (validated)
    return p.Hi == 32 ? launch_indexer_hi<FUSED, 32, GEN, 1>(mq, mk, p, sm_count, stream)
                      : launch_indexer_hi<FUSED, 64, GEN, 1>(mq, mk, p, sm_count, stream);
  }
  if (p.q_sf) {  // mxfp8 inputs: 32 or 64 heads (validated)
    return p.Hi == 32 ? launch_indexer_hi<FUSED, 32, GEN, 2>(mq, mk, p, sm_count, stream)
                      : launch_indexer_hi<FUSED, 64, GEN, 2>(mq, mk, p, sm_count, stream);
  }
  switch (p.Hi) {
    case 8: return launch_indexer_hi<FUSED, 8, GEN, 0>(mq, mk, p, sm_count, stream);
    case 16: return launch_indexer_hi<FUSED, 16, GEN, 0>(mq, mk, p, sm_count, stream);
    case 32: return launch_indexer_hi<FUSED, 32, GEN, 0>(mq, mk, p, sm_count, stream);
    default: return launch_indexer_hi<FUSED, 64, GEN, 0>(mq, mk, p, sm_count, stream);
  }
}

template <int FUSED>
int launch_indexer(const CUtensorMap& mq, const CUtensorMap& mk, IndexerParams& p, int sm_count, cudaStream_t stream) {
  return is_plain(p.g) ? launch_indexer_gen<FUSED, 0>(mq, mk, p, sm_count, stream)
                       : launch_indexer_gen<FUSED, 1>(mq, mk, p, sm_count, stream);
}

// Candidate capacity per row: four equal segments, one per key quarter of a
// 128-key tile.  A row touches at most ceil(s_max/128)+1 tiles and a segment
// receives at most 32 keys per tile, so short rows hold every key they could
// emit; long rows get max(4096, 2k) per segment, which the running threshold
// normally keeps far from full, and a segment that does fill is compacted to
// its top-k in place (fused_compact says when that can happen).
int64_t fused_whole(int s_max) { return 32ll * ((s_max + kKeyTile - 1) / kKeyTile + 1); }
int64_t fused_bound(int k) { return 2ll * k > 4096 ? 2ll * k : 4096; }
int fused_cap(int s_max, int k) {
  const int64_t whole = fused_whole(s_max), bound = fused_bound(k);
  return static_cast<int>(4 * (whole < bound ? whole : bound));
}
int fused_compact(int s_max, int k) { return fused_whole(s_max) > fused_bound(k) ? 1 : 0; }

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Dense scores (arguments already validated).
int run_dense(const Inputs& in, const Geom& g, float* scores, int64_t ld, int sms, cudaStream_t stream) {
  CUtensorMap mq, mk;
  int rc = make_maps(in, &mq, &mk);
  if (rc != DSA_OK) return rc;
  IndexerParams p{};
  fill_params(p, in, g);
  p.scores = scores;
  p.ld = ld;
  return launch_indexer<0>(mq, mk, p, sms, stream);
}

}  // namespace

extern "C" int dsa_indexer_scores(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens,
                                  int n_docs, int T, int Hi, int d, int s_max, float* scores, int64_t ld,
                                  cudaStream_t stream) {
  dsa::clear_error();
  int rc = validate_indexer(qi, ki, w, cu_seqlens, n_docs, T, Hi, d, s_max, "dsa_indexer_scores");
  if (rc != DSA_OK) return rc;
  if (!scores) return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_scores: NULL scores");
  if (ld < s_max || ld % 4 != 0) return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_scores: need ld >= s_max, ld % 4 == 0");
  int sms = 0;
  rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  return run_dense(Inputs{qi, ki, w, nullptr, nullptr, T, T, Hi, d}, plain_geom(cu_seqlens, n_docs, s_max), scores, ld,
                   sms, stream);
}

extern "C" int dsa_indexer_scores_ratio(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens_q,
                                        const int32_t* cu_seqlens_k, const int32_t* q_causal_offsets, int n_docs,
                                        int Tq, int Tk, int Hi, int d, int ratio, int s_max, float* scores, int64_t ld,
                                        cudaStream_t stream) {
  dsa::clear_error();
  int rc = validate_ratio(qi, ki, w, cu_seqlens_q, cu_seqlens_k, n_docs, Tq, Tk, Hi, d, ratio, s_max,
                          "dsa_indexer_scores_ratio");
  if (rc != DSA_OK) return rc;
  if (!scores) return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_scores_ratio: NULL scores");
  if (ld < s_max || ld % 4 != 0)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_scores_ratio: need ld >= s_max, ld % 4 == 0");
  int sms = 0;
  rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  const Geom g{cu_seqlens_q, cu_seqlens_k, q_causal_offsets, n_docs, ratio, s_max};
  return run_dense(Inputs{qi, ki, w, nullptr, nullptr, Tq, Tk, Hi, d}, g, scores, ld, sms, stream);
}

// Workspace of the fused path: per-row segment counts [T][4], per-row final
// threshold bins [T] (two keys), then the candidate segments [T][cap].
size_t ws_tau_offset(int T) { return align256(static_cast<size_t>(T) * 16); }
size_t ws_cand_offset(int T) { return ws_tau_offset(T) + align256(static_cast<size_t>(T) * 8); }

extern "C" size_t dsa_indexer_topk_workspace_size(int T, int Hi, int d, int k, int s_max) {
  if (T < 1 || Hi < 1 || d < 1 || k < 1 || k > DSA_MAX_TOPK || s_max < 1) return 0;
  const size_t cap = static_cast<size_t>(fused_cap(s_max, k));
  return ws_cand_offset(T) + align256(static_cast<size_t>(T) * cap * 8);
}

namespace {

int check_workspace(int T, int Hi, int d, int k, int s_max, const void* workspace, size_t ws_bytes, const char* fn) {
  if (k < 1 || k > DSA_MAX_TOPK) return dsa::set_error(DSA_ERR_VALUE, "%s: need 1 <= k <= %d", fn, DSA_MAX_TOPK);
  const size_t need = dsa_indexer_topk_workspace_size(T, Hi, d, k, s_max);
  if (!workspace || ws_bytes < need || !dsa::aligned(workspace, 256))
    return dsa::set_error(DSA_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned and >= %zu bytes", fn, need);
  return DSA_OK;
}

// Stage 1 launch (arguments already validated).
int run_candidates(const Inputs& in, const Geom& g, int k, void* workspace, int sms, cudaStream_t stream) {
  CUtensorMap mq, mk;
  int rc = make_maps(in, &mq, &mk);
  if (rc != DSA_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int Tq = in.Tq;
  IndexerParams p{};
  fill_params(p, in, g);
  p.cand_cnt = reinterpret_cast<int32_t*>(ws);
  p.cand_tau = reinterpret_cast<uint2*>(ws + ws_tau_offset(Tq));
  p.cand = reinterpret_cast<uint2*>(ws + ws_cand_offset(Tq));
  p.cap = fused_cap(g.s_max, k);
  p.compact = fused_compact(g.s_max, k);
  p.k = k;
  int bins = kHistWords / p.qb;
  int bits = 0;
  while ((1 << bits) < bins) ++bits;
  p.hist_bits = bits;
  return launch_indexer<1>(mq, mk, p, sms, stream);
}

// Stage 2 launch (arguments already validated).
// True when stage 2 runs its multi-row form (the only form that can also write logits).
bool select_is_fast(int s_max, int) { return s_max <= kSelMaxLen; }

template <int GEN>
int run_select_gen(const Geom& g, int T, int k, void* workspace, int32_t* idx, int32_t* topk_length, float* logits,
                   int sms, cudaStream_t stream) {
  const int cap = fused_cap(g.s_max, k);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int32_t* cand_cnt = reinterpret_cast<const int32_t*>(ws);
  const uint2* cand_tau = reinterpret_cast<const uint2*>(ws + ws_tau_offset(T));
  const uint2* cand = reinterpret_cast<const uint2*>(ws + ws_cand_offset(T));
  uint32_t* status = dsa::device_status_ptr();
  if (select_is_fast(g.s_max, k)) {
    const size_t smem = sizeof(MultiShared);
    if (cudaFuncSetAttribute(fused_select_multi_kernel<GEN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return dsa::launch_error("fused_select_multi_kernel smem attribute");
    const int grid = T < kMCtasPerSm * sms ? T : kMCtasPerSm * sms;
    fused_select_multi_kernel<GEN><<<grid, kMThreads, smem, stream>>>(g, T, k, cand, cand_cnt, cand_tau, cap, idx,
                                                                      topk_length, logits, status);
    return dsa::launch_error("fused_select_multi_kernel");
  }
  const size_t smem = sizeof(dsa::TopkShared);
  if (cudaFuncSetAttribute(fused_select_kernel<GEN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return dsa::launch_error("fused_select_kernel smem attribute");
  fused_select_kernel<GEN><<<T, dsa::kTopkThreads, smem, stream>>>(g, T, k, cand, cand_cnt, cap, idx, topk_length,
                                                                   status);
  return dsa::launch_error("fused_select_kernel");
}

int run_select(const Geom& g, int T, int k, void* workspace, int32_t* idx, int32_t* topk_length, float* logits,
               int sms, cudaStream_t stream) {
  return is_plain(g) ? run_select_gen<0>(g, T, k, workspace, idx, topk_length, logits, sms, stream)
                     : run_select_gen<1>(g, T, k, workspace, idx, topk_length, logits, sms, stream);
}

// Both stages plus the optional outputs of the pages' combined call (arguments
// already validated; logits may be NULL only when softmax and lse are).
int run_fused(const Inputs& in, const Geom& g, int k, int32_t* idx, int32_t* topk_length, float* logits,
              float* softmax, float* lse, void* workspace, int sms, cudaStream_t stream) {
  int rc = run_candidates(in, g, k, workspace, sms, stream);
  if (rc != DSA_OK) return rc;
  rc = run_select(g, in.Tq, k, workspace, idx, topk_length, logits, sms, stream);
  if (rc != DSA_OK || (!softmax && !lse)) return rc;
  return dsa_topk_softmax(logits, idx, in.Tq, k, softmax, lse, stream);
}

}  // namespace

extern "C" int dsa_indexer_candidates(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens,
                                      int n_docs, int T, int Hi, int d, int k, int s_max, void* workspace,
                                      size_t ws_bytes, cudaStream_t stream) {
  dsa::clear_error();
  int rc = validate_indexer(qi, ki, w, cu_seqlens, n_docs, T, Hi, d, s_max, "dsa_indexer_candidates");
  if (rc != DSA_OK) return rc;
  rc = check_workspace(T, Hi, d, k, s_max, workspace, ws_bytes, "dsa_indexer_candidates");
  if (rc != DSA_OK) return rc;
  int sms = 0;
  rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  return run_candidates(Inputs{qi, ki, w, nullptr, nullptr, T, T, Hi, d}, plain_geom(cu_seqlens, n_docs, s_max), k,
                        workspace, sms, stream);
}

extern "C" int dsa_select_candidates(const int32_t* cu_seqlens, int n_docs, int T, int Hi, int d, int k, int s_max,
                                     const void* workspace, size_t ws_bytes, int32_t* idx, int32_t* topk_length,
                                     cudaStream_t stream) {
  dsa::clear_error();
  if (!cu_seqlens) return dsa::set_error(DSA_ERR_VALUE, "dsa_select_candidates: NULL cu_seqlens");
  if (n_docs < 1 || T < 1) return dsa::set_error(DSA_ERR_VALUE, "dsa_select_candidates: need n_docs >= 1 and T >= 1");
  if (s_max < 1 || s_max > T) return dsa::set_error(DSA_ERR_VALUE, "dsa_select_candidates: need 1 <= s_max <= T");
  if (!idx) return dsa::set_error(DSA_ERR_VALUE, "dsa_select_candidates: NULL idx");
  int rc = check_workspace(T, Hi, d, k, s_max, workspace, ws_bytes, "dsa_select_candidates");
  if (rc != DSA_OK) return rc;
  int sms = 0;
  rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  return run_select(plain_geom(cu_seqlens, n_docs, s_max), T, k, const_cast<void*>(workspace), idx, topk_length,
                    nullptr, sms, stream);
}

extern "C" int dsa_indexer_topk(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens, int n_docs,
                                int T, int Hi, int d, int k, int s_max, int32_t* idx, int32_t* topk_length,
                                void* workspace, size_t ws_bytes, cudaStream_t stream) {
  dsa::clear_error();
  int rc = validate_indexer(qi, ki, w, cu_seqlens, n_docs, T, Hi, d, s_max, "dsa_indexer_topk");
  if (rc != DSA_OK) return rc;
  if (!idx) return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_topk: NULL idx");
  rc = check_workspace(T, Hi, d, k, s_max, workspace, ws_bytes, "dsa_indexer_topk");
  if (rc != DSA_OK) return rc;
  int sms = 0;
  rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  return run_fused(Inputs{qi, ki, w, nullptr, nullptr, T, T, Hi, d}, plain_geom(cu_seqlens, n_docs, s_max), k, idx,
                   topk_length, nullptr, nullptr, nullptr, workspace, sms, stream);
}

// The fused call with the outputs that come with the indices on the pages'
// combined indexer + top-k: aligned logits, and optionally their softmax and
// log-sum-exp (dsa_topk_softmax over the logits).
extern "C" int dsa_indexer_topk_ex(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens,
                                   int n_docs, int T, int Hi, int d, int k, int s_max, int32_t* idx,
                                   int32_t* topk_length, float* logits, float* softmax, float* lse, void* workspace,
                                   size_t ws_bytes, cudaStream_t stream) {
  dsa::clear_error();
  int rc = validate_indexer(qi, ki, w, cu_seqlens, n_docs, T, Hi, d, s_max, "dsa_indexer_topk_ex");
  if (rc != DSA_OK) return rc;
  if (!idx || !logits) return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_topk_ex: NULL idx or logits");
  rc = check_workspace(T, Hi, d, k, s_max, workspace, ws_bytes, "dsa_indexer_topk_ex");
  if (rc != DSA_OK) return rc;
  if (!select_is_fast(s_max, k))
    return dsa::set_error(DSA_ERR_UNSUPPORTED,
                          "dsa_indexer_topk_ex: logits need rows of at most %d columns (s_max = %d)", kSelMaxLen, s_max);
  int sms = 0;
  rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  return run_fused(Inputs{qi, ki, w, nullptr, nullptr, T, T, Hi, d}, plain_geom(cu_seqlens, n_docs, s_max), k, idx,
                   topk_length, logits, softmax, lse, workspace, sms, stream);
}

// The combined call over a compressed key prefix with the ratio-causal mask
// (cuDNN DSA page, sections 3 and 4): ids are global key rows cu_k[b] + j.
extern "C" int dsa_indexer_topk_ratio(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens_q,
                                      const int32_t* cu_seqlens_k, const int32_t* q_causal_offsets, int n_docs, int Tq,
                                      int Tk, int Hi, int d, int ratio, int k, int s_max, int32_t* idx,
                                      int32_t* topk_length, float* logits, float* softmax, float* lse,
                                      void* workspace, size_t ws_bytes, cudaStream_t stream) {
  dsa::clear_error();
  int rc = validate_ratio(qi, ki, w, cu_seqlens_q, cu_seqlens_k, n_docs, Tq, Tk, Hi, d, ratio, s_max,
                          "dsa_indexer_topk_ratio");
  if (rc != DSA_OK) return rc;
  if (!idx) return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_topk_ratio: NULL idx");
  if ((softmax || lse) && !logits)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_topk_ratio: softmax and lse need logits");
  rc = check_workspace(Tq, Hi, d, k, s_max, workspace, ws_bytes, "dsa_indexer_topk_ratio");
  if (rc != DSA_OK) return rc;
  if (logits && !select_is_fast(s_max, k))
    return dsa::set_error(DSA_ERR_UNSUPPORTED,
                          "dsa_indexer_topk_ratio: logits need rows of at most %d columns (s_max = %d)", kSelMaxLen,
                          s_max);
  int sms = 0;
  rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  const Geom g{cu_seqlens_q, cu_seqlens_k, q_causal_offsets, n_docs, ratio, s_max};
  return run_fused(Inputs{qi, ki, w, nullptr, nullptr, Tq, Tk, Hi, d}, g, k, idx, topk_length, logits, softmax, lse,
                   workspace, sms, stream);
}

// ---- FP8 inputs (cuDNN DSA page, section 3 precision path "fp8": E4M3 Q/K
// with fp32 descales, one per (token, head) for Q and per key row for K).
namespace {
int validate_fp8(const void* qi8, const void* ki8, const float* q_scale, const float* k_scale, const float* w,
                 const int32_t* cu_q, const int32_t* cu_k, int n_docs, int Tq, int Tk, int Hi, int d, int ratio,
                 int s_max, const char* fn) {
  int rc = validate_ratio(qi8, ki8, w, cu_q, cu_k, n_docs, Tq, Tk, Hi, d, ratio, s_max, fn);
  if (rc != DSA_OK) return rc;
  if (!q_scale || !k_scale) return dsa::set_error(DSA_ERR_VALUE, "%s: NULL q_scale or k_scale", fn);
  if (d != 128 || (Hi != 32 && Hi != 64))
    return dsa::set_error(DSA_ERR_VALUE, "%s: fp8 inputs need d = 128 and Hi in {32, 64} (got d %d, Hi %d)", fn, d, Hi);
  return DSA_OK;
}
}  // namespace

extern "C" int dsa_indexer_scores_fp8(const void* qi8, const void* ki8, const float* q_scale, const float* k_scale,
                                      const float* w, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                      const int32_t* q_causal_offsets, int n_docs, int Tq, int Tk, int Hi, int d,
                                      int ratio, int s_max, float* scores, int64_t ld, cudaStream_t stream) {
  dsa::clear_error();
  int rc = validate_fp8(qi8, ki8, q_scale, k_scale, w, cu_seqlens_q, cu_seqlens_k, n_docs, Tq, Tk, Hi, d, ratio, s_max,
                        "dsa_indexer_scores_fp8");
  if (rc != DSA_OK) return rc;
  if (!scores) return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_scores_fp8: NULL scores");
  if (ld < s_max || ld % 4 != 0)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_scores_fp8: need ld >= s_max, ld % 4 == 0");
  int sms = 0;
  rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  const Geom g{cu_seqlens_q, cu_seqlens_k, q_causal_offsets, n_docs, ratio, s_max};
  return run_dense(Inputs{qi8, ki8, w, q_scale, k_scale, Tq, Tk, Hi, d}, g, scores, ld, sms, stream);
}

extern "C" int dsa_indexer_topk_fp8(const void* qi8, const void* ki8, const float* q_scale, const float* k_scale,
                                    const float* w, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                    const int32_t* q_causal_offsets, int n_docs, int Tq, int Tk, int Hi, int d,
                                    int ratio, int k, int s_max, int32_t* idx, int32_t* topk_length, float* logits,
                                    float* softmax, float* lse, void* workspace, size_t ws_bytes,
                                    cudaStream_t stream) {
  dsa::clear_error();
  int rc = validate_fp8(qi8, ki8, q_scale, k_scale, w, cu_seqlens_q, cu_seqlens_k, n_docs, Tq, Tk, Hi, d, ratio, s_max,
                        "dsa_indexer_topk_fp8");
  if (rc != DSA_OK) return rc;
  if (!idx) return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_topk_fp8: NULL idx");
  if ((softmax || lse) && !logits)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_topk_fp8: softmax and lse need logits");
  rc = check_workspace(Tq, Hi, d, k, s_max, workspace, ws_bytes, "dsa_indexer_topk_fp8");
  if (rc != DSA_OK) return rc;
  if (logits && !select_is_fast(s_max, k))
    return dsa::set_error(DSA_ERR_UNSUPPORTED,
                          "dsa_indexer_topk_fp8: logits need rows of at most %d columns (s_max = %d)", kSelMaxLen,
                          s_max);
  int sms = 0;
  rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  const Geom g{cu_seqlens_q, cu_seqlens_k, q_causal_offsets, n_docs, ratio, s_max};
  return run_fused(Inputs{qi8, ki8, w, q_scale, k_scale, Tq, Tk, Hi, d}, g, k, idx, topk_length, logits, softmax, lse,
                   workspace, sms, stream);
}

// ---- MXFP8 inputs (cuDNN DSA page, section 3 precision path "mxfp8": E4M3
// Q/K with block-scaled E8M0 scales, one per 32 elements of d).
namespace {
int validate_mxfp8(const void* qi8, const void* ki8, const uint8_t* q_sf, const uint8_t* k_sf, const float* w,
                   const int32_t* cu_q, const int32_t* cu_k, int n_docs, int Tq, int Tk, int Hi, int d, int ratio,
                   int s_max, const char* fn) {
  int rc = validate_ratio(qi8, ki8, w, cu_q, cu_k, n_docs, Tq, Tk, Hi, d, ratio, s_max, fn);
  if (rc != DSA_OK) return rc;
  if (!q_sf || !k_sf) return dsa::set_error(DSA_ERR_VALUE, "%s: NULL q_sf or k_sf", fn);
  if (!dsa::aligned(q_sf, 4) || !dsa::aligned(k_sf, 4))
    return dsa::set_error(DSA_ERR_VALUE, "%s: q_sf and k_sf must be 4-byte aligned", fn);
  if (d != 128 || (Hi != 32 && Hi != 64))
    return dsa::set_error(DSA_ERR_VALUE, "%s: mxfp8 inputs need d = 128 and Hi in {32, 64} (got d %d, Hi %d)", fn, d,
                          Hi);
  return DSA_OK;
}
Inputs mx_inputs(const void* qi8, const void* ki8, const uint8_t* q_sf, const uint8_t* k_sf, const float* w, int Tq,
                 int Tk, int Hi, int d) {
  Inputs in{qi8, ki8, w, nullptr, nullptr, Tq, Tk, Hi, d};
  in.q_sf = reinterpret_cast<const uint32_t*>(q_sf);
  in.k_sf = reinterpret_cast<const uint32_t*>(k_sf);
  return in;
}
}  // namespace

extern "C" int dsa_indexer_scores_mxfp8(const void* qi8, const void* ki8, const uint8_t* q_sf, const uint8_t* k_sf,
                                        const float* w, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                        const int32_t* q_causal_offsets, int n_docs, int Tq, int Tk, int Hi, int d,
                                        int ratio, int s_max, float* scores, int64_t ld, cudaStream_t stream) {
  dsa::clear_error();
  int rc = validate_mxfp8(qi8, ki8, q_sf, k_sf, w, cu_seqlens_q, cu_seqlens_k, n_docs, Tq, Tk, Hi, d, ratio, s_max,
                          "dsa_indexer_scores_mxfp8");
  if (rc != DSA_OK) return rc;
  if (!scores) return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_scores_mxfp8: NULL scores");
  if (ld < s_max || ld % 4 != 0)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_scores_mxfp8: need ld >= s_max, ld % 4 == 0");
  int sms = 0;
  rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  const Geom g{cu_seqlens_q, cu_seqlens_k, q_causal_offsets, n_docs, ratio, s_max};
  return run_dense(mx_inputs(qi8, ki8, q_sf, k_sf, w, Tq, Tk, Hi, d), g, scores, ld, sms, stream);
}

extern "C" int dsa_indexer_topk_mxfp8(const void* qi8, const void* ki8, const uint8_t* q_sf, const uint8_t* k_sf,
                                      const float* w, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                      const int32_t* q_causal_offsets, int n_docs, int Tq, int Tk, int Hi, int d,
                                      int ratio, int k, int s_max, int32_t* idx, int32_t* topk_length, float* logits,
                                      float* softmax, float* lse, void* workspace, size_t ws_bytes,
                                      cudaStream_t stream) {
  dsa::clear_error();
  int rc = validate_mxfp8(qi8, ki8, q_sf, k_sf, w, cu_seqlens_q, cu_seqlens_k, n_docs, Tq, Tk, Hi, d, ratio, s_max,
                          "dsa_indexer_topk_mxfp8");
  if (rc != DSA_OK) return rc;
  if (!idx) return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_topk_mxfp8: NULL idx");
  if ((softmax || lse) && !logits)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_topk_mxfp8: softmax and lse need logits");
  rc = check_workspace(Tq, Hi, d, k, s_max, workspace, ws_bytes, "dsa_indexer_topk_mxfp8");
  if (rc != DSA_OK) return rc;
  if (logits && !select_is_fast(s_max, k))
    return dsa::set_error(DSA_ERR_UNSUPPORTED,
                          "dsa_indexer_topk_mxfp8: logits need rows of at most %d columns (s_max = %d)", kSelMaxLen,
                          s_max);
  int sms = 0;
  rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  const Geom g{cu_seqlens_q, cu_seqlens_k, q_causal_offsets, n_docs, ratio, s_max};
  return run_fused(mx_inputs(qi8, ki8, q_sf, k_sf, w, Tq, Tk, Hi, d), g, k, idx, topk_length, logits, softmax, lse,
                   workspace, sms, stream);
}

// ---------------------------------------------------------------------------
// dsa_indexer_topk_noalloc: the fused call with its scratch in a fixed,
// file-scope device array instead of a caller-provided workspace.  The array
// is DSA_NOALLOC_SCRATCH_BYTES long and exists on every GPU that loads this
// library until the process exits.  Host code cannot pass the array's name to
// a kernel (on the host it is only a stand-in symbol), so the first call on
// each device looks up its device address with cudaGetSymbolAddress while that
// device is current and caches it.
static __device__ __align__(256) uint8_t g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kNoAllocMaxDevices];
}  // namespace

extern "C" int dsa_indexer_topk_noalloc(const void* qi, const void* ki, const float* w, const int32_t* cu_seqlens,
                                        int n_docs, int T, int Hi, int d, int k, int s_max, int32_t* idx,
                                        int32_t* topk_length, cudaStream_t stream) {
  dsa::clear_error();
  int rc = validate_indexer(qi, ki, w, cu_seqlens, n_docs, T, Hi, d, s_max, "dsa_indexer_topk_noalloc");
  if (rc != DSA_OK) return rc;
  if (k < 1 || k > DSA_MAX_TOPK)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_indexer_topk_noalloc: need 1 <= k <= %d", DSA_MAX_TOPK);
  const size_t need = dsa_indexer_topk_workspace_size(T, Hi, d, k, s_max);
  if (need > DSA_NOALLOC_SCRATCH_BYTES)
    return dsa::set_error(DSA_ERR_WORKSPACE,
                          "dsa_indexer_topk_noalloc: these shapes need %zu bytes of scratch but the fixed array holds "
                          "%zu; call dsa_indexer_topk with a workspace instead",
                          need, static_cast<size_t>(DSA_NOALLOC_SCRATCH_BYTES));
  rc = dsa::check_device(nullptr);
  if (rc != DSA_OK) return rc;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
    cudaGetLastError();
    return dsa::set_error(DSA_ERR_UNSUPPORTED, "dsa_indexer_topk_noalloc: unusable device ordinal");
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return dsa::set_error(DSA_ERR_CUDA, "dsa_indexer_topk_noalloc: cannot resolve the scratch array: %s",
                              cudaGetErrorString(e));
      }
      g_noalloc_addr[dev] = p;
    }
    scratch = g_noalloc_addr[dev];
  }
  return dsa_indexer_topk(qi, ki, w, cu_seqlens, n_docs, T, Hi, d, k, s_max, idx, topk_length, scratch,
                          DSA_NOALLOC_SCRATCH_BYTES, stream);
}
