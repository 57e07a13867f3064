// attention_bwd.cu -- sparse MQA attention backward on tcgen05 (cuDNN Frontend
// DSA page, section 2 Sparse Attention Backward: q, the latent kv (K = V),
// out, dout, the KV-only lse, the sink and the top-k ids in; dq, dkv and
// d_sink out).  With the forward's s_j = scale * q . k_j over the valid
// slots and L = logaddexp(lse_kv, sink):
//   P_j = exp(s_j - L),  dS_j = P_j * (dout . v_j - dout . out),
//   dq = scale * sum_j dS_j k_j,
//   dkv[id_j] += scale * dS_j q  (+ P_j dout on the value dims),
//   d_sink = -sum over rows of exp(sink - L) * (dout . out).
//
// Four launches, all deterministic in this variant (no floating-point atomics):
//  1. bwd_prep_kernel: per (token, head) the log2-domain normaliser L and
//     delta = dout . out, and the row's d_sink term.
//  2. bwd_dq_kernel: per unit (token, 64-head group), in 64-key tiles: the
//     selected kv rows are gathered as in the forward; one MMA sequence
//     (M = 64 keys, N = 128) computes S^T and dP^T together, the query and
//     dout rows of the unit standing side by side as its B operand; eight
//     warps form P and scale * dS from them, write both to global memory for
//     launch 3 and dS^T (bf16) to shared memory; a second MMA sequence
//     accumulates dq^T = K^T . dS^T in TMEM (four M = 128 blocks and one
//     M = 64 block for dims 512..575).  The kv tile buffer is single: the
//     query and dout rows take the room of the forward's second buffer.
//  3. bwd_dkv_kernel: 152 lanes (one per SM); lane c owns one fp32 copy
//     ("shard") of dkv and takes tokens c, c + 152, ... in order.  Per
//     64-slot tile one MMA sequence forms the tile's key rows
//     [scale dS | P] . [q ; dout] (M = 64 keys, K = 128, N = 128 dims at a
//     time) in TMEM, and the drain warps add them into the lane's shard:
//     each row has one writer per block and the tiles go in slot order, so
//     every shard value receives its terms in a fixed order with no race
//     (repeated ids within a tile are first folded in slot order).
//  4. bwd_reduce_*_kernel: dkv = the shards summed in lane order; d_sink =
//     the row terms summed in row order.
// The non-deterministic variant (the pages' default) runs the same launches
// except that bwd_dkv_kernel<true> adds each slot's dkv row straight into
// dkv with fp32 vector atomics (red.global.add on 16 bytes), so there are no
// shards to read, write or reduce and the updates are served by L2.
#include <climits>

#include "common.cuh"

namespace {

constexpr int kKeys = 64;
constexpr int kHG = 64;
constexpr int kDqk = 576, kDv = 512;
constexpr int kNqk = kDqk / 64;  // 9 chunks of 64 dims
constexpr int kNv = kDv / 64;    // 8
constexpr uint32_t kChunkBytes = kKeys * 128;  // 64 rows x 64 bf16
constexpr int kGatherWarps = 6;
constexpr int kGatherThreads = kGatherWarps * 32;
constexpr int kGatherKeys = kGatherThreads / 8;
constexpr int kGatherSteps = (kKeys + kGatherKeys - 1) / kGatherKeys;
constexpr int kMmaWarp = kGatherWarps;       // S/dP product, query + dout loads
constexpr int kSoftWarp0 = kMmaWarp + 1;
constexpr int kSoftWarps = 8;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kMma2Warp = kSoftWarp0 + kSoftWarps;  // dq product
constexpr int kThreads = (kMma2Warp + 1) * 32;      // 512
constexpr uint32_t kTmemCols = 512;
constexpr int kSCol = 0;     // S^T at columns 0..63, dP^T at 64..127
constexpr int kQCol = 128;   // dq^T blocks at 128 + 64*m (m = 0..3), the M = 64 block at 384
constexpr int kLanes = 152;  // dkv shards: one CTA per SM of a GB300 in the dkv pass
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ shared
struct DqLayout {
  uint32_t qd, kv, ds, small, bars, misc, total;
};
// qd: for c < 8, 16 KB = query chunk c (64 heads) then dout chunk c; then the
// query's chunk 8 (8 KB).  kv: 9 chunks.  ds: dS^T, 64 keys x 64 heads.
__host__ __device__ inline DqLayout dq_layout() {
  DqLayout L;
  uint32_t o = 0;
  L.qd = o;
  o += kNv * 2 * kChunkBytes + kChunkBytes;
  L.kv = o;
  o += kNqk * kChunkBytes;
  L.ds = o;
  o += kChunkBytes;
  L.small = o;
  o += 2 * kHG * 4;  // L2 | delta of the unit's heads
  L.bars = o;
  o += 16 * 8;
  L.misc = o;
  o += 16;
  L.total = o;
  return L;
}

struct BwdParams {
  const int32_t* idx;
  const int32_t* topk_length;
  const uint8_t* kv;  // latent rows, kDqk bf16
  const float2* stats;  // [T, H]: (log2-domain L, delta)
  __nv_bfloat16* dq;    // [T, H, kDqk]
  __nv_bfloat16* ds_g;  // [T, K, Hp]: scale * dS
  __nv_bfloat16* p_g;   // [T, K, Hp]: P
  uint32_t* status;
  int T, Tkv, H, G, K, Hp;
  float scale, scale_log2;
};

__device__ __forceinline__ int unit_len(const BwdParams& p, int t) {
  int L = p.K;
  if (p.topk_length) {
    L = __ldg(p.topk_length + t);
    L = L < 0 ? 0 : (L > p.K ? p.K : L);
  }
  return L;
}

__device__ __forceinline__ bool elect_sync() {
  uint32_t is = 0;
  asm volatile(
      "{\n .reg .pred P;\n elect.sync _|P, 0xffffffff;\n selp.u32 %0, 1, 0, P;\n}" : "=r"(is));
  return is != 0;
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
               "r"(src_bytes), "l"(policy)
               : "memory");
}

// ------------------------------------------------------------- 1. prep
// One warp per (token, head): delta = dout . out (fp32 over bf16 inputs),
// L = logaddexp(lse_kv, sink) (+inf for an empty row, whose lse_kv is +inf),
// stored as (L * log2(e), delta), and the row's d_sink term
// -exp(sink - L) * delta.
__global__ void bwd_prep_kernel(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
                                const float* __restrict__ lse_kv, const float* __restrict__ sink, int64_t rows, int H,
                                float2* __restrict__ stats, float* __restrict__ dsink_part) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint4* o4 = reinterpret_cast<const uint4*>(out + r * kDv);
  const uint4* d4 = reinterpret_cast<const uint4*>(dout + r * kDv);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {  // 512 bf16 = 64 x 16 bytes, two per lane
    const uint4 a = __ldg(o4 + lane + 32 * i), b = __ldg(d4 + lane + 32 * i);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __bfloat1622float2(a2[e]), y = __bfloat1622float2(b2[e]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    const int h = static_cast<int>(r % H);
    const float l = __ldg(lse_kv + r);
    const float sk = sink ? __ldg(sink + h) : -INFINITY;
    float L;
    if (l == INFINITY || sk == INFINITY) {
      L = INFINITY;
    } else {
      const float m = fmaxf(l, sk);
      L = m == -INFINITY ? -INFINITY : m + logf(expf(l - m) + expf(sk - m));
    }
    stats[r] = make_float2(L * kLog2e, acc);
    dsink_part[r] = (sink && L != INFINITY) ? -expf(sk - L) * acc : 0.f;
  }
}

// --------------------------------------------------------------- 2. dq
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                  const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dsa::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const DqLayout L = dq_layout();
  uint8_t* qd = smem + L.qd;
  uint8_t* kvbuf = smem + L.kv;
  uint8_t* dsbuf = smem + L.ds;
  float* l2s = reinterpret_cast<float*>(smem + L.small);
  float* dls = l2s + kHG;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + 1;
  uint64_t* s_full = bars + 2;
  uint64_t* s_empty = bars + 3;
  uint64_t* p_full = bars + 4;
  uint64_t* q_full = bars + 5;
  uint64_t* q_empty = bars + 6;
  uint64_t* o_done = bars + 7;
  uint64_t* drain = bars + 8;  // [2]: the MMA issuers' exit commits
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_units = p.T * p.G;

  if (threadIdx.x == 0) {
    dsa::mbar_init(&drain[0], 1);
    dsa::mbar_init(&drain[1], 1);
    dsa::mbar_init(kv_full, kGatherThreads);
    dsa::mbar_init(kv_empty, 1);
    dsa::mbar_init(s_full, 1);
    dsa::mbar_init(s_empty, kSoftWarps);
    dsa::mbar_init(p_full, kSoftWarps);
    dsa::mbar_init(q_full, 1);
    dsa::mbar_init(q_empty, 1);
    dsa::mbar_init(o_done, 1);
    *abort_flag = 0;
    dsa::fence_barrier_init();
  }
  if (warp == kMmaWarp) dsa::tmem_alloc(tmem_slot, kTmemCols);
  dsa::tc_fence_before();
  __syncthreads();
  dsa::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const dsa::Waiter wt = dsa::make_waiter(abort_flag, p.status);

  if (warp < kGatherWarps) {
    // ------------------------------------------------------------ gather
    // as in the forward: thread g covers piece (g & 7) of key (g >> 3) +
    // kGatherKeys * kg for all nine 64-dim chunks; one tile buffer
    const int g = threadIdx.x;
    const int piece = g & 7;
    const uint64_t keep = dsa::l2_policy_evict_last();
    uint32_t tile_ctr = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int uu = n_units - 1 - u;
      const int t = uu / p.G;
      const int len = unit_len(p, t);
      const int nt = (len + kKeys - 1) / kKeys;
      const int32_t* irow = p.idx + static_cast<int64_t>(t) * p.K;
      int nxt[kGatherSteps];
#pragma unroll
      for (int kg = 0; kg < kGatherSteps; ++kg) {
        const int j = kg * kGatherKeys + (g >> 3);
        nxt[kg] = (j < kKeys && j < len) ? __ldcs(irow + j) : -1;
      }
      for (int i = 0; i < nt; ++i, ++tile_ctr) {
        int id[kGatherSteps];
#pragma unroll
        for (int kg = 0; kg < kGatherSteps; ++kg) {
          id[kg] = (nxt[kg] >= 0 && nxt[kg] < p.Tkv) ? nxt[kg] : -1;
          const int jk = kg * kGatherKeys + (g >> 3);
          const int j = (i + 1) * kKeys + jk;
          nxt[kg] = (i + 1 < nt && jk < kKeys && j < len) ? __ldcs(irow + j) : -1;
        }
        if (!dsa::mbar_wait(kv_empty, (tile_ctr & 1) ^ 1, wt)) { ok = false; break; }
        dsa::fence_proxy_async_smem();
        const uint32_t buf = dsa::smem_u32(kvbuf);
#pragma unroll
        for (int kg = 0; kg < kGatherSteps; ++kg) {
          const int key = kg * kGatherKeys + (g >> 3);
          if (key >= kKeys) continue;
          const uint32_t nbytes = id[kg] >= 0 ? 16u : 0u;
          const int64_t row = id[kg] >= 0 ? id[kg] : 0;
          const uint8_t* krow = p.kv + row * (kDqk * 2) + piece * 16;
          for (int c = 0; c < kNqk; ++c)
            cp_async16(buf + c * kChunkBytes + dsa::sw128_offset(key, piece * 16), krow + c * 128, nbytes, keep);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        dsa::mbar_arrive(kv_full);
      }
    }
  } else if (warp == kMmaWarp || warp == kMma2Warp) {
    const bool leader = elect_sync();
    const uint32_t kv_addr = dsa::smem_u32(kvbuf);
    auto next_unit = [&](int u) {
      for (; u < n_units; u += gridDim.x)
        if (unit_len(p, (n_units - 1 - u) / p.G) > 0) return u;
      return n_units;
    };
    auto unit_tiles = [&](int u) { return (unit_len(p, (n_units - 1 - u) / p.G) + kKeys - 1) / kKeys; };
    if (warp == kMmaWarp) {
      // S^T and dP^T of a tile in one sequence: D[key, n] for n < 64 is
      // kv . q (dims 0..575), for n >= 64 kv . dout (dims 0..511)
      constexpr uint32_t idesc_qd = dsa::idesc_bf16(kKeys, 2 * kHG, 0, 0);
      constexpr uint32_t idesc_q = dsa::idesc_bf16(kKeys, kHG, 0, 0);
      const uint64_t qd_desc = dsa::smem_desc(dsa::smem_u32(qd), 16, 1024, dsa::kSwizzle128B);
      const uint64_t kv_desc = dsa::smem_desc(kv_addr, 16, 1024, dsa::kSwizzle128B);
      const uint64_t policy = dsa::l2_policy_evict_first();
      if (leader) {
        dsa::tma_prefetch_desc(&map_q);
        dsa::tma_prefetch_desc(&map_do);
      }
      auto load_qd = [&](int u) {
        const int uu = n_units - 1 - u;
        const int t = uu / p.G, g = uu - (uu / p.G) * p.G;
        if (leader) {
          dsa::mbar_expect_tx(q_full, (kNqk + kNv) * kChunkBytes);
          for (int c = 0; c < kNqk; ++c)
            dsa::tma_load_3d_hint(qd + c * 2 * kChunkBytes, &map_q, c * 64, g * kHG, t, q_full, policy);
          for (int c = 0; c < kNv; ++c)
            dsa::tma_load_3d_hint(qd + c * 2 * kChunkBytes + kChunkBytes, &map_do, c * 64, g * kHG, t, q_full, policy);
        }
        __syncwarp();
      };
      uint32_t tile_ctr = 0, unit_ctr = 0;
      bool ok = true;
      bool q_pending = false;  // a query + dout load is in flight that no wait has consumed
      int u = next_unit(blockIdx.x);
      if (u < n_units) {
        load_qd(u);
        q_pending = true;
      }
      while (u < n_units && ok) {
        const int nt = unit_tiles(u);
        const int u_next = next_unit(u + gridDim.x);
        if (!dsa::mbar_wait_warp(q_full, unit_ctr & 1, wt)) break;
        q_pending = false;
        for (int i = 0; i < nt; ++i, ++tile_ctr) {
          if (!dsa::mbar_wait_warp(s_empty, (tile_ctr & 1) ^ 1, wt) ||
              !dsa::mbar_wait_warp(kv_full, tile_ctr & 1, wt)) {
            ok = false;
            break;
          }
          dsa::fence_proxy_async_smem();  // cp.async (generic proxy) writes -> tcgen05 reads
          dsa::tc_fence_after();
          const uint32_t d = tmem_base + kSCol;
          for (int c = 0; c < kNqk; ++c) {
            const uint64_t ac = kv_desc + c * (kChunkBytes >> 4), bc = qd_desc + c * (2 * kChunkBytes >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              dsa::umma_bf16_if(leader, d, ac + kk * 2, bc + kk * 2, c < kNv ? idesc_qd : idesc_q, (c | kk) != 0);
          }
          if (leader) dsa::umma_commit(s_full);
          __syncwarp();
        }
        if (!ok) break;
        if (leader) dsa::umma_commit(q_empty);
        __syncwarp();
        if (u_next < n_units) {
          if (!dsa::mbar_wait_warp(q_empty, unit_ctr & 1, wt)) break;
          load_qd(u_next);
          q_pending = true;
        }
        ++unit_ctr;
        u = u_next;
      }
      // leave nothing in flight: the unconsumed query + dout load (only after
      // an abort), then every MMA this warp issued
      if (leader) {
        if (q_pending) dsa::mbar_drain(q_full, unit_ctr & 1, p.status);
        dsa::umma_drain(&drain[0], p.status);
      }
      __syncwarp();
    } else {
      // dq^T[dim, head] += kv^T[dim, key] . dS^T[key, head]: four M = 128
      // blocks over dims 0..511 and one M = 64 block over dims 512..575
      constexpr uint32_t idesc_m128 = dsa::idesc_bf16(128, kHG, 1, 1);
      constexpr uint32_t idesc_m64 = dsa::idesc_bf16(64, kHG, 1, 1);
      const uint64_t v_desc = dsa::smem_desc(kv_addr, kChunkBytes, 1024, dsa::kSwizzle128B);
      const uint64_t ds_desc = dsa::smem_desc(dsa::smem_u32(dsbuf), kChunkBytes, 1024, dsa::kSwizzle128B);
      uint32_t tile_ctr = 0;
      bool ok = true;
      for (int u = next_unit(blockIdx.x); u < n_units && ok; u = next_unit(u + gridDim.x)) {
        const int nt = unit_tiles(u);
        for (int i = 0; i < nt; ++i, ++tile_ctr) {
          if (!dsa::mbar_wait_warp(p_full, tile_ctr & 1, wt)) {
            ok = false;
            break;
          }
          dsa::tc_fence_after();
          for (int mb = 0; mb < 5; ++mb) {
            const uint64_t am = v_desc + mb * (2 * kChunkBytes >> 4);
            const uint32_t d = tmem_base + kQCol + mb * kHG;
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk)
              dsa::umma_bf16_if(leader, d, am + kk * (2048 >> 4), ds_desc + kk * (2048 >> 4),
                                mb < 4 ? idesc_m128 : idesc_m64, (i > 0 || kk > 0) ? 1u : 0u);
          }
          if (leader) {
            dsa::umma_commit(o_done);
            dsa::umma_commit(kv_empty);
          }
          __syncwarp();
        }
      }
      if (leader) dsa::umma_drain(&drain[1], p.status);  // every dq MMA issued has completed
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------ P, dS and dq out
    const int sw = warp - kSoftWarp0;
    const int st = threadIdx.x - kSoftWarp0 * 32;
    const int quarter = warp & 3;
    const int hh = sw >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // 16-lane loads as in the forward: keys kA, kB of the quarter's 16 and
    // heads hbase + 8j + e; register 4j+e is (kA, head), 4j+2+e is (kB, head)
    const int kA = quarter * 16 + (lane >> 2), kB = kA + 8;
    const int hbase = hh * 32 + 2 * (lane & 3);
    uint32_t tile_ctr = 0;
    bool ok = true;
    // a wait of this warp gave up (warp-uniform): the warp skips the rest of
    // the unit's TMEM work, and the eight warps leave together at the unit's
    // last barrier, which carries the flag
    bool failed = false;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int uu = n_units - 1 - u;
      const int t = uu / p.G, g = uu - (uu / p.G) * p.G;
      const int hv = min(kHG, p.H - g * kHG);
      const int len = unit_len(p, t);
      const int nt = (len + kKeys - 1) / kKeys;
      const int64_t hrow = static_cast<int64_t>(t) * p.H + g * kHG;
      if (nt == 0) {
        for (int h = 0; h < hv; ++h)
          for (int dd = st; dd < kDqk; dd += kSoftThreads) p.dq[(hrow + h) * kDqk + dd] = __float2bfloat16_rn(0.f);
        continue;
      }
      named_bar(1, kSoftThreads);  // the previous unit's readers of l2s / dls are done
      if (st < kHG) {
        const float2 sv = st < hv ? __ldg(p.stats + hrow + st) : make_float2(INFINITY, 0.f);
        l2s[st] = sv.x;
        dls[st] = sv.y;
      }
      named_bar(1, kSoftThreads);
      const int32_t* irow = p.idx + static_cast<int64_t>(t) * p.K;
      int nA = kA < len ? __ldcs(irow + kA) : -1;
      int nB = kB < len ? __ldcs(irow + kB) : -1;
      for (int i = 0; i < nt; ++i, ++tile_ctr) {
        const uint32_t ph = tile_ctr & 1;
        const int jA = i * kKeys + kA, jB = i * kKeys + kB;
        const bool vA = jA < len && nA >= 0 && nA < p.Tkv;
        const bool vB = jB < len && nB >= 0 && nB < p.Tkv;
        if (i + 1 < nt) {
          nA = jA + kKeys < len ? __ldcs(irow + jA + kKeys) : -1;
          nB = jB + kKeys < len ? __ldcs(irow + jB + kKeys) : -1;
        }
        if (!dsa::mbar_wait_warp(s_full, ph, wt)) {
          failed = true;
          break;
        }
        dsa::tc_fence_after();
        uint32_t xs[16], dps[16];
        dsa::tmem_ld16x256b_x4(tmem_base + lane_off + kSCol + hh * 32, xs);
        dsa::tmem_ld16x256b_x4(tmem_base + lane_off + kSCol + kHG + hh * 32, dps);
        dsa::tmem_wait_ld();
        dsa::tc_fence_before();
        __syncwarp();
        if (lane == 0) dsa::mbar_arrive(s_empty);
        // P = 2^(s*scale*log2(e) - L2), scale * dS = scale * P * (dP - delta)
        float pv[16], dv[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = hbase + 8 * j + e;
            const float l2 = l2s[h], dl = dls[h];
            const float pa = vA ? ex2(fmaf(__uint_as_float(xs[4 * j + e]), p.scale_log2, -l2)) : 0.f;
            const float pb = vB ? ex2(fmaf(__uint_as_float(xs[4 * j + 2 + e]), p.scale_log2, -l2)) : 0.f;
            pv[4 * j + e] = pa;
            pv[4 * j + 2 + e] = pb;
            dv[4 * j + e] = p.scale * pa * (__uint_as_float(dps[4 * j + e]) - dl);
            dv[4 * j + 2 + e] = p.scale * pb * (__uint_as_float(dps[4 * j + 2 + e]) - dl);
          }
        }
        // dS^T rows kA and kB (heads hbase + 8j + {0, 1} at 16-byte unit
        // hh*4 + j of the row, 128-byte swizzle), as the forward's P^T
        uint8_t* prowA = dsbuf + kA * 128 + 4 * (lane & 3);
        uint8_t* prowB = dsbuf + kB * 128 + 4 * (lane & 3);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int un = hh * 4 + j;
          *reinterpret_cast<uint32_t*>(prowA + ((un ^ (kA & 7)) * 16)) = pack_bf16x2(dv[4 * j], dv[4 * j + 1]);
          *reinterpret_cast<uint32_t*>(prowB + ((un ^ (kB & 7)) * 16)) = pack_bf16x2(dv[4 * j + 2], dv[4 * j + 3]);
        }
        // the same values (bf16) for the dkv launch: [T, K, Hp]
        const int64_t col0 = static_cast<int64_t>(g) * kHG + hbase;
        if (jA < len) {
          const int64_t o = (static_cast<int64_t>(t) * p.K + jA) * p.Hp + col0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<uint32_t*>(p.ds_g + o + 8 * j) = pack_bf16x2(dv[4 * j], dv[4 * j + 1]);
            *reinterpret_cast<uint32_t*>(p.p_g + o + 8 * j) = pack_bf16x2(pv[4 * j], pv[4 * j + 1]);
          }
        }
        if (jB < len) {
          const int64_t o = (static_cast<int64_t>(t) * p.K + jB) * p.Hp + col0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<uint32_t*>(p.ds_g + o + 8 * j) = pack_bf16x2(dv[4 * j + 2], dv[4 * j + 3]);
            *reinterpret_cast<uint32_t*>(p.p_g + o + 8 * j) = pack_bf16x2(pv[4 * j + 2], pv[4 * j + 3]);
          }
        }
        dsa::fence_proxy_async_smem();
        dsa::tc_fence_before();
        __syncwarp();
        if (lane == 0) dsa::mbar_arrive(p_full);
      }
      // ---- dq of the unit: dq^T blocks from TMEM (scale already in dS)
      if (!failed) failed = !dsa::mbar_wait_warp(o_done, (tile_ctr - 1) & 1, wt);
      dsa::tc_fence_after();
      const int hcount = min(32, hv - hh * 32);
      for (int mb = 0; mb < 4 && !failed; ++mb) {
        uint32_t v[32];
        dsa::tmem_ld32(tmem_base + lane_off + kQCol + mb * kHG + hh * 32, v);
        dsa::tmem_wait_ld();
        __nv_bfloat16* o = p.dq + (hrow + hh * 32) * kDqk + mb * 128 + quarter * 32 + lane;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c < hcount) __stcs(o, __float2bfloat16_rn(__uint_as_float(v[c])));
          o += kDqk;
        }
      }
      if (!failed) {
        // dims 512..575: an M = 64 accumulator (dim 512 + r in lane
        // 32*(r/16) + r%16), read like S^T
        uint32_t v[16];
        dsa::tmem_ld16x256b_x4(tmem_base + lane_off + kQCol + 4 * kHG + hh * 32, v);
        dsa::tmem_wait_ld();
        const int dA = 512 + quarter * 16 + (lane >> 2), dB = dA + 8;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = hbase + 8 * j + e;
            if (h < hv) {
              p.dq[(hrow + h) * kDqk + dA] = __float2bfloat16_rn(__uint_as_float(v[4 * j + e]));
              p.dq[(hrow + h) * kDqk + dB] = __float2bfloat16_rn(__uint_as_float(v[4 * j + 2 + e]));
            }
          }
        }
      }
      dsa::tc_fence_before();
      if (dsa::named_bar_any(1, kSoftThreads, failed)) {
        ok = false;
        break;
      }
    }
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    dsa::tc_fence_after();
    dsa::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// -------------------------------------------------------------- 3. dkv
// warp 0 TMA, warp 1 MMA, warps 2..9 drain + shard update: two per TMEM lane
// quarter, one per 64-column half of a block
constexpr int kDkvThreads = 320;
constexpr int kDrainThreads = kDkvThreads - 64;
// staging row stride (floats): 4 floats of padding put the eight keys a warp
// writes at once in different banks (unpadded rows 512 bytes apart collide)
constexpr int kStageLd = 132;

struct DkvLayout {
  uint32_t qd, a, stage, ids, bars, misc, total;
};
__host__ __device__ inline DkvLayout dkv_layout() {
  DkvLayout L;
  uint32_t o = 0;
  L.qd = o;  // as in bwd_dq_kernel: query chunk c, dout chunk c, ... query chunk 8
  o += kNv * 2 * kChunkBytes + kChunkBytes;
  L.a = o;  // two buffers of [scale dS chunk | P chunk] (64 slots x 64 heads each)
  o += 2 * 2 * kChunkBytes;
  L.stage = o;  // 64 keys x 128 dims fp32, rows padded to kStageLd
  o += kKeys * kStageLd * 4;
  L.ids = o;  // ids of the tile, first slot of each id in the tile
  o += 2 * kKeys * 4;
  L.bars = o;
  o += 16 * 8;
  L.misc = o;
  o += 16;
  L.total = o;
  return L;
}

struct DkvParams {
  const int32_t* idx;
  const int32_t* topk_length;
  float* shards;  // [kLanes][Tkv][kDqk]; the atomic variant: dkv [Tkv][kDqk]
  uint32_t* status;
  int T, Tkv, H, G, K, Hp;
};

__device__ __forceinline__ int dkv_len(const DkvParams& p, int t) {
  int L = p.K;
  if (p.topk_length) {
    L = __ldg(p.topk_length + t);
    L = L < 0 ? 0 : (L > p.K ? p.K : L);
  }
  return L;
}

// Lane blockIdx.x (of kLanes) takes units (t, g) with t = lane, lane + kLanes,
// ...; per 64-slot tile and per block of 128 dims (64 for dims 512..575)
// D[key, dim] = sum_h scale dS[key, h] q[h, dim] + sum_h P[key, h] dout[h, dim]
// (M = 64 keys, K = 64 + 64 heads, B MN-major), added into the lane's shard
// (ATOMIC: into dkv, one fp32 vector atomic per 4 dims of each valid slot).
template <bool ATOMIC>
__global__ void __launch_bounds__(kDkvThreads, 1)
    bwd_dkv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                   const __grid_constant__ CUtensorMap map_ds, const __grid_constant__ CUtensorMap map_p,
                   const DkvParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dsa::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const DkvLayout L = dkv_layout();
  uint8_t* qd = smem + L.qd;
  uint8_t* abuf = smem + L.a;
  float* stage = reinterpret_cast<float*>(smem + L.stage);
  int32_t* tids = reinterpret_cast<int32_t*>(smem + L.ids);
  int32_t* first = tids + kKeys;
  volatile int* dupflag = reinterpret_cast<volatile int*>(smem + L.misc + 8);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* qd_full = bars;
  uint64_t* qd_empty = bars + 1;
  uint64_t* a_full = bars + 2;   // [2]
  uint64_t* a_empty = bars + 4;  // [2]
  uint64_t* d_full = bars + 6;   // [2]
  uint64_t* d_empty = bars + 8;  // [2]
  uint64_t* drain = bars + 10;   // the MMA issuer's exit commit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lane_id = blockIdx.x;
  const int n_units = p.T * p.G;

  if (threadIdx.x == 0) {
    dsa::mbar_init(qd_full, 1);
    dsa::mbar_init(qd_empty, 1);
    for (int b = 0; b < 2; ++b) {
      dsa::mbar_init(&a_full[b], 1);
      dsa::mbar_init(&a_empty[b], 1);
      dsa::mbar_init(&d_full[b], 1);
      dsa::mbar_init(&d_empty[b], 8);  // one arrive per drain warp
    }
    dsa::mbar_init(drain, 1);
    *abort_flag = 0;
    dsa::fence_barrier_init();
  }
  if (warp == 1) dsa::tmem_alloc(tmem_slot, 256);
  dsa::tc_fence_before();
  __syncthreads();
  dsa::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const dsa::Waiter wt = dsa::make_waiter(abort_flag, p.status);
  // units of this lane, in order: u = lane_id + kLanes * k over (t, g), t-major
  auto unit_tiles = [&](int u) { return (dkv_len(p, u / p.G) + kKeys - 1) / kKeys; };

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t policy = dsa::l2_policy_evict_first();
      dsa::tma_prefetch_desc(&map_q);
      dsa::tma_prefetch_desc(&map_do);
      dsa::tma_prefetch_desc(&map_ds);
      dsa::tma_prefetch_desc(&map_p);
      uint32_t tile_ctr = 0, unit_ctr = 0;
      uint32_t qd_issued = 0;  // query + dout loads issued: load m completes phase m of qd_full
      for (int u = lane_id; u < n_units; u += kLanes) {
        const int nt = unit_tiles(u);
        if (nt == 0) continue;
        const int t = u / p.G, g = u - (u / p.G) * p.G;
        if (!dsa::mbar_wait(qd_empty, (unit_ctr & 1) ^ 1, wt)) break;
        ++qd_issued;
        dsa::mbar_expect_tx(qd_full, (kNqk + kNv) * kChunkBytes);
        for (int c = 0; c < kNqk; ++c)
          dsa::tma_load_3d_hint(qd + c * 2 * kChunkBytes, &map_q, c * 64, g * kHG, t, qd_full, policy);
        for (int c = 0; c < kNv; ++c)
          dsa::tma_load_3d_hint(qd + c * 2 * kChunkBytes + kChunkBytes, &map_do, c * 64, g * kHG, t, qd_full, policy);
        bool ok = true;
        for (int i = 0; i < nt; ++i, ++tile_ctr) {
          const int b = tile_ctr & 1;
          if (!dsa::mbar_wait(&a_empty[b], ((tile_ctr >> 1) & 1) ^ 1, wt)) { ok = false; break; }
          dsa::mbar_expect_tx(&a_full[b], 2 * kChunkBytes);
          const int row = t * p.K + i * kKeys;
          uint8_t* dst = abuf + b * 2 * kChunkBytes;
          dsa::tma_load_2d_hint(dst, &map_ds, g * kHG, row, &a_full[b], policy);
          dsa::tma_load_2d_hint(dst + kChunkBytes, &map_p, g * kHG, row, &a_full[b], policy);
        }
        if (!ok) break;
        ++unit_ctr;
      }
      // every copy issued has landed before the CTA leaves (all were consumed
      // unless the kernel aborted): the newest query + dout load and the newest
      // load of each of the two [scale dS | P] buffers (tile i went to buffer
      // i & 1, phase (i >> 1) & 1; a buffer is reloaded only once consumed)
      if (qd_issued > 0) dsa::mbar_drain(qd_full, (qd_issued - 1) & 1, p.status);
      for (uint32_t j = 1; j <= tile_ctr && j <= 2; ++j) {
        const uint32_t i = tile_ctr - j;
        dsa::mbar_drain(&a_full[i & 1], (i >> 1) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    const bool leader = elect_sync();
    constexpr uint32_t idesc_n128 = dsa::idesc_bf16(kKeys, 128, 0, 1);
    constexpr uint32_t idesc_n64 = dsa::idesc_bf16(kKeys, 64, 0, 1);
    const uint32_t qd_addr = dsa::smem_u32(qd), a_addr = dsa::smem_u32(abuf);
    uint32_t tile_ctr = 0, unit_ctr = 0, blk_ctr = 0;
    bool ok = true;
    for (int u = lane_id; u < n_units && ok; u += kLanes) {
      const int nt = unit_tiles(u);
      if (nt == 0) continue;
      if (!dsa::mbar_wait_warp(qd_full, unit_ctr & 1, wt)) break;
      for (int i = 0; i < nt; ++i, ++tile_ctr) {
        const int b = tile_ctr & 1;
        if (!dsa::mbar_wait_warp(&a_full[b], (tile_ctr >> 1) & 1, wt)) { ok = false; break; }
        dsa::tc_fence_after();
        const uint32_t a0 = a_addr + b * 2 * kChunkBytes;
        for (int nb = 0; nb < 5 && ok; ++nb, ++blk_ctr) {
          const int db = blk_ctr & 1;
          if (!dsa::mbar_wait_warp(&d_empty[db], ((blk_ctr >> 1) & 1) ^ 1, wt)) {
            ok = false;
            break;
          }
          dsa::tc_fence_after();
          const uint32_t d = tmem_base + db * 128;
          const uint32_t bq = qd_addr + nb * 2 * (2 * kChunkBytes);  // query chunk 2nb
          const int ksteps = nb < 4 ? 8 : 4;  // dims 512..575 have no value part
#pragma unroll 1
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint32_t as = a0 + (kk < 4 ? 0u : kChunkBytes) + (kk & 3) * 32;
            const uint32_t bs = bq + (kk < 4 ? 0u : kChunkBytes) + (kk & 3) * 2048;
            const uint64_t ad = dsa::smem_desc(as, 16, 1024, dsa::kSwizzle128B);
            const uint64_t bd = dsa::smem_desc(bs, 2 * kChunkBytes, 1024, dsa::kSwizzle128B);
            dsa::umma_bf16_if(leader, d, ad, bd, nb < 4 ? idesc_n128 : idesc_n64, kk > 0 ? 1u : 0u);
          }
          if (leader) dsa::umma_commit(&d_full[db]);
          __syncwarp();
        }
        if (!ok) break;
        if (leader) dsa::umma_commit(&a_empty[b]);
        __syncwarp();
      }
      if (!ok) break;
      if (leader) dsa::umma_commit(qd_empty);
      __syncwarp();
      ++unit_ctr;
    }
    if (leader) dsa::umma_drain(drain, p.status);  // every MMA issued has completed
    __syncwarp();
  } else {
    // ------------------------------------------- drain + shard update
    const int dt = threadIdx.x - 64;       // 0..255
    const int quarter = warp & 3;          // TMEM lane quarter (warps 2..5)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int kA = quarter * 16 + (lane >> 2), kB = kA + 8;
    float* shard = ATOMIC ? p.shards : p.shards + static_cast<int64_t>(lane_id) * p.Tkv * kDqk;  // ATOMIC: dkv
    uint32_t blk_ctr = 0;
    bool ok = true;
    // a wait of this warp gave up (warp-uniform): it skips its TMEM reads and
    // shard writes, and the four warps leave together at the block's last
    // barrier, which carries the flag
    bool failed = false;
    if constexpr (ATOMIC) {
      // Each warp drains one 64-column half of its own TMEM lane quarter (keys
      // 16*quarter .. +15 of the tile) through its own part of the staging
      // tile and adds it into dkv, two rows (256 contiguous bytes each) per
      // warp instruction: no barrier across the eight warps per block, and
      // each tile's ids are read once.
      const int r0 = quarter * 16;
      const int half = (warp - 2) >> 2;
      const int c0 = 64 * half;  // this warp's columns of a block: [c0, c0 + 64)
      for (int u = lane_id; u < n_units && ok; u += kLanes) {
        const int len = dkv_len(p, u / p.G);
        const int nt = (len + kKeys - 1) / kKeys;
        const int t = u / p.G;
        for (int i = 0; i < nt && ok; ++i) {
          int my = -1;  // lane k < 16: id of key r0 + k of the tile (-1: absent)
          if (lane < 16) {
            const int j = i * kKeys + r0 + lane;
            const int id = j < len ? __ldg(p.idx + static_cast<int64_t>(t) * p.K + j) : -1;
            my = (id >= 0 && id < p.Tkv) ? id : -1;
          }
          int ids[8];  // id of row 2k + lane / 16 of the warp's 16
#pragma unroll
          for (int k = 0; k < 8; ++k) ids[k] = __shfl_sync(0xffffffffu, my, 2 * k + (lane >> 4));
          for (int nb = 0; nb < 5; ++nb, ++blk_ctr) {
            const int db = blk_ctr & 1;
            const bool active = c0 < (nb < 4 ? 128 : 64);
            if (!failed) failed = !dsa::mbar_wait_warp(&d_full[db], (blk_ctr >> 1) & 1, wt);
            dsa::tc_fence_after();
            if (!failed && active) {
              uint32_t v[2][16];
#pragma unroll
              for (int q2 = 0; q2 < 2; ++q2)
                dsa::tmem_ld16x256b_x4(tmem_base + lane_off + db * 128 + c0 + 32 * q2, v[q2]);
              dsa::tmem_wait_ld();
#pragma unroll
              for (int q2 = 0; q2 < 2; ++q2) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const int col = c0 + 32 * q2 + 8 * j + 2 * (lane & 3);
                  *reinterpret_cast<float2*>(stage + kA * kStageLd + col) =
                      make_float2(__uint_as_float(v[q2][4 * j]), __uint_as_float(v[q2][4 * j + 1]));
                  *reinterpret_cast<float2*>(stage + kB * kStageLd + col) =
                      make_float2(__uint_as_float(v[q2][4 * j + 2]), __uint_as_float(v[q2][4 * j + 3]));
                }
              }
            }
            dsa::tc_fence_before();
            __syncwarp();
            if (lane == 0) dsa::mbar_arrive(&d_empty[db]);  // this warp's TMEM reads are done
            if (!failed && active) {
              const int cl = c0 + 4 * (lane & 15);
              float* base = shard + nb * 128 + cl;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                if (ids[k] < 0) continue;
                const int r = r0 + 2 * k + (lane >> 4);
                const float4 sv = *reinterpret_cast<const float4*>(stage + r * kStageLd + cl);
                atomicAdd(reinterpret_cast<float4*>(base + static_cast<int64_t>(ids[k]) * kDqk), sv);
              }
            }
            __syncwarp();  // this warp's staging columns are read before the next block rewrites them
          }
          // the eight warps leave together, at a tile's end, if any wait gave up
          if (dsa::named_bar_any(1, kDrainThreads, failed)) {
            ok = false;
            break;
          }
        }
      }
    } else {
      for (int u = lane_id; u < n_units && ok; u += kLanes) {
        const int len = dkv_len(p, u / p.G);
        const int nt = (len + kKeys - 1) / kKeys;
        const int t = u / p.G;
        for (int i = 0; i < nt && ok; ++i) {
          // ids of the tile (-1: absent) and, per slot, the first slot of the
          // tile with the same id
          named_bar(1, kDrainThreads);  // previous tile's readers of tids / first / stage are done
          if (dt < kKeys) {
            const int j = i * kKeys + dt;
            int id = j < len ? __ldg(p.idx + static_cast<int64_t>(t) * p.K + j) : -1;
            tids[dt] = (id >= 0 && id < p.Tkv) ? id : -1;
          }
          if (dt == 0) *dupflag = 0;
          named_bar(1, kDrainThreads);
          if (dt < kKeys) {
            const int id = tids[dt];
            int f = dt;
            if (id >= 0)
              for (int r = 0; r < dt; ++r)
                if (tids[r] == id) {
                  f = r;
                  break;
                }
            first[dt] = f;
            if (f != dt) *dupflag = 1;
          }
          named_bar(1, kDrainThreads);  // first[] of the tile complete
          if (!*dupflag) {
            // No id repeats in this tile (the usual case): each warp updates
            // the rows of its own TMEM lane quarter (keys 16*quarter .. +15),
            // one 512-byte row per warp instruction, with no barrier across
            // the drain warps per block.  Each row has one writer per block,
            // which adds the same fp32 value to it as the path below, so the
            // result is the same bits; the barrier at the tile's end orders
            // these writes before a later tile's reads of the same rows.
            const int r0 = quarter * 16;
            const int c0 = 64 * ((warp - 2) >> 2);  // this warp's columns of a block: [c0, c0 + 64)
            const int cl = c0 + 4 * (lane & 15);
            const int* ids = tids + r0 + (lane >> 4);  // row 2k + lane / 16 of the warp's 16: ids[2k]
            float4 pa[8], pn[8];
            auto load_rows = [&](int nb, float4 (&a)[8]) {
              const bool on = c0 < (nb < 4 ? 128 : 64);
              const float4* src = reinterpret_cast<const float4*>(shard + nb * 128 + cl);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int id = ids[2 * k];
                a[k] = (on && id >= 0) ? src[static_cast<int64_t>(id) * (kDqk / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
              }
            };
            load_rows(0, pa);
            for (int nb = 0; nb < 5; ++nb, ++blk_ctr) {
              const int db = blk_ctr & 1;
              const bool active = c0 < (nb < 4 ? 128 : 64);
              if (nb + 1 < 5) load_rows(nb + 1, pn);
              if (!failed) failed = !dsa::mbar_wait_warp(&d_full[db], (blk_ctr >> 1) & 1, wt);
              dsa::tc_fence_after();
              if (!failed && active) {
                uint32_t v[2][16];
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2)
                  dsa::tmem_ld16x256b_x4(tmem_base + lane_off + db * 128 + c0 + 32 * q2, v[q2]);
                dsa::tmem_wait_ld();
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    const int col = c0 + 32 * q2 + 8 * j + 2 * (lane & 3);
                    *reinterpret_cast<float2*>(stage + kA * kStageLd + col) =
                        make_float2(__uint_as_float(v[q2][4 * j]), __uint_as_float(v[q2][4 * j + 1]));
                    *reinterpret_cast<float2*>(stage + kB * kStageLd + col) =
                        make_float2(__uint_as_float(v[q2][4 * j + 2]), __uint_as_float(v[q2][4 * j + 3]));
                  }
                }
              }
              dsa::tc_fence_before();
              __syncwarp();
              if (lane == 0) dsa::mbar_arrive(&d_empty[db]);  // this warp's TMEM reads are done
              if (!failed && active) {
                float4* base = reinterpret_cast<float4*>(shard + nb * 128 + cl);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const int id = ids[2 * k];
                  if (id < 0) continue;
                  const int r = r0 + 2 * k + (lane >> 4);
                  const float4 sv = *reinterpret_cast<const float4*>(stage + r * kStageLd + cl);
                  base[static_cast<int64_t>(id) * (kDqk / 4)] =
                      make_float4(pa[k].x + sv.x, pa[k].y + sv.y, pa[k].z + sv.z, pa[k].w + sv.w);
                }
              }
              __syncwarp();  // this warp's staging columns are read before the next block rewrites them
#pragma unroll
              for (int k = 0; k < 8; ++k) pa[k] = pn[k];
            }
            // the eight warps leave together, at the tile's end, if any wait gave up
            if (dsa::named_bar_any(1, kDrainThreads, failed)) {
              ok = false;
              break;
            }
            continue;
          }
          // A tile with repeated ids.  The shard values this thread updates:
          // thread (key group kg, 4-dim column c4) owns rows kg + 4k of each
          // block of dims; a repeated id is updated once, through its first
          // slot, so no two threads write one value.  Earlier updates of the
          // same values, by any thread, were ordered before the reads by the
          // barrier that ended the previous tile (or block).  The first four
          // drain warps (one per TMEM lane quarter) do the work; the other
          // four only take part in the barriers.
          const bool worker = dt < 128;
          const int kg = dt >> 5, c4 = dt & 31;
          for (int nb = 0; nb < 5; ++nb, ++blk_ctr) {
            const int db = blk_ctr & 1;
            const int nd = nb < 4 ? 128 : 64;
            const bool col_on = 4 * c4 < nd;
            float4* base = reinterpret_cast<float4*>(shard + nb * 128 + 4 * c4);
            if (!failed) failed = !dsa::mbar_wait_warp(&d_full[db], (blk_ctr >> 1) & 1, wt);
            dsa::tc_fence_after();
            if (!failed && worker) {
              for (int h2 = 0; h2 < 2; ++h2) {  // two 64-column halves
                if (64 * h2 >= nd) break;
                uint32_t v[2][16];
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2)
                  dsa::tmem_ld16x256b_x4(tmem_base + lane_off + db * 128 + 64 * h2 + 32 * q2, v[q2]);
                dsa::tmem_wait_ld();
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    const int col = 64 * h2 + 32 * q2 + 8 * j + 2 * (lane & 3);
                    *reinterpret_cast<float2*>(stage + kA * kStageLd + col) =
                        make_float2(__uint_as_float(v[q2][4 * j]), __uint_as_float(v[q2][4 * j + 1]));
                    *reinterpret_cast<float2*>(stage + kB * kStageLd + col) =
                        make_float2(__uint_as_float(v[q2][4 * j + 2]), __uint_as_float(v[q2][4 * j + 3]));
                  }
                }
              }
            }
            dsa::tc_fence_before();
            named_bar(1, kDrainThreads);  // stage and first[] complete
            if (lane == 0) dsa::mbar_arrive(&d_empty[db]);
            if (*dupflag) {
              // repeated ids: later slots fold into the first one, in slot order
              if (dt < nd)
                for (int r = 1; r < kKeys; ++r)
                  if (first[r] != r) stage[first[r] * kStageLd + dt] += stage[r * kStageLd + dt];
              named_bar(1, kDrainThreads);
            }
            if (col_on && !failed && worker) {
#pragma unroll
              for (int k = 0; k < kKeys / 4; ++k) {
                const int r = kg + 4 * k;
                const int id = tids[r];
                if (id >= 0 && first[r] == r) {
                  const float4 s = *reinterpret_cast<const float4*>(stage + r * kStageLd + 4 * c4);
                  const float4 a = base[static_cast<int64_t>(id) * (kDqk / 4)];
                  base[static_cast<int64_t>(id) * (kDqk / 4)] = make_float4(a.x + s.x, a.y + s.y, a.z + s.z, a.w + s.w);
                }
              }
            }
            // stage is read before the next block overwrites it; the group
            // leaves together if any warp's wait gave up
            if (dsa::named_bar_any(1, kDrainThreads, failed)) {
              ok = false;
              break;
            }
          }
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    dsa::tc_fence_after();
    dsa::tmem_dealloc(tmem_base, 256);
  }
}

// ---------------------------------------------------------- 4. reductions
// dkv[i] = sum over lanes c = 0..kLanes-1 of shard c, in lane order.
__global__ void bwd_reduce_dkv_kernel(const float4* __restrict__ shards, int64_t n4, float4* __restrict__ dkv) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  float4 s = __ldcs(shards + i);
  for (int c = 1; c < kLanes; ++c) {
    const float4 v = __ldcs(shards + c * n4 + i);
    s.x += v.x;
    s.y += v.y;
    s.z += v.z;
    s.w += v.w;
  }
  dkv[i] = s;
}

// d_sink[h] = sum over rows of dsink_part[t, h]: one block per head, fixed
// strided partial sums then a fixed tree.
__global__ void bwd_reduce_sink_kernel(const float* __restrict__ part, int T, int H, float* __restrict__ dsink) {
  __shared__ float red[256];
  const int h = blockIdx.x;
  float s = 0.f;
  for (int t = threadIdx.x; t < T; t += 256) s += part[static_cast<int64_t>(t) * H + h];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) dsink[h] = red[0];
}

}  // namespace

namespace {

struct BwdWorkspace {
  float2* stats;
  float* dsink_part;
  __nv_bfloat16* ds_g;
  __nv_bfloat16* p_g;
  float* shards;
  size_t total;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

BwdWorkspace bwd_workspace(void* base, int T, int Tkv, int H, int K, bool deterministic) {
  BwdWorkspace w{};
  const size_t th = static_cast<size_t>(T) * H;
  const size_t hp = static_cast<size_t>((H + kHG - 1) / kHG) * kHG;
  const size_t tkh = static_cast<size_t>(T) * K * hp;
  uint8_t* b = static_cast<uint8_t*>(base);
  size_t o = 0;
  w.stats = reinterpret_cast<float2*>(b + o);
  o += align256(th * sizeof(float2));
  w.dsink_part = reinterpret_cast<float*>(b + o);
  o += align256(th * sizeof(float));
  w.ds_g = reinterpret_cast<__nv_bfloat16*>(b + o);
  o += align256(tkh * 2);
  w.p_g = reinterpret_cast<__nv_bfloat16*>(b + o);
  o += align256(tkh * 2);
  w.shards = deterministic ? reinterpret_cast<float*>(b + o) : nullptr;
  if (deterministic) o += align256(static_cast<size_t>(kLanes) * Tkv * kDqk * sizeof(float));
  w.total = o;
  return w;
}

}  // namespace

extern "C" size_t dsa_sparse_attn_bwd_workspace_size_ex(int T, int Tkv, int H, int K, int deterministic) {
  if (T < 0 || Tkv < 1 || H < 1 || H > 128 || K < 1) return 0;
  return bwd_workspace(nullptr, T, Tkv, H, K, deterministic != 0).total;
}

extern "C" size_t dsa_sparse_attn_bwd_workspace_size(int T, int Tkv, int H, int K) {
  return dsa_sparse_attn_bwd_workspace_size_ex(T, Tkv, H, K, 1);
}

namespace {

int run_bwd(const void* q, const void* kv, const void* out, const void* dout, const float* lse_kv, const float* sink,
            const int32_t* idx, const int32_t* topk_length, int T, int Tkv, int H, int Dqk, int Dv, int K, float scale,
            void* dq, float* dkv, float* d_sink, bool deterministic, void* workspace, size_t ws_bytes,
            cudaStream_t stream) {
  if (Dqk != kDqk || Dv != kDv)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_sparse_attn_bwd: (Dqk, Dv) must be (576, 512): the latent K = V layout");
  if (T < 0 || Tkv < 1 || H < 1 || H > 128 || K < 1)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_sparse_attn_bwd: need T >= 0, Tkv >= 1, 1 <= H <= 128, K >= 1");
  if (!(scale > 0.f) || !(scale < INFINITY))
    return dsa::set_error(DSA_ERR_VALUE, "dsa_sparse_attn_bwd: scale must be finite and > 0");
  if (!dkv || (T > 0 && (!q || !kv || !out || !dout || !lse_kv || !idx || !dq)))
    return dsa::set_error(DSA_ERR_VALUE, "dsa_sparse_attn_bwd: NULL pointer");
  if (!dsa::aligned(q, 16) || !dsa::aligned(kv, 16) || !dsa::aligned(out, 16) || !dsa::aligned(dout, 16) ||
      !dsa::aligned(dkv, 16))
    return dsa::set_error(DSA_ERR_VALUE, "dsa_sparse_attn_bwd: q, kv, out, dout and dkv must be 16-byte aligned");
  const size_t need = dsa_sparse_attn_bwd_workspace_size_ex(T, Tkv, H, K, deterministic ? 1 : 0);
  if (!workspace || ws_bytes < need || !dsa::aligned(workspace, 256))
    return dsa::set_error(DSA_ERR_WORKSPACE, "dsa_sparse_attn_bwd: workspace must be 256-byte aligned and >= %zu bytes",
                          need);
  int sms = 0;
  int rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  const size_t dkv_bytes = static_cast<size_t>(Tkv) * kDqk * sizeof(float);
  if (T == 0) {
    if (cudaMemsetAsync(dkv, 0, dkv_bytes, stream) != cudaSuccess ||
        (d_sink && cudaMemsetAsync(d_sink, 0, H * sizeof(float), stream) != cudaSuccess))
      return dsa::launch_error("dsa_sparse_attn_bwd: memset");
    return DSA_OK;
  }
  const BwdWorkspace w = bwd_workspace(workspace, T, Tkv, H, K, deterministic);
  const int G = (H + kHG - 1) / kHG;
  const int Hp = G * kHG;
  uint32_t* status = dsa::device_status_ptr();

  // 1. per (token, head) statistics
  const int64_t rows = static_cast<int64_t>(T) * H;
  bwd_prep_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse_kv, sink, rows, H, w.stats,
      w.dsink_part);
  if ((rc = dsa::launch_error("bwd_prep_kernel")) != DSA_OK) return rc;

  CUtensorMap mq, mdo;
  rc = dsa::encode_tensor_map_3d(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kDqk, H, T, static_cast<uint64_t>(kDqk) * 2,
                                 static_cast<uint64_t>(kDqk) * H * 2, 64, kHG, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != DSA_OK) return rc;
  rc = dsa::encode_tensor_map_3d(&mdo, dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kDv, H, T, static_cast<uint64_t>(kDv) * 2,
                                 static_cast<uint64_t>(kDv) * H * 2, 64, kHG, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != DSA_OK) return rc;

  // 2. dq, and P / scale * dS for the dkv pass
  BwdParams p{};
  p.idx = idx;
  p.topk_length = topk_length;
  p.kv = static_cast<const uint8_t*>(kv);
  p.stats = w.stats;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.ds_g = w.ds_g;
  p.p_g = w.p_g;
  p.status = status;
  p.T = T;
  p.Tkv = Tkv;
  p.H = H;
  p.G = G;
  p.K = K;
  p.Hp = Hp;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  const size_t smem_dq = dq_layout().total + 1024;
  if (cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_dq)) !=
      cudaSuccess)
    return dsa::launch_error("bwd_dq_kernel smem attribute");
  const int units = T * G;
  bwd_dq_kernel<<<units < sms ? units : sms, kThreads, smem_dq, stream>>>(mq, mdo, p);
  if ((rc = dsa::launch_error("bwd_dq_kernel")) != DSA_OK) return rc;

  // 3. dkv into the lanes' shards (the atomic variant: into dkv itself)
  const size_t shard_bytes = deterministic ? static_cast<size_t>(kLanes) * Tkv * kDqk * sizeof(float) : dkv_bytes;
  if (cudaMemsetAsync(deterministic ? static_cast<void*>(w.shards) : static_cast<void*>(dkv), 0, shard_bytes,
                      stream) != cudaSuccess)
    return dsa::launch_error("dsa_sparse_attn_bwd: shard memset");
  CUtensorMap mds, mp;
  const uint64_t tk = static_cast<uint64_t>(T) * K;
  rc = dsa::encode_tensor_map_2d(&mds, w.ds_g, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Hp, tk, static_cast<uint64_t>(Hp) * 2,
                                 64, kKeys, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != DSA_OK) return rc;
  rc = dsa::encode_tensor_map_2d(&mp, w.p_g, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Hp, tk, static_cast<uint64_t>(Hp) * 2,
                                 64, kKeys, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != DSA_OK) return rc;
  DkvParams dp{};
  dp.idx = idx;
  dp.topk_length = topk_length;
  dp.shards = deterministic ? w.shards : dkv;
  dp.status = status;
  dp.T = T;
  dp.Tkv = Tkv;
  dp.H = H;
  dp.G = G;
  dp.K = K;
  dp.Hp = Hp;
  const size_t smem_dkv = dkv_layout().total + 1024;
  auto dkv_kernel = deterministic ? bwd_dkv_kernel<false> : bwd_dkv_kernel<true>;
  if (cudaFuncSetAttribute(dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_dkv)) !=
      cudaSuccess)
    return dsa::launch_error("bwd_dkv_kernel smem attribute");
  dkv_kernel<<<kLanes, kDkvThreads, smem_dkv, stream>>>(mq, mdo, mds, mp, dp);
  if ((rc = dsa::launch_error("bwd_dkv_kernel")) != DSA_OK) return rc;

  // 4. fixed-order reductions (the atomic variant has no shards to reduce)
  if (deterministic) {
    const int64_t n4 = static_cast<int64_t>(Tkv) * kDqk / 4;
    bwd_reduce_dkv_kernel<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, stream>>>(
        reinterpret_cast<const float4*>(w.shards), n4, reinterpret_cast<float4*>(dkv));
    if ((rc = dsa::launch_error("bwd_reduce_dkv_kernel")) != DSA_OK) return rc;
  }
  if (d_sink) {
    bwd_reduce_sink_kernel<<<H, 256, 0, stream>>>(w.dsink_part, T, H, d_sink);
    if ((rc = dsa::launch_error("bwd_reduce_sink_kernel")) != DSA_OK) return rc;
  }
  return DSA_OK;
}

}  // namespace

extern "C" int dsa_sparse_attn_bwd(const void* q, const void* kv, const void* out, const void* dout,
                                   const float* lse_kv, const float* sink, const int32_t* idx,
                                   const int32_t* topk_length, int T, int Tkv, int H, int Dqk, int Dv, int K,
                                   float scale, void* dq, float* dkv, float* d_sink, void* workspace,
                                   size_t ws_bytes, cudaStream_t stream) {
  dsa::clear_error();
  return run_bwd(q, kv, out, dout, lse_kv, sink, idx, topk_length, T, Tkv, H, Dqk, Dv, K, scale, dq, dkv, d_sink, true,
                 workspace, ws_bytes, stream);
}

extern "C" int dsa_sparse_attn_bwd_ex(const void* q, const void* kv, const void* out, const void* dout,
                                      const float* lse_kv, const float* sink, const int32_t* idx,
                                      const int32_t* topk_length, int T, int Tkv, int H, int Dqk, int Dv, int K,
                                      float scale, void* dq, float* dkv, float* d_sink, int deterministic,
                                      void* workspace, size_t ws_bytes, cudaStream_t stream) {
  dsa::clear_error();
  return run_bwd(q, kv, out, dout, lse_kv, sink, idx, topk_length, T, Tkv, H, Dqk, Dv, K, scale, dq, dkv, d_sink,
                 deterministic != 0, workspace, ws_bytes, stream);
}
