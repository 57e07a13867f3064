// attention.cu -- sparse MQA attention forward on tcgen05.
//
// cuDNN Frontend DSA page, section 1 (Sparse Attention Forward): for query
// row t, head h and valid top-k slot j, s_j = scale * q[t,h,:] . kv[idx_j, :];
// invalid or out-of-range ids are absent; duplicates are separate slots; the
// sink enters only the denominator.  Shapes follow NeMo glm_moe_dsa
// cudnn_sparse_attention (q [T,H,576], latent kv [T,1,576], V = first 512
// dims) and, with a separate 256-dim V, NeMo qwen3_8_flash_next
// cudnn_sparse_gqa_attention.
//
// Work unit = (token t, group g of 64 heads).  The selected KV rows are
// gathered once per unit, in tiles of 64 keys, and shared by all 64 heads
// (MQA).  At 64 heads the step needs ~120 FLOP per gathered byte, so the
// kernel is organised around keeping the gather streaming: two 64-key tile
// buffers alternate (a 128-key tile would not fit twice next to the resident
// query), and eight warps gather with cp.async, each warp instruction moving
// four 128-byte row segments into their 128-byte-swizzled slots (rows of
// invalid slots are zero-filled without reading memory).
//
// Products ("swap AB", the 64 heads are the N side of both):
//   MMA1  S^T[key, head]  = KV[key, 0:Dqk] . Q[head, 0:Dqk]^T  (M=64 keys, N=64)
//   MMA2  O^T[dim, head] += V^T[dim, key] . P^T[key, head]     (M=128 value
//         dims per instruction group, N=64, K=16 keys per instruction)
// S^T (two buffers) and O^T live in TMEM.  An M=64 accumulator occupies
// lanes 0..15 of each 32-lane quarter (row r in lane 32*(r/16) + r%16).
// MMA1 and MMA2 are issued by two different warps, each as soon as its
// inputs are ready, so MMA1 of tile i+1 (two S buffers) can run while
// softmax(i) does and MMA2(i) never queues behind a whole MMA1.
//
// Softmax: 8 warps, two per TMEM lane quarter; lanes 0..15 of a warp own one
// key each and 32 heads (the warp's head half).  Per head a reference maximum
// is kept (online softmax); the running sums and O^T are rescaled only when
// a tile's maximum exceeds the reference by more than 2^8, which leaves the
// result exact because numerator and denominator use the same reference.
// p = 2^(x - m) with x = s*scale*log2(e); P^T goes to shared memory as bf16.
// The epilogue reduces the per-thread sums, adds the sink to the
// denominator and writes out (bf16), lse (sink included) and optionally
// lse_kv and max_logits.
//
// Warps: 0..7 gather, 8..15 softmax and epilogue, 16 = TMEM allocation,
// MMA1 issue and query loads (TMA), 17 = MMA2 issue, 18..19 idle (they fill
// the fifth warpgroup, whose registers go to the softmax).  Persistent CTAs
// take units from the longest rows down.
#include <climits>

#include "common.cuh"

namespace {

constexpr int kKeys = 64;                       // keys per tile
constexpr int kHG = 64;                         // heads per group
// cp.async gather bandwidth grows with the warps issuing it (measured on
// GB300, random 1152-byte rows into 64-key tiles: 4 warps 30 B/clk/SM,
// 6 warps 36, 8 warps 49), so the gather gets eight warps (two keys each per
// tile); five warpgroups in all, with registers moved from the gather and
// MMA warpgroups to the softmax ones.
constexpr int kGatherWarps = 8;
constexpr int kGatherThreads = kGatherWarps * 32;
constexpr int kGatherKeys = kGatherThreads / 8;                   // keys one gather step covers
constexpr int kGatherSteps = (kKeys + kGatherKeys - 1) / kGatherKeys;  // steps per tile
constexpr int kSoftWarp0 = kGatherWarps;            // warpgroups 2 and 3
constexpr int kSoftWarps = 8;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kMmaWarp = kSoftWarp0 + kSoftWarps;   // MMA1 and query loads (warpgroup 4)
constexpr int kMma2Warp = kMmaWarp + 1;             // MMA2
constexpr int kThreads = (kMmaWarp + 4) * 32;       // 640: five warpgroups (the last two warps idle)
// Register split: launched at kLaunchRegs per thread; the softmax warpgroups
// raise theirs to kSoftRegs, the others lower theirs to kLeanRegs
// (3 x 128 x kLeanRegs + 2 x 128 x kSoftRegs <= 640 x kLaunchRegs).
constexpr int kLaunchRegs = 96, kLeanRegs = 56, kSoftRegs = 152;
static_assert(3 * 128 * kLeanRegs + 2 * 128 * kSoftRegs <= kThreads * kLaunchRegs, "register split exceeds the launch");
constexpr uint32_t kChunkBytes = kKeys * 128;   // 64 keys x 64 bf16
constexpr uint32_t kQChunkBytes = kHG * 128;    // 64 heads x 64 bf16
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kTheta = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr int kSCol = 0;     // S^T buffers at columns 0 and 64
constexpr int kOCol = 128;   // O^T blocks at 128 + 64*m

struct AttnParams {
  const int32_t* idx;
  const int32_t* topk_length;
  const float* sink;
  const uint8_t* kv;   // latent (or K) rows of kv_row_bytes
  const uint8_t* v;    // separate V rows of v_row_bytes, or nullptr
  __nv_bfloat16* out;
  float* lse;
  float* lse_kv;
  float* max_logits;
  float* lse_indexer;  // [T, H] or nullptr
  uint32_t* status;
  int T, Tkv, H, G, K, Dv;
  int snap_tiles;  // indexer_topk / 64: lse_indexer is taken after this many tiles (0: off)
  int n_qk;      // Dqk / 64
  int n_v;       // Dv / 64
  int n_chunks;  // 64-dim chunks per tile buffer
  int v_first;   // chunk index of value dims 0..63
  int p_alias;   // chunk whose space holds P^T, or -1 (separate buffers)
  int kv_row_bytes, v_row_bytes;
  float scale_log2;
};

struct Layout {
  uint32_t q, kv, p, small, bars, misc, total;
  uint32_t buf_bytes;
};

__host__ __device__ inline Layout make_layout(int n_qk, int n_chunks, int p_alias) {
  Layout L;
  uint32_t o = 0;
  L.q = o;
  o += n_qk * kQChunkBytes;
  L.kv = o;
  L.buf_bytes = n_chunks * kChunkBytes;
  o += 2 * L.buf_bytes;
  if (p_alias >= 0) {
    L.p = 0xFFFFFFFFu;  // P^T of buffer b lives in chunk p_alias of buffer b
  } else {
    L.p = o;
    o += 2 * kChunkBytes;
  }
  L.small = o;
  o += (4 * 64 + 4 * 64 + 64 + 64 + 64 + 16) * 4;  // wmax | red | alpha | mref | fac | exflag
  L.bars = o;
  o += 16 * 8;
  L.misc = o;
  o += 16;
  L.total = o;
  return L;
}

__device__ __forceinline__ int ord_f32(float f) {
  int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float unord_f32(int i) { return __int_as_float(i >= 0 ? i : (i ^ 0x7FFFFFFF)); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One lane of the (converged) warp: true there, false elsewhere.
__device__ __forceinline__ bool elect_sync() {
  uint32_t is = 0;
  asm volatile(
      "{\n .reg .pred P;\n elect.sync _|P, 0xffffffff;\n selp.u32 %0, 1, 0, P;\n}" : "=r"(is));
  return is != 0;
}

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ int unit_len(const AttnParams& p, int t) {
  int L = p.K;
  if (p.topk_length) {
    L = __ldg(p.topk_length + t);
    L = L < 0 ? 0 : (L > p.K ? p.K : L);
  }
  return L;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 16-byte global -> shared copy; src_bytes = 0 fills zeros without reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
               "r"(src_bytes), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap map_q, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dsa::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const Layout L = make_layout(p.n_qk, p.n_chunks, p.p_alias);
  uint8_t* qbuf = smem + L.q;
  uint8_t* kvbuf = smem + L.kv;
  int* wmax = reinterpret_cast<int*>(smem + L.small);  // [4 quarters][64 heads]
  float* red = reinterpret_cast<float*>(wmax + 256);   // [4][64]
  float* alpha = red + 256;                            // [64]
  float* mref = alpha + 64;                            // [64]
  float* fac = mref + 64;                              // [64]
  int* exflag = reinterpret_cast<int*>(fac + 64);      // [2][8]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* kv_full = bars;        // [2]
  uint64_t* kv_empty = bars + 2;   // [2]
  uint64_t* s_full = bars + 4;     // [2]
  uint64_t* s_empty = bars + 6;    // [2]
  uint64_t* p_full = bars + 8;     // [2]
  uint64_t* q_full = bars + 10;
  uint64_t* q_empty = bars + 11;
  uint64_t* o_done = bars + 12;
  uint64_t* drain = bars + 13;     // [2]: the MMA issuers' exit commits
  // Completes once per unit, after the unit's last MMA2.  The epilogue waits
  // on it rather than on o_done: o_done completes once per tile, and a parity
  // wait for the last tile's phase would also pass while the tile before it
  // is still running (its phase has the other parity).  Nothing orders that
  // tile's MMA2 before the softmax of the last tile; for the rescale, which
  // waits on o_done for tile i-1 while processing tile i, MMA2 of tile i-2 has
  // completed (it released the buffer that tile i was gathered into).
  uint64_t* o_unit = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_units = p.T * p.G;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      dsa::mbar_init(&kv_full[b], kGatherThreads);
      dsa::mbar_init(&kv_empty[b], 1);
      dsa::mbar_init(&s_full[b], 1);
      dsa::mbar_init(&s_empty[b], kSoftWarps);
      dsa::mbar_init(&p_full[b], kSoftWarps);
    }
    dsa::mbar_init(q_full, 1);
    dsa::mbar_init(q_empty, 1);
    dsa::mbar_init(o_done, 1);
    dsa::mbar_init(&drain[0], 1);
    dsa::mbar_init(&drain[1], 1);
    dsa::mbar_init(o_unit, 1);
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
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLeanRegs));
    // ------------------------------------------------------------ gather
    // Thread g covers piece (g & 7) (16 bytes) of key (g >> 3) + kGatherKeys*kg
    // (keys below 64 only), for every step kg and every 64-dim chunk: one warp
    // instruction = 4 keys x 128 B.
    const int g = threadIdx.x;
    const int piece = g & 7;
    // The gathered rows (kv, v) are re-read by every query row: keep them in L2
    // while the streamed q, ids and outputs pass through.
    const uint64_t keep = dsa::l2_policy_evict_last();
    uint32_t tile_ctr = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int uu = n_units - 1 - u;
      const int t = uu / p.G;
      const int len = unit_len(p, t);
      const int nt = (len + kKeys - 1) / kKeys;
      const int32_t* irow = p.idx + static_cast<int64_t>(t) * p.K;
      // ids are loaded one tile ahead so that their latency hides behind the
      // previous tile's copies
      int nxt[kGatherSteps];
#pragma unroll
      for (int kg = 0; kg < kGatherSteps; ++kg) {
        const int j = kg * kGatherKeys + (g >> 3);
        nxt[kg] = (j < kKeys && j < len) ? __ldcs(irow + j) : -1;
      }
      for (int i = 0; i < nt; ++i, ++tile_ctr) {
        const int b = tile_ctr & 1;
        int id[kGatherSteps];
#pragma unroll
        for (int kg = 0; kg < kGatherSteps; ++kg) {
          id[kg] = (nxt[kg] >= 0 && nxt[kg] < p.Tkv) ? nxt[kg] : -1;
          const int jk = kg * kGatherKeys + (g >> 3);
          const int j = (i + 1) * kKeys + jk;
          nxt[kg] = (i + 1 < nt && jk < kKeys && j < len) ? __ldcs(irow + j) : -1;
        }
        if (!dsa::mbar_wait(&kv_empty[b], ((tile_ctr >> 1) & 1) ^ 1, wt)) { ok = false; break; }
        dsa::fence_proxy_async_smem();
        const uint32_t buf = dsa::smem_u32(kvbuf) + b * L.buf_bytes;
#pragma unroll
        for (int kg = 0; kg < kGatherSteps; ++kg) {
          const int key = kg * kGatherKeys + (g >> 3);
          if (key >= kKeys) continue;
          const uint32_t nbytes = id[kg] >= 0 ? 16u : 0u;
          const int64_t row = id[kg] >= 0 ? id[kg] : 0;
          // checked build: the row is inside kv (and v), the slot inside the tile buffer
          if (!dsa::check(row < p.Tkv && (p.n_qk + (p.v ? p.n_v : 0)) * kChunkBytes <= L.buf_bytes, p.status))
            continue;
          const uint8_t* krow = p.kv + row * p.kv_row_bytes + piece * 16;
          for (int c = 0; c < p.n_qk; ++c)
            cp_async16(buf + c * kChunkBytes + dsa::sw128_offset(key, piece * 16), krow + c * 128, nbytes, keep);
          if (p.v) {
            const uint8_t* vrow = p.v + row * p.v_row_bytes + piece * 16;
            for (int c = 0; c < p.n_v; ++c)
              cp_async16(buf + (p.n_qk + c) * kChunkBytes + dsa::sw128_offset(key, piece * 16), vrow + c * 128,
                         nbytes, keep);
          }
        }
        // the tile is signalled with a plain release arrive once this thread's
        // copies have landed (cp.async.mbarrier.arrive, which signals from the
        // copy engine, gave stale tiles on GB300 when other warps arrived on
        // other barriers meanwhile; waiting here costs nothing measurable,
        // the next tile's buffer is not free before these copies land anyway)
        cp_async_wait_all();
        dsa::mbar_arrive(&kv_full[b]);
      }
    }
  } else if (warp >= kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLeanRegs));
    if (warp != kMmaWarp && warp != kMma2Warp) goto done;  // the warpgroup's two spare warps
    // ------------------------------------------------------------ MMA issue
    // Two issuing warps, one per product, so that neither waits behind the
    // other's instructions: warp kMmaWarp issues MMA1 (and loads the query),
    // warp kMma2Warp issues MMA2 as soon as a tile's P is written, which
    // frees the tile buffer for the next gather sooner.  Each warp runs its
    // loop converged, so that control flow and the operand descriptors stay
    // warp-uniform, and one elected lane issues each instruction.  The
    // descriptors are built once and advanced by constant offsets (the
    // start-address field counts 16-byte units): with 64-key tiles the tensor
    // core finishes an instruction in a few dozen cycles, so issue cost counts.
    const bool leader = elect_sync();
    const uint32_t kv_addr = dsa::smem_u32(kvbuf);
    const uint32_t buf16 = L.buf_bytes >> 4;
    // next unit of this CTA that has at least one tile (n_units if none)
    auto next_unit = [&](int u) {
      for (; u < n_units; u += gridDim.x)
        if (unit_len(p, (n_units - 1 - u) / p.G) > 0) return u;
      return n_units;
    };
    auto unit_tiles = [&](int u) { return (unit_len(p, (n_units - 1 - u) / p.G) + kKeys - 1) / kKeys; };
    if (warp == kMmaWarp) {
      constexpr uint32_t idesc1 = dsa::idesc_bf16(kKeys, kHG, 0, 0);
      const uint64_t q_desc = dsa::smem_desc(dsa::smem_u32(qbuf), 16, 1024, dsa::kSwizzle128B);
      const uint64_t kv_desc = dsa::smem_desc(kv_addr, 16, 1024, dsa::kSwizzle128B);
      const uint64_t q_policy = dsa::l2_policy_evict_first();  // each query tile is read once
      if (leader) dsa::tma_prefetch_desc(&map_q);
      auto load_q = [&](int u) {
        const int uu = n_units - 1 - u;
        const int t = uu / p.G, g = uu - (uu / p.G) * p.G;
        if (leader) {
          dsa::mbar_expect_tx(q_full, p.n_qk * kQChunkBytes);
          for (int c = 0; c < p.n_qk; ++c)
            dsa::tma_load_3d_hint(qbuf + c * kQChunkBytes, &map_q, c * 64, g * kHG, t, q_full, q_policy);
        }
        __syncwarp();
      };
      uint32_t tile_ctr = 0, unit_ctr = 0;
      bool ok = true;
      bool q_pending = false;  // a query load is in flight that no wait has consumed
      int u = next_unit(blockIdx.x);
      if (u < n_units) {
        load_q(u);
        q_pending = true;
      }
      while (u < n_units && ok) {
        const int nt = unit_tiles(u);
        const int u_next = next_unit(u + gridDim.x);
        if (!dsa::mbar_wait_warp(q_full, unit_ctr & 1, wt)) break;
        q_pending = false;
        // MMA1(tc): S^T[tc&1] = KV(tile tc) . Q^T; needs the tile and a free S buffer
        for (int i = 0; i < nt; ++i, ++tile_ctr) {
          const int b = tile_ctr & 1;
          // every lane waits on its own (as fast as one elected lane would);
          // only a leader whose waits succeeded issues, and the lanes agree
          // on leaving at the end of the tile, where they sync anyway
          const bool got = dsa::mbar_wait(&s_empty[b], ((tile_ctr >> 1) & 1) ^ 1, wt) &&
                           dsa::mbar_wait(&kv_full[b], (tile_ctr >> 1) & 1, wt);
          dsa::fence_proxy_async_smem();  // cp.async (generic proxy) writes -> tcgen05 reads
          dsa::tc_fence_after();
          const uint64_t a0 = kv_desc + b * buf16;
          const uint32_t d = tmem_base + kSCol + b * 64;
          dsa::check(kSCol + b * 64 + kKeys <= static_cast<int>(kOCol), p.status);  // S^T stays clear of O^T
          for (int c = 0; c < p.n_qk; ++c) {
            const uint64_t ac = a0 + c * (kChunkBytes >> 4), bc = q_desc + c * (kQChunkBytes >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              dsa::umma_bf16_if(leader && got, d, ac + kk * 2, bc + kk * 2, idesc1, (c | kk) != 0);
          }
          if (leader && got) dsa::umma_commit(&s_full[b]);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        // the query buffer is free once this unit's MMA1 have run
        if (leader) dsa::umma_commit(q_empty);
        __syncwarp();
        if (u_next < n_units) {
          if (!dsa::mbar_wait_warp(q_empty, unit_ctr & 1, wt)) break;
          load_q(u_next);
          q_pending = true;
        }
        ++unit_ctr;
        u = u_next;
      }
      // leave nothing in flight: the query load no wait consumed (only after
      // an abort), then every MMA1 this warp issued
      if (leader) {
        if (q_pending) dsa::mbar_drain(q_full, unit_ctr & 1, p.status);
        dsa::umma_drain(&drain[0], p.status);
      }
      __syncwarp();
    } else {
      constexpr uint32_t idesc2 = dsa::idesc_bf16(128, kHG, 1, 1);
      const uint64_t v_desc = dsa::smem_desc(kv_addr + p.v_first * kChunkBytes, kChunkBytes, 1024, dsa::kSwizzle128B);
      const uint64_t p_desc =
          p.p_alias >= 0 ? dsa::smem_desc(kv_addr + p.p_alias * kChunkBytes, kChunkBytes, 1024, dsa::kSwizzle128B)
                         : dsa::smem_desc(dsa::smem_u32(smem) + L.p, kChunkBytes, 1024, dsa::kSwizzle128B);
      const uint32_t pbuf16 = p.p_alias >= 0 ? buf16 : (kChunkBytes >> 4);
      uint32_t tile_ctr = 0;
      bool ok = true;
      for (int u = next_unit(blockIdx.x); u < n_units && ok; u = next_unit(u + gridDim.x)) {
        const int nt = unit_tiles(u);
        // MMA2(tc): O^T += V^T(tile tc) . P^T(tile tc); releases the tile buffer
        for (int i = 0; i < nt; ++i, ++tile_ctr) {
          const int b = tile_ctr & 1;
          const bool got = dsa::mbar_wait(&p_full[b], (tile_ctr >> 1) & 1, wt);  // as MMA1: agreed at the tile end
          dsa::tc_fence_after();
          const uint64_t a0 = v_desc + b * buf16, b0 = p_desc + b * pbuf16;
          for (int mb = 0; mb < p.n_v / 2; ++mb) {
            const uint64_t am = a0 + mb * (2 * kChunkBytes >> 4);
            const uint32_t d = tmem_base + kOCol + mb * kHG;
            if (!dsa::check(kOCol + (mb + 1) * kHG <= static_cast<int>(kTmemCols), p.status)) break;
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk)
              dsa::umma_bf16_if(leader && got, d, am + kk * (2048 >> 4), b0 + kk * (2048 >> 4), idesc2, (i > 0 || kk > 0) ? 1u : 0u);
          }
          if (leader && got) {
            dsa::umma_commit(o_done);
            dsa::umma_commit(&kv_empty[b]);
          }
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
        }
        if (ok && leader) dsa::umma_commit(o_unit);  // the unit's O^T is complete
        __syncwarp();
      }
      if (leader) dsa::umma_drain(&drain[1], p.status);  // every MMA2 issued has completed
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftRegs));
    // ------------------------------------------------------------ softmax + epilogue
    const int sw = warp - kSoftWarp0;           // 0..7
    const int st = threadIdx.x - kSoftWarp0 * 32;  // 0..255
    const int quarter = warp & 3;               // TMEM lane quarter
    const int hh = sw >> 2;                     // head half: heads hh*32 .. hh*32+31
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // S^T is read with 16-lane loads (shape 16x256b) so that all 32 threads
    // of a warp hold scores: thread `lane` gets keys kA = lane/4 and kB =
    // lane/4 + 8 of its quarter's 16 and heads hbase + 8j + e (j = 0..3,
    // e = 0..1) of its head half; register 4j+e is (kA, head), 4j+2+e is (kB, head).
    const int kA = quarter * 16 + (lane >> 2), kB = kA + 8;
    const int hbase = hh * 32 + 2 * (lane & 3);
    const bool want_max = p.max_logits != nullptr;
    uint32_t tile_ctr = 0;
    bool ok = true;
    // A wait of this thread gave up.  The eight warps only leave together,
    // at a point that reduces the flag over the group (the per-tile exflag
    // word, or the unit's last barrier); until then a thread whose wait
    // failed carries on with the tile: its TMEM loads and stores stay in the
    // allocation and its global stores in the outputs, so the garbage it may
    // compute is harmless in a kernel that is aborting, and no collective
    // instruction ever sees a diverged warp.
    bool failed = false;
    uint32_t unit_ctr = 0;  // units with at least one tile so far (phases of o_unit)
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int uu = n_units - 1 - u;
      const int t = uu / p.G, g = uu - (uu / p.G) * p.G;
      const int hv = min(kHG, p.H - g * kHG);
      const int len = unit_len(p, t);
      const int nt = (len + kKeys - 1) / kKeys;
      const int64_t orow = static_cast<int64_t>(t) * p.H + g * kHG;
      if (nt == 0) {
        for (int h = 0; h < hv; ++h)
          for (int d = st; d < p.Dv; d += kSoftThreads) p.out[(orow + h) * p.Dv + d] = __float2bfloat16_rn(0.f);
        if (st < hv) {
          p.lse[orow + st] = p.sink ? __ldg(p.sink + g * kHG + st) : -INFINITY;
          if (p.lse_kv) p.lse_kv[orow + st] = INFINITY;
          if (p.max_logits) p.max_logits[orow + st] = -INFINITY;
          if (p.lse_indexer) p.lse_indexer[orow + st] = INFINITY;
        }
        continue;
      }
      float l_part[8];  // [j*2 + e]: running sum of p for head hbase + 8j + e over this thread's keys
      float m_max = -INFINITY;  // exact maximum of head st (threads st < 64), for max_logits
#pragma unroll
      for (int h = 0; h < 8; ++h) l_part[h] = 0.f;
      const int32_t* irow = p.idx + static_cast<int64_t>(t) * p.K;
      int nA = kA < len ? __ldcs(irow + kA) : -1;
      int nB = kB < len ? __ldcs(irow + kB) : -1;
      for (int i = 0; i < nt; ++i, ++tile_ctr) {
        const int b = tile_ctr & 1;
        const uint32_t ph = (tile_ctr >> 1) & 1;
        const int jA = i * kKeys + kA, jB = i * kKeys + kB;
        const bool vA = jA < len && nA >= 0 && nA < p.Tkv;
        const bool vB = jB < len && nB >= 0 && nB < p.Tkv;
        if (i + 1 < nt) {
          nA = jA + kKeys < len ? __ldcs(irow + jA + kKeys) : -1;
          nB = jB + kKeys < len ? __ldcs(irow + jB + kKeys) : -1;
        }
        if (!failed) failed = !dsa::mbar_wait(&s_full[b], ph, wt);
        dsa::tc_fence_after();
        float x[16];
        {
          uint32_t v[16];
          dsa::tmem_ld16x256b_x4(tmem_base + lane_off + kSCol + b * 64 + hh * 32, v);
          dsa::tmem_wait_ld();
#pragma unroll
          for (int r = 0; r < 16; ++r) x[r] = __uint_as_float(v[r]);
        }
        dsa::tc_fence_before();
        __syncwarp();
        if (lane == 0) dsa::mbar_arrive(&s_empty[b]);
        // y = s*log2(e) - m for the current reference m of each head; a tile
        // whose scores pass m + theta anywhere moves the reference first
        float y[16];
        bool ex = false;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 m2 = *reinterpret_cast<const float2*>(mref + hbase + 8 * j);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float m = e ? m2.y : m2.x;
            y[4 * j + e] = vA ? fmaf(x[4 * j + e], p.scale_log2, -m) : -INFINITY;
            y[4 * j + 2 + e] = vB ? fmaf(x[4 * j + 2 + e], p.scale_log2, -m) : -INFINITY;
            ex |= (y[4 * j + e] > kTheta) || (y[4 * j + 2 + e] > kTheta);
          }
        }
        // bit 0: some thread of the warp passes the reference; bit 1: some
        // thread's wait gave up (one reduction, where a vote was due anyway)
        const uint32_t wflags = __reduce_or_sync(0xffffffffu, (ex ? 1u : 0u) | (failed ? 2u : 0u));
        if (lane == 0) exflag[(tile_ctr & 1) * 8 + sw] = static_cast<int>(wflags);
        named_bar(1, kSoftThreads);
        // the first tile of a unit always sets the reference (mref still holds
        // the previous unit's, so its y above are discarded)
        bool reduce = want_max || i == 0;
        bool need_rescale = false;
        int any_failed = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const int f = exflag[(tile_ctr & 1) * 8 + w];
          reduce |= (f & 1) != 0;
          any_failed |= f & 2;
        }
        if (any_failed) {  // every softmax thread read the same flags: the group leaves together
          ok = false;
          break;
        }
        if (reduce) {
          // tile maximum per head: this thread's two keys, then the 8 threads
          // that share its heads (lane bits 2..4)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float mx = fmaxf(vA ? x[4 * j + e] * p.scale_log2 : -INFINITY,
                               vB ? x[4 * j + 2 + e] * p.scale_log2 : -INFINITY);
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
              if (lane < 4) wmax[quarter * 64 + hbase + 8 * j + e] = ord_f32(mx);
            }
          }
          named_bar(1, kSoftThreads);
          if (st < 64) {
            int r = max(max(wmax[st], wmax[64 + st]), max(wmax[128 + st], wmax[192 + st]));
            const float tmax = unord_f32(r);
            const float mo = i == 0 ? -INFINITY : mref[st];
            const float mn = (tmax > mo + kTheta) ? tmax : mo;
            alpha[st] = (mn == mo) ? 1.f : ex2(mo - mn);
            mref[st] = mn;
            m_max = fmaxf(m_max, tmax);
          }
          named_bar(1, kSoftThreads);
          bool rescale = false;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 a2 = *reinterpret_cast<const float2*>(alpha + hbase + 8 * j);
            const float2 m2 = *reinterpret_cast<const float2*>(mref + hbase + 8 * j);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float a = e ? a2.y : a2.x;
              const float m = e ? m2.y : m2.x;
              rescale |= a != 1.f;
              l_part[2 * j + e] *= a;
              y[4 * j + e] = vA ? fmaf(x[4 * j + e], p.scale_log2, -m) : -INFINITY;
              y[4 * j + 2 + e] = vB ? fmaf(x[4 * j + 2 + e], p.scale_log2, -m) : -INFINITY;
            }
          }
          // warp-uniform: the rescale below loads the warp's 32 heads from TMEM
          // (heads whose reference did not move have alpha = 1)
          need_rescale = __any_sync(0xffffffffu, rescale) && i > 0;
        }
        // P^T rows kA and kB: heads hbase + 8j + {0, 1} are 4 bytes at 16-byte
        // unit hh*4 + j of the row (128-byte swizzle: unit ^ (key & 7))
        uint8_t* pbase = p.p_alias >= 0 ? kvbuf + b * L.buf_bytes + p.p_alias * kChunkBytes : smem + L.p + b * kChunkBytes;
        uint8_t* prowA = pbase + kA * 128 + 4 * (lane & 3);
        uint8_t* prowB = pbase + kB * 128 + 4 * (lane & 3);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float a0 = ex2(y[4 * j]), a1 = ex2(y[4 * j + 1]);
          const float b0 = ex2(y[4 * j + 2]), b1 = ex2(y[4 * j + 3]);
          l_part[2 * j] += a0 + b0;
          l_part[2 * j + 1] += a1 + b1;
          const int u = hh * 4 + j;
          *reinterpret_cast<uint32_t*>(prowA + ((u ^ (kA & 7)) * 16)) = pack_bf16x2(a0, a1);
          *reinterpret_cast<uint32_t*>(prowB + ((u ^ (kB & 7)) * 16)) = pack_bf16x2(b0, b1);
        }
        // O^T columns of heads whose reference moved get alpha[h]; this runs after
        // P is written so that the scores are no longer live.
        if (need_rescale) {
          // MMA2 of the previous tile must have landed before O^T is scaled
          if (!failed) failed = !dsa::mbar_wait(o_done, ((tile_ctr - 1) & 1), wt);
          dsa::tc_fence_after();
          const float* a32 = alpha + hh * 32;
          for (int mb = 0; mb < p.n_v / 2; ++mb) {
            const uint32_t ta = tmem_base + lane_off + kOCol + mb * kHG + hh * 32;
            uint32_t v[32];
            dsa::tmem_ld32(ta, v);
            dsa::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * a32[c]);
            dsa::tmem_st32(ta, v);
          }
          dsa::tmem_wait_st();
        }
        dsa::fence_proxy_async_smem();
        dsa::tc_fence_before();
        __syncwarp();
        if (lane == 0) dsa::mbar_arrive(&p_full[b]);
        // lse_indexer: the LSE of the slots of the first snap_tiles tiles (all
        // of a shorter row), from the sums so far, relative to the current
        // reference like the final statistics
        if (p.snap_tiles > 0 && i == min(p.snap_tiles, nt) - 1) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float v = l_part[2 * j + e];
              v += __shfl_xor_sync(0xffffffffu, v, 4);
              v += __shfl_xor_sync(0xffffffffu, v, 8);
              v += __shfl_xor_sync(0xffffffffu, v, 16);
              if (lane < 4) red[quarter * 64 + hbase + 8 * j + e] = v;
            }
          }
          named_bar(1, kSoftThreads);
          if (st < hv) {
            const float l = red[st] + red[64 + st] + red[128 + st] + red[192 + st];
            p.lse_indexer[orow + st] = l > 0.f ? (mref[st] + log2f(l)) * kLn2 : INFINITY;
          }
          named_bar(1, kSoftThreads);  // red is read before the epilogue reuses it
        }
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      if (!failed) failed = !dsa::mbar_wait(o_unit, unit_ctr & 1, wt);
      ++unit_ctr;
      dsa::tc_fence_after();
      // per-head sums over the quarter's 16 keys: the 8 threads sharing a head
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = l_part[2 * j + e];
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 8);
          v += __shfl_xor_sync(0xffffffffu, v, 16);
          if (lane < 4) red[quarter * 64 + hbase + 8 * j + e] = v;
        }
      }
      named_bar(1, kSoftThreads);
      if (st < 64) {
        const float l = red[st] + red[64 + st] + red[128 + st] + red[192 + st];
        const float mc = mref[st];
        const float sk = (p.sink && st < hv) ? __ldg(p.sink + g * kHG + st) * kLog2e : -INFINITY;
        float f = 0.f, lse_v, lkv, mlog = -INFINITY;
        if (l > 0.f) {
          const float M = fmaxf(mc, sk);
          const float a = exp2f(mc - M);
          const float z = l * a + exp2f(sk - M);
          f = a / z;
          lse_v = (M + log2f(z)) * kLn2;
          lkv = (mc + log2f(l)) * kLn2;
          if (want_max) mlog = m_max * kLn2;  // x = s*log2(e), so max s = max x * ln(2)
        } else {
          lse_v = sk * kLn2;
          lkv = INFINITY;
        }
        fac[st] = f;
        if (st < hv) {
          p.lse[orow + st] = lse_v;
          if (p.lse_kv) p.lse_kv[orow + st] = lkv;
          if (p.max_logits) p.max_logits[orow + st] = mlog;
        }
      }
      named_bar(1, kSoftThreads);
      {
        const float* f32 = fac + hh * 32;
        const int hcount = min(32, hv - hh * 32);  // real heads in this warp's half
        for (int mb = 0; mb < p.n_v / 2; ++mb) {
          uint32_t v[32];
          dsa::tmem_ld32(tmem_base + lane_off + kOCol + mb * kHG + hh * 32, v);
          dsa::tmem_wait_ld();
          __nv_bfloat16* o = p.out + (orow + hh * 32) * p.Dv + mb * 128 + quarter * 32 + lane;
          // checked build: the head rows written are inside out [T, H, Dv]
          const bool in_out =
              dsa::check(hcount <= 0 || (orow + hh * 32 + hcount) * p.Dv <= static_cast<int64_t>(p.T) * p.H * p.Dv,
                         p.status);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c < hcount && in_out) __stcs(o, __float2bfloat16_rn(__uint_as_float(v[c]) * f32[c]));
            o += p.Dv;
          }
        }
      }
      dsa::tc_fence_before();
      // the unit's last barrier: the group leaves together if any warp's wait gave up
      if (dsa::named_bar_any(1, kSoftThreads, failed)) {
        ok = false;
        break;
      }
    }
  }

done:
  __syncthreads();
  if (warp == kMmaWarp) {
    dsa::tc_fence_after();
    dsa::tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

extern "C" int dsa_sparse_attn_fwd_ex(const void* q, const void* kv, const void* v, const int32_t* idx,
                                      const int32_t* topk_length, const float* sink, int T, int Tkv, int H, int Dqk,
                                      int Dv, int K, float scale, void* out, float* lse, float* lse_kv,
                                      float* max_logits, int indexer_topk, float* lse_indexer, cudaStream_t stream) {
  dsa::clear_error();
  if (indexer_topk < 0 || indexer_topk % 64 != 0 || indexer_topk > K)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_sparse_attn_fwd: indexer_topk must be a multiple of 64 in [0, K]");
  if (indexer_topk > 0 && T > 0 && !lse_indexer)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_sparse_attn_fwd: lse_indexer is NULL while indexer_topk > 0");
  const bool latent = (Dqk == 576 || Dqk == 512) && Dv == 512 && v == nullptr;
  const bool separate = Dqk == 256 && Dv == 256 && v != nullptr;
  if (!latent && !separate)
    return dsa::set_error(DSA_ERR_VALUE,
                          "dsa_sparse_attn_fwd: (Dqk, Dv) must be (576|512, 512) with v == NULL or (256, 256) with v");
  if (T < 0 || Tkv < 1 || H < 1 || H > 128 || K < 0)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_sparse_attn_fwd: need T >= 0, Tkv >= 1, 1 <= H <= 128, K >= 0");
  if (!(scale > 0.f) || !(scale < INFINITY))
    return dsa::set_error(DSA_ERR_VALUE, "dsa_sparse_attn_fwd: scale must be finite and > 0");
  if (T > 0 && (!q || !kv || !out || !lse || (K > 0 && !idx)))
    return dsa::set_error(DSA_ERR_VALUE, "dsa_sparse_attn_fwd: NULL pointer");
  if (!dsa::aligned(q, 16) || !dsa::aligned(kv, 16) || (v && !dsa::aligned(v, 16)) || !dsa::aligned(out, 16))
    return dsa::set_error(DSA_ERR_VALUE, "dsa_sparse_attn_fwd: q, kv, v and out must be 16-byte aligned");
  int sms = 0;
  int rc = dsa::check_device(&sms);
  if (rc != DSA_OK) return rc;
  if (T == 0) return DSA_OK;

  AttnParams p{};
  p.idx = idx;
  p.topk_length = topk_length;
  p.sink = sink;
  p.kv = static_cast<const uint8_t*>(kv);
  p.v = static_cast<const uint8_t*>(v);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.lse_kv = lse_kv;
  p.max_logits = max_logits;
  p.lse_indexer = indexer_topk > 0 ? lse_indexer : nullptr;
  p.snap_tiles = indexer_topk / kKeys;
  p.status = dsa::device_status_ptr();
  p.T = T;
  p.Tkv = Tkv;
  p.H = H;
  p.G = (H + kHG - 1) / kHG;
  p.K = K;
  p.Dv = Dv;
  p.n_qk = Dqk / 64;
  p.n_v = Dv / 64;
  p.kv_row_bytes = Dqk * 2;
  p.v_row_bytes = Dv * 2;
  p.scale_log2 = scale * kLog2e;
  if (latent) {
    p.n_chunks = p.n_qk;
    p.v_first = 0;
    p.p_alias = Dqk == 576 ? 8 : -1;
  } else {
    p.n_chunks = p.n_qk + p.n_v;
    p.v_first = p.n_qk;
    p.p_alias = -1;
  }
  CUtensorMap mq;
  rc = dsa::encode_tensor_map_3d(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Dqk, H, T, static_cast<uint64_t>(Dqk) * 2,
                                 static_cast<uint64_t>(Dqk) * H * 2, 64, kHG, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != DSA_OK) return rc;
  const Layout L = make_layout(p.n_qk, p.n_chunks, p.p_alias);
  const size_t smem = L.total + 1024;
  {
    // the register split assumes the launch count it was sized for: with
    // fewer registers at launch the softmax warps' increase could not be met
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, sparse_attn_kernel) != cudaSuccess || fa.numRegs != kLaunchRegs)
      return dsa::set_error(DSA_ERR_CUDA, "sparse_attn_kernel: compiled with %d registers per thread, expected %d",
                            fa.numRegs, kLaunchRegs);
  }
  if (cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return dsa::launch_error("sparse_attn_kernel smem attribute");
  const int units = T * p.G;
  const int grid = units < sms ? units : sms;
  sparse_attn_kernel<<<grid, kThreads, smem, stream>>>(mq, p);
  return dsa::launch_error("sparse_attn_kernel");
}

extern "C" int dsa_sparse_attn_fwd(const void* q, const void* kv, const void* v, const int32_t* idx,
                                   const int32_t* topk_length, const float* sink, int T, int Tkv, int H, int Dqk,
                                   int Dv, int K, float scale, void* out, float* lse, float* lse_kv, float* max_logits,
                                   cudaStream_t stream) {
  return dsa_sparse_attn_fwd_ex(q, kv, v, idx, topk_length, sink, T, Tkv, H, Dqk, Dv, K, scale, out, lse, lse_kv,
                                max_logits, 0, nullptr, stream);
}
