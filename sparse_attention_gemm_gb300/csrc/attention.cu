// attention.cu -- sparse MQA attention forward on tcgen05.
//
// cuDNN Frontend DSA page, section 1 (Sparse Attention Forward): for query
// row t, head h and valid top-k slot j, s_j = scale * q[t,h,:] . kv[idx_j, :];
// invalid or out-of-range ids are absent; duplicates are separate slots; the
// sink enters only the denominator.  Shapes follow NeMo glm_moe_dsa
// cudnn_sparse_attention (q [T,H,576], latent kv [T,1,576], V = first 512
// dims) and, with a separate V of 256 dims, NeMo qwen3_8_flash_next
// cudnn_sparse_gqa_attention.
//
// Work unit = (token t, group g of 64 heads).  Per unit the selected KV rows
// are gathered once (TMA tile::gather4, four rows per instruction) into a
// 128-key tile and shared by all 64 heads of the group (MQA).  Both products
// are "swap AB" so that the 128-wide M of tcgen05.mma is keys or value dims,
// never the 64 heads:
//   MMA1  S^T[key, head]  = KV[key, 0:Dqk] . Q[head, 0:Dqk]^T   (M=128, N=64)
//   MMA2  O^T[dim, head] += V^T[dim, key] . P^T[key, head]      (M=128 per
//         128 value dims, N=64, K=16 keys per instruction)
// S^T and O^T live in TMEM.  Softmax threads own one key (one TMEM lane):
// they scale the 64 scores, keep a running per-head reference maximum
// (online softmax; the accumulator is rescaled only when the maximum grows by
// more than 2^8, which leaves the result exact), exponentiate, accumulate
// per-thread row sums and write P^T (bf16) to shared memory for MMA2.
// The epilogue reduces the row sums, adds the sink to the denominator and
// writes out (bf16), lse (sink included), and optionally lse_kv and
// max_logits.
//
// Warp roles (192 threads): warp 0 gathers (all 32 lanes issue gather4 for 4
// keys each) and loads Q; warp 1 allocates TMEM and issues MMAs; warps 2..5
// run softmax and epilogue.  The KV tile is split into 16 KB chunks of 64
// dims, each with its own full/empty barrier, so the next tile's gather
// starts as soon as MMA2 releases the chunks it no longer reads.
#include <climits>

#include "common.cuh"

namespace {

constexpr int kKeys = 128;
constexpr int kHG = 64;
constexpr int kThreads = 192;
constexpr int kSoftWarps = 4;
constexpr uint32_t kChunkBytes = kKeys * 128;  // 128 keys x 64 bf16
constexpr uint32_t kQChunkBytes = kHG * 128;   // 64 heads x 64 bf16
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kTheta = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr int kSCol = 0;
constexpr int kOCol = 64;

struct AttnParams {
  const int32_t* idx;
  const int32_t* topk_length;
  const float* sink;
  __nv_bfloat16* out;
  float* lse;
  float* lse_kv;
  float* max_logits;
  uint32_t* status;
  int T, Tkv, H, G, K, Dv;
  int n_qk;      // Dqk / 64
  int n_v;       // Dv / 64
  int n_chunks;  // KV chunks per tile
  int v_first;   // chunk index of value dims 0..63
  int p_alias;   // chunk whose buffer holds P^T, or -1 (separate buffer)
  float scale_log2;
};

struct Layout {
  uint32_t q, kv, p, small, bars, misc, total;
};

__host__ __device__ inline Layout make_layout(int n_qk, int n_chunks, int p_alias) {
  Layout L;
  uint32_t o = 0;
  L.q = o;
  o += n_qk * kQChunkBytes;
  L.kv = o;
  o += n_chunks * kChunkBytes;
  if (p_alias >= 0) {
    L.p = L.kv + p_alias * kChunkBytes;
  } else {
    L.p = o;
    o += kChunkBytes;
  }
  L.small = o;
  o += (64 * 4 + 4 * 64 + 4 * 64 + 8) * 4;  // m_cur m_max alpha fac | wmax | red | exflag
  L.bars = o;
  o += (16 + 16 + 6) * 8;
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

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ int unit_tiles(const AttnParams& p, int t, int* len_out) {
  int L = p.K;
  if (p.topk_length) {
    L = __ldg(p.topk_length + t);
    L = L < 0 ? 0 : (L > p.K ? p.K : L);
  }
  *len_out = L;
  return (L + kKeys - 1) / kKeys;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_v, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dsa::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const Layout L = make_layout(p.n_qk, p.n_chunks, p.p_alias);
  uint8_t* qbuf = smem + L.q;
  uint8_t* kvbuf = smem + L.kv;
  uint8_t* pbuf = smem + L.p;
  float* m_cur = reinterpret_cast<float*>(smem + L.small);
  float* m_max = m_cur + 64;
  float* alpha = m_cur + 128;
  float* fac = m_cur + 192;
  int* wmax = reinterpret_cast<int*>(m_cur + 256);
  float* red = m_cur + 512;
  int* exflag = reinterpret_cast<int*>(m_cur + 768);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + 16;
  uint64_t* q_full = bars + 32;
  uint64_t* q_empty = bars + 33;
  uint64_t* s_full = bars + 34;
  uint64_t* s_empty = bars + 35;
  uint64_t* p_full = bars + 36;
  uint64_t* o_done = bars + 37;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_units = p.T * p.G;

  if (threadIdx.x == 0) {
    for (int c = 0; c < p.n_chunks; ++c) {
      dsa::mbar_init(&kv_full[c], 1);
      dsa::mbar_init(&kv_empty[c], 1);
    }
    dsa::mbar_init(q_full, 1);
    dsa::mbar_init(q_empty, 1);
    dsa::mbar_init(s_full, 1);
    dsa::mbar_init(s_empty, kSoftWarps);
    dsa::mbar_init(p_full, kSoftWarps);
    dsa::mbar_init(o_done, 1);
    *abort_flag = 0;
    dsa::fence_barrier_init();
  }
  if (warp == 1) dsa::tmem_alloc(tmem_slot, kTmemCols);
  dsa::tc_fence_before();
  __syncthreads();
  dsa::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ gather
    if (lane == 0) {
      dsa::tma_prefetch_desc(&map_q);
      dsa::tma_prefetch_desc(&map_k);
      dsa::tma_prefetch_desc(&map_v);
    }
    uint32_t tile_ctr = 0, unit_ctr = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int uu = n_units - 1 - u;
      const int t = uu / p.G, g = uu - (uu / p.G) * p.G;
      int len;
      const int nt = unit_tiles(p, t, &len);
      if (nt == 0) continue;
      int good = 1;
      if (lane == 0) {
        if (unit_ctr > 0 && !dsa::mbar_wait(q_empty, (unit_ctr - 1) & 1, abort_flag, p.status)) good = 0;
        if (good) {
          dsa::mbar_expect_tx(q_full, p.n_qk * kQChunkBytes);
          for (int c = 0; c < p.n_qk; ++c) dsa::tma_load_3d(qbuf + c * kQChunkBytes, &map_q, c * 64, g * kHG, t, q_full);
        }
      }
      if (!__shfl_sync(0xffffffffu, good, 0)) { ok = false; break; }
      ++unit_ctr;
      const int32_t* irow = p.idx + static_cast<int64_t>(t) * p.K;
      for (int i = 0; i < nt && ok; ++i, ++tile_ctr) {
        int y[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = i * kKeys + lane * 4 + e;
          int id = j < len ? __ldg(irow + j) : -1;
          y[e] = (id >= 0 && id < p.Tkv) ? id : -1;
        }
        for (int c = 0; c < p.n_chunks; ++c) {
          if (lane == 0) {
            good = dsa::mbar_wait(&kv_empty[c], (tile_ctr & 1) ^ 1, abort_flag, p.status);
            if (good) dsa::mbar_expect_tx(&kv_full[c], kChunkBytes);
          }
          if (!__shfl_sync(0xffffffffu, good, 0)) { ok = false; break; }
          const bool is_v = c >= p.n_qk;
          const CUtensorMap* m = is_v ? &map_v : &map_k;
          const int x = (is_v ? c - p.n_qk : c) * 64;
          dsa::tma_gather4(kvbuf + c * kChunkBytes + lane * 512, m, x, y[0], y[1], y[2], y[3], &kv_full[c]);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (lane == 0) {
      constexpr uint32_t idesc1 = dsa::idesc_bf16(kKeys, kHG, 0, 0);
      constexpr uint32_t idesc2 = dsa::idesc_bf16(kKeys, kHG, 1, 1);
      const uint32_t q_addr = dsa::smem_u32(qbuf), kv_addr = dsa::smem_u32(kvbuf), p_addr = dsa::smem_u32(pbuf);
      const uint32_t tS = tmem_base + kSCol;
      uint32_t tile_ctr = 0, unit_ctr = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const int uu = n_units - 1 - u;
        const int t = uu / p.G;
        int len;
        const int nt = unit_tiles(p, t, &len);
        if (nt == 0) continue;
        if (!dsa::mbar_wait(q_full, unit_ctr & 1, abort_flag, p.status)) break;
        ++unit_ctr;
        for (int i = 0; i < nt; ++i, ++tile_ctr) {
          const uint32_t ph = tile_ctr & 1;
          // MMA1: S^T = KV . Q^T over the Dqk chunks
          if (!dsa::mbar_wait(s_empty, ph ^ 1, abort_flag, p.status)) { ok = false; break; }
          for (int c = 0; c < p.n_qk; ++c) {
            if (!dsa::mbar_wait(&kv_full[c], ph, abort_flag, p.status)) { ok = false; break; }
            dsa::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = dsa::smem_desc(kv_addr + c * kChunkBytes + kk * 32, 16, 1024, dsa::kSwizzle128B);
              const uint64_t bd = dsa::smem_desc(q_addr + c * kQChunkBytes + kk * 32, 16, 1024, dsa::kSwizzle128B);
              dsa::umma_bf16(tS, ad, bd, idesc1, (c | kk) != 0);
            }
          }
          if (!ok) break;
          dsa::umma_commit(s_full);
          // chunks read only by MMA1 (and not holding P^T) are free now
          for (int c = 0; c < p.n_qk; ++c) {
            const bool is_value = (c >= p.v_first && c < p.v_first + p.n_v);
            if (!is_value && c != p.p_alias) dsa::umma_commit(&kv_empty[c]);
          }
          if (i == nt - 1) dsa::umma_commit(q_empty);
          // MMA2: O^T += V^T . P^T, 128 value dims per instruction group
          if (!dsa::mbar_wait(p_full, ph, abort_flag, p.status)) { ok = false; break; }
          dsa::tc_fence_after();
          for (int mb = 0; mb < p.n_v / 2 && ok; ++mb) {
            const int c0 = p.v_first + 2 * mb;
            if (c0 >= p.n_qk) {  // separate V: these chunks were not waited for by MMA1
              if (!dsa::mbar_wait(&kv_full[c0], ph, abort_flag, p.status) ||
                  !dsa::mbar_wait(&kv_full[c0 + 1], ph, abort_flag, p.status)) {
                ok = false;
                break;
              }
              dsa::tc_fence_after();
            }
            const uint32_t tO = tmem_base + kOCol + mb * kHG;
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk) {
              const uint64_t ad =
                  dsa::smem_desc(kv_addr + c0 * kChunkBytes + kk * 2048, kChunkBytes, 1024, dsa::kSwizzle128B);
              const uint64_t bd = dsa::smem_desc(p_addr + kk * 2048, kChunkBytes, 1024, dsa::kSwizzle128B);
              dsa::umma_bf16(tO, ad, bd, idesc2, (i > 0 || kk > 0) ? 1u : 0u);
            }
            dsa::umma_commit(&kv_empty[c0]);
            dsa::umma_commit(&kv_empty[c0 + 1]);
          }
          if (!ok) break;
          dsa::umma_commit(o_done);
          if (p.p_alias >= 0) dsa::umma_commit(&kv_empty[p.p_alias]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int st = threadIdx.x - 64;  // 0..127
    const int wq = warp - 2;          // softmax warp 0..3
    const int quarter = warp & 3;     // TMEM lane quarter
    const int key_lane = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const bool want_max = p.max_logits != nullptr;
    uint32_t tile_ctr = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int uu = n_units - 1 - u;
      const int t = uu / p.G, g = uu - (uu / p.G) * p.G;
      const int hv = min(kHG, p.H - g * kHG);
      int len;
      const int nt = unit_tiles(p, t, &len);
      const int64_t orow = static_cast<int64_t>(t) * p.H + g * kHG;  // first (t, head) row of the group
      if (nt == 0) {
        for (int h = 0; h < hv; ++h)
          for (int d = st; d < p.Dv; d += 128) p.out[(orow + h) * p.Dv + d] = __float2bfloat16_rn(0.f);
        if (st < hv) {
          p.lse[orow + st] = p.sink ? __ldg(p.sink + g * kHG + st) : -INFINITY;
          if (p.lse_kv) p.lse_kv[orow + st] = INFINITY;
          if (p.max_logits) p.max_logits[orow + st] = -INFINITY;
        }
        continue;
      }
      if (st < 64) {
        m_cur[st] = -INFINITY;
        m_max[st] = -INFINITY;
      }
      float l_part[64];
#pragma unroll
      for (int h = 0; h < 64; ++h) l_part[h] = 0.f;
      named_bar(1, 128);
      const int32_t* irow = p.idx + static_cast<int64_t>(t) * p.K;

      for (int i = 0; i < nt; ++i, ++tile_ctr) {
        const uint32_t ph = tile_ctr & 1;
        if (!dsa::mbar_wait(s_full, ph, abort_flag, p.status)) { ok = false; break; }
        dsa::tc_fence_after();
        float x[64];
        {
          uint32_t va[32], vb[32];
          dsa::tmem_ld32(tmem_base + lane_off + kSCol, va);
          dsa::tmem_ld32(tmem_base + lane_off + kSCol + 32, vb);
          dsa::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) {
            x[h] = __uint_as_float(va[h]);
            x[h + 32] = __uint_as_float(vb[h]);
          }
        }
        dsa::tc_fence_before();
        __syncwarp();
        if (lane == 0) dsa::mbar_arrive(s_empty);

        const int j = i * kKeys + key_lane;
        const int id = j < len ? __ldg(irow + j) : -1;
        const bool valid = j < len && id >= 0 && id < p.Tkv;
        bool ex = false;
#pragma unroll
        for (int h = 0; h < 64; ++h) {
          x[h] = valid ? x[h] * p.scale_log2 : -INFINITY;
          ex |= x[h] > m_cur[h] + kTheta;
        }
        const bool ex_warp = __any_sync(0xffffffffu, ex);
        if (lane == 0) exflag[(ph << 2) + wq] = ex_warp ? 1 : 0;
        named_bar(1, 128);
        const bool reduce = want_max || exflag[ph << 2] || exflag[(ph << 2) + 1] || exflag[(ph << 2) + 2] ||
                            exflag[(ph << 2) + 3];
        if (reduce) {
#pragma unroll
          for (int h = 0; h < 64; ++h) {
            const int r = __reduce_max_sync(0xffffffffu, ord_f32(x[h]));
            if (lane == (h & 31)) wmax[wq * 64 + h] = r;
          }
          named_bar(1, 128);
          if (st < 64) {
            int r = wmax[st];
            r = max(r, wmax[64 + st]);
            r = max(r, wmax[128 + st]);
            r = max(r, wmax[192 + st]);
            const float tmax = unord_f32(r);
            m_max[st] = fmaxf(m_max[st], tmax);
            const float mo = m_cur[st];
            const float mn = (tmax > mo + kTheta) ? tmax : mo;
            alpha[st] = (mn == mo) ? 1.f : exp2f(mo - mn);
            m_cur[st] = mn;
          }
          named_bar(1, 128);
          bool rescale = false;
#pragma unroll
          for (int h = 0; h < 64; ++h) {
            const float a = alpha[h];
            rescale |= a != 1.f;
            l_part[h] *= a;
          }
          if (rescale && i > 0) {
            // O^T columns of heads whose reference maximum moved get alpha[h];
            // MMA2 of the previous tile must have landed first.
            if (!dsa::mbar_wait(o_done, ph ^ 1, abort_flag, p.status)) { ok = false; break; }
            dsa::tc_fence_after();
            for (int mb = 0; mb < p.n_v / 2; ++mb) {
              for (int half = 0; half < 2; ++half) {
                const uint32_t ta = tmem_base + lane_off + kOCol + mb * kHG + half * 32;
                uint32_t v[32];
                dsa::tmem_ld32(ta, v);
                dsa::tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha[half * 32 + c]);
                dsa::tmem_st32(ta, v);
              }
            }
            dsa::tmem_wait_st();
          }
        }
        // P^T row of this key: 64 bf16 = 8 chunks of 16 bytes, 128-byte swizzle
        uint8_t* prow = pbuf + key_lane * 128;
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int h0 = c16 * 8 + e * 2;
            const float p0 = valid ? exp2f(x[h0] - m_cur[h0]) : 0.f;
            const float p1 = valid ? exp2f(x[h0 + 1] - m_cur[h0 + 1]) : 0.f;
            l_part[h0] += p0;
            l_part[h0 + 1] += p1;
            w4[e] = pack_bf16x2(p0, p1);
          }
          const int pos = (c16 ^ (key_lane & 7)) * 16;
          *reinterpret_cast<uint4*>(prow + pos) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        dsa::fence_proxy_async_smem();
        dsa::tc_fence_before();
        __syncwarp();
        if (lane == 0) dsa::mbar_arrive(p_full);
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      if (!dsa::mbar_wait(o_done, (tile_ctr - 1) & 1, abort_flag, p.status)) { ok = false; break; }
      dsa::tc_fence_after();
      // l_part summed over the 128 key threads: transpose-reduce within the
      // warp (lane ends with heads 2*lane, 2*lane+1), then across warps.
#pragma unroll
      for (int off = 16, n = 32; off >= 1; off >>= 1, n >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < n; ++k) {
          const float send = upper ? l_part[k] : l_part[k + n];
          const float keep = upper ? l_part[k + n] : l_part[k];
          l_part[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      red[wq * 64 + 2 * lane] = l_part[0];
      red[wq * 64 + 2 * lane + 1] = l_part[1];
      named_bar(1, 128);
      if (st < 64) {
        const float l = red[st] + red[64 + st] + red[128 + st] + red[192 + st];
        const float mc = m_cur[st];
        const float sk = (p.sink && st < hv) ? __ldg(p.sink + g * kHG + st) * kLog2e : -INFINITY;
        float f = 0.f, lse_v, lkv, mlog;
        if (l > 0.f) {
          const float M = fmaxf(mc, sk);
          const float a = exp2f(mc - M);
          const float z = l * a + exp2f(sk - M);
          f = a / z;
          lse_v = (M + log2f(z)) * kLn2;
          lkv = (mc + log2f(l)) * kLn2;
          mlog = m_max[st] * kLn2;  // x = s * log2(e), so max s = max x * ln(2)
        } else {
          lse_v = sk * kLn2;
          lkv = INFINITY;
          mlog = -INFINITY;
        }
        fac[st] = f;
        if (st < hv) {
          p.lse[orow + st] = lse_v;
          if (p.lse_kv) p.lse_kv[orow + st] = lkv;
          if (p.max_logits) p.max_logits[orow + st] = mlog;
        }
      }
      named_bar(1, 128);
      for (int mb = 0; mb < p.n_v / 2; ++mb) {
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32];
          dsa::tmem_ld32(tmem_base + lane_off + kOCol + mb * kHG + half * 32, v);
          dsa::tmem_wait_ld();
          const int d = mb * 128 + key_lane;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int h = half * 32 + c;
            if (h < hv) p.out[(orow + h) * p.Dv + d] = __float2bfloat16_rn(__uint_as_float(v[c]) * fac[h]);
          }
        }
      }
      dsa::tc_fence_before();
      named_bar(1, 128);
    }
  }

  __syncthreads();
  if (warp == 1) {
    dsa::tc_fence_after();
    dsa::tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

extern "C" int dsa_sparse_attn_fwd(const void* q, const void* kv, const void* v, const int32_t* idx,
                                   const int32_t* topk_length, const float* sink, int T, int Tkv, int H, int Dqk,
                                   int Dv, int K, float scale, void* out, float* lse, float* lse_kv, float* max_logits,
                                   cudaStream_t stream) {
  dsa::clear_error();
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
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.lse_kv = lse_kv;
  p.max_logits = max_logits;
  p.status = dsa::device_status_ptr();
  p.T = T;
  p.Tkv = Tkv;
  p.H = H;
  p.G = (H + kHG - 1) / kHG;
  p.K = K;
  p.Dv = Dv;
  p.n_qk = Dqk / 64;
  p.n_v = Dv / 64;
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
  CUtensorMap mq, mk, mv;
  rc = dsa::encode_tensor_map_3d(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Dqk, H, T, static_cast<uint64_t>(Dqk) * 2,
                                 static_cast<uint64_t>(Dqk) * H * 2, 64, kHG, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != DSA_OK) return rc;
  rc = dsa::encode_tensor_map_2d(&mk, kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Dqk, Tkv, static_cast<uint64_t>(Dqk) * 2,
                                 64, 1, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != DSA_OK) return rc;
  if (separate) {
    rc = dsa::encode_tensor_map_2d(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Dv, Tkv, static_cast<uint64_t>(Dv) * 2, 64,
                                   1, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != DSA_OK) return rc;
  } else {
    mv = mk;
  }
  const Layout L = make_layout(p.n_qk, p.n_chunks, p.p_alias);
  const size_t smem = L.total + 1024;
  if (cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return dsa::launch_error("sparse_attn_kernel smem attribute");
  const int units = T * p.G;
  const int grid = units < sms ? units : sms;
  sparse_attn_kernel<<<grid, kThreads, smem, stream>>>(mq, mk, mv, p);
  return dsa::launch_error("sparse_attn_kernel");
}
