// common.cuh -- shared device/host helpers of libdsa (sm_103a only).
//
// Inline-PTX wrappers for the Blackwell features the kernels use: mbarriers
// with bounded waits, TMA tiled and gather4 loads, tcgen05 (TMEM allocation,
// MMA issue/commit, TMEM loads/stores, fences) and the shared-memory and
// instruction descriptors that tcgen05.mma reads.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dsa.h"

#ifndef DSA_WAIT_TIMEOUT_NS
#define DSA_WAIT_TIMEOUT_NS 2000000000ull  // 2 s: no legitimate wait comes close
#endif

// The checked build (-DDSA_CHECKED) range-checks the indices and offsets of
// the kernels' shared-memory, TMEM and global accesses before using them: a
// failed check ORs DSA_STATUS_CHECK_FAILED into the status word and the
// access is skipped (never a trap).  In the normal build every check is the
// constant true and compiles away.
#ifdef DSA_CHECKED
#define DSA_CHECKED_BUILD 1
#else
#define DSA_CHECKED_BUILD 0
#endif

namespace dsa {

// ----------------------------------------------------------------- host side
int set_error(int code, const char* fmt, ...);   // records dsa_last_error, returns code
void clear_error();
int check_device(int* sm_count);                 // DSA_OK when the current device is sm_103
uint32_t* device_status_ptr();                   // device address of the status word
int launch_error(const char* what);              // maps cudaGetLastError to DSA_ERR_CUDA

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
int encode_tensor_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                         uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                         uint32_t box_outer, CUtensorMapSwizzle swizzle);
// 3-D map [d2][d1][d0] (d0 innermost, contiguous) with box {b0, b1, b2}.
int encode_tensor_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t d0,
                         uint64_t d1, uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                         uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle swizzle);

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// --------------------------------------------------------------- device side
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t elect_one_lane() { return (threadIdx.x & 31) == 0; }

// ---- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of a phase (try_wait may suspend the thread for a
// while; this returns at once), for threads that poll several barriers.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The library's control block on each device.  Kernels receive the address
// of `status` (the word they OR their DSA_STATUS_* bits into); the limit of
// the bounded waits sits 8 bytes after it: 0 means DSA_WAIT_TIMEOUT_NS, any
// other value (set by dsa_set_wait_limit_ns) replaces it.
struct DeviceControl {
  uint32_t status;
  uint32_t reserved;
  uint64_t wait_limit_ns;
};

static_assert(offsetof(DeviceControl, wait_limit_ns) == 2 * sizeof(uint32_t), "limit 8 bytes after status");

__device__ __forceinline__ uint64_t wait_limit(const uint32_t* status) {
  const uint64_t v = *reinterpret_cast<const volatile uint64_t*>(status + 2);
  return v ? v : DSA_WAIT_TIMEOUT_NS;
}

// What a bounded wait needs: the CTA's abort flag (shared memory), the
// device status word, and whether the wait-limit hook shortened the limit
// below the default (read once per thread when its role starts).
struct Waiter {
  volatile int* abort;
  uint32_t* status;
  bool poll;
};
__device__ __forceinline__ Waiter make_waiter(volatile int* abort, uint32_t* status) {
  const uint64_t v = *reinterpret_cast<const volatile uint64_t*>(status + 2);
  return Waiter{abort, status, v != 0 && v < DSA_WAIT_TIMEOUT_NS};
}

// Bounded wait.  Returns false when the kernel is aborting: either another
// thread already raised *abort, or this wait exceeded the wait limit, in
// which case DSA_STATUS_WAIT_TIMEOUT is OR-ed into the status word first.
// try_wait suspends the thread until the phase completes or a hardware time
// slice ends; under a limit shortened by the failure-detection hook the wait
// polls without suspending instead, so that any wait not satisfied at its
// first probe gives up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Waiter& w) {
  if (w.poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  const uint64_t limit = wait_limit(w.status);
  while (true) {
    if (w.poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (globaltimer() - t0 > limit) {
      atomicOr(w.status, DSA_STATUS_WAIT_TIMEOUT);
      *w.abort = 1;
      return false;
    }
  }
}

// The same wait taken by a whole converged warp: every lane waits and the
// lanes agree on the outcome, so that what follows (tcgen05.ld, which all 32
// lanes must execute, __syncwarp, an elected issuer) sees one decision.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, const Waiter& w) {
  const bool ok = mbar_wait(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

// Before a CTA that is aborting leaves, each thread waits for the
// asynchronous work it issued and nobody consumed (a TMA copy landing in
// shared memory, MMAs reading shared memory and writing TMEM), so that none
// of it outlives the CTA's shared memory and TMEM.  Bounded by
// DSA_WAIT_TIMEOUT_NS whatever the wait-limit override and the abort flag
// say; DSA_STATUS_DRAIN_TIMEOUT if it gave up.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > DSA_WAIT_TIMEOUT_NS) {
      atomicOr(status, DSA_STATUS_DRAIN_TIMEOUT);
      return;
    }
  }
}

// Named barrier `id` over `n` threads (whole warps, converged) that also
// returns, to every participant, whether `pred` held for any of them: the one
// point where a group whose members may have seen different waits give up
// takes a single decision to leave.
__device__ __forceinline__ bool named_bar_any(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// In-kernel range check of the checked build: true when `ok`; otherwise the
// failure is recorded and the caller skips the access.
__device__ __forceinline__ bool check(bool ok, uint32_t* status) {
  if (DSA_CHECKED_BUILD && !ok) {
    atomicOr(status, DSA_STATUS_CHECK_FAILED);
    return false;
  }
  return true;
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tcgen05.mma, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// L2 eviction-priority policies for the .L2::cache_hint forms below.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Four rows y0..y3 (any order, any value; rows outside the tensor read as zero)
// of a box that is one row high and box_inner elements wide, starting at column x.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, int x, int y0, int y1, int y2, int y3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar))
      : "memory");
}

// Contiguous global -> shared copy through the TMA unit (16-byte aligned
// addresses, size a multiple of 16), completing on *bar.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Bulk prefetch of [p, p + bytes) into L2 (p 16-byte aligned, bytes a
// multiple of 16): fire-and-forget, holds no registers or shared memory.
__device__ __forceinline__ void l2_prefetch_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes));
}

// ---- tcgen05 / TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// umma_bf16 issued only by the threads whose `issue` is true, as a predicated
// instruction that the whole (converged) warp executes.  Issue-rate matters
// for small tiles: one thread issuing back to back measured ~50 cycles per
// instruction this way on GB300 and ~85 with a branch around each
// instruction (M = 64 x N = 64 x K = 16 runs in 32 cycles on the tensor core).
__device__ __forceinline__ void umma_bf16_if(bool issue, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p, q; setp.ne.b32 p, %4, 0; setp.ne.b32 q, %5, 0;\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(static_cast<uint32_t>(issue))
      : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4 (8-bit floats in, fp32
// accumulate; K = 32 elements = 32 bytes per instruction).
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= (A * 2^(sfa - 127)) * (B * 2^(sfb - 127))^T, kind::mxf8f6f4
// with E8M0 block scales (scale_vec::1X: one scale per row of A and of B for
// the instruction's 32 elements of K).  The scales are read from TMEM (see
// idesc_mxf8 for which byte of which column).
__device__ __forceinline__ void umma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %6, 0; tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], "
      "%1, %2, %3, [%4], [%5], p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// umma_f8 / umma_mxf8 issued only where `issue` is true (see umma_bf16_if).
__device__ __forceinline__ void umma_f8_if(bool issue, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p, q; setp.ne.b32 p, %4, 0; setp.ne.b32 q, %5, 0;\n"
      " @q tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(static_cast<uint32_t>(issue))
      : "memory");
}
__device__ __forceinline__ void umma_mxf8_if(bool issue, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                             uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p, q; setp.ne.b32 p, %6, 0; setp.ne.b32 q, %7, 0;\n"
      " @q tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p; }" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate),
      "r"(static_cast<uint32_t>(issue))
      : "memory");
}
// Shared memory -> TMEM copy of 32 rows of 16 bytes, written to lanes r,
// r + 32, r + 64 and r + 96 (row r) at 4 consecutive columns.  Issued, like
// the MMAs, by one thread; it executes in order with the MMAs that thread
// issues afterwards.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t s_desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(s_desc) : "memory");
}
// Arrive on *bar once all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// An issuing thread's last step before its CTA leaves: every tcgen05.mma it
// issued has completed (commit to `bar`, fresh at phase 0, and a bounded wait).
__device__ __forceinline__ void umma_drain(uint64_t* bar, uint32_t* status) {
  umma_commit(bar);
  mbar_drain(bar, 0, status);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// tcgen05.wait::ld with the 32 destination registers of an earlier
// tcgen05.ld passed through it: no use of them can be scheduled before the
// wait, which matters when other loads' registers are read in between.
__device__ __forceinline__ void tmem_wait_ld_pin(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 16 consecutive 32-bit columns; thread i of the warp gets lane
// (warp's quarter base + i), columns col .. col+15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 16 lanes x 32 consecutive 32-bit columns spread over all 32 threads (shape
// 16x256b, 4 repetitions): with q = i/4 and c = 2*(i%4), thread i gets, for
// repetition j, r[4j] = (lane q, column 8j+c), r[4j+1] = (q, 8j+c+1),
// r[4j+2] = (q+8, 8j+c), r[4j+3] = (q+8, 8j+c+1), lanes counted from taddr's.
__device__ __forceinline__ void tmem_ld16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%"
      "20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 32 lanes x 64 consecutive columns (two 32-column loads, one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  uint32_t(&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
  uint32_t(&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%"
      "19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format, version 1).
//   start: smem byte address; lbo/sbo: leading/stride byte offsets;
//   layout: 0 none, 2 = 128-byte swizzle, 4 = 64-byte, 6 = 32-byte.
__device__ __forceinline__ uint64_t smem_desc(uint32_t start, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((start >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(layout & 0x7u) << 61;
  return d;
}
constexpr uint32_t kSwizzle128B = 2;

// (d0, d1) = (a0 * b0 + d0, a1 * b1 + d1): two fp32 fmas with round to
// nearest in one packed instruction (fma.rn.f32x2); each lane is exactly
// fmaf(a_i, b_i, d_i).
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n mov.b64 z, {%0, %1};\n"
      " fma.rn.f32x2 z, x, y, z;\n mov.b64 {%0, %1}, z;\n}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Instruction descriptor for kind::f16 with bf16 A/B and an fp32 accumulator.
// a_mn / b_mn select MN-major (1) or K-major (0) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor for kind::mxf8f6f4 with block scales: E4M3 A and B,
// K-major, UE8M0 scales (bit 23), and which byte of the 32-bit scale word the
// MMA uses for A (bits 29-30) and for B (bits 4-5).  Measured placement of
// the scales (M = 128, N = 256): the scale of A-row m is read from TMEM lane
// m, column sfa + m / 32; the scale of B-row n, for the output rows of lane
// quarter q, from lane 32 q + n % 32, column sfb + n / 32.  One
// tcgen05.cp.32x128b.warpx4 of a 128-row block laid out [r][m / 32][byte]
// (16 bytes per r = m % 32) puts every scale where it is read.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int a_sf_id, int b_sf_id) {
  return (static_cast<uint32_t>(b_sf_id) << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24) | (static_cast<uint32_t>(a_sf_id) << 29);
}

// Instruction descriptor for kind::f8f6f4 with E4M3 A and B (format code 0
// for both), K-major operands and an fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Offset of byte `b` (multiple of 16) of row `r` inside a 128-byte-swizzled
// tile whose rows are 128 bytes (TMA CU_TENSOR_MAP_SWIZZLE_128B layout, tile
// base 1024-byte aligned): the 16-byte chunk index is XOR-ed with r % 8.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t b) {
  return r * 128u + ((((b >> 4) ^ r) & 7u) << 4) + (b & 15u);
}

// Order-preserving map fp32 -> uint32 (larger float <=> larger key); -0.0 is
// folded onto +0.0 so that equal values get equal keys.
__device__ __forceinline__ uint32_t f32_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_f32(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

}  // namespace dsa
