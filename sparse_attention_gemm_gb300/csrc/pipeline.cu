// pipeline.cu -- one DSA forward step from host buffers, with the copies
// overlapped with the kernels.
//
// The step needs qi, ki, w (1.1 GB at T = 65536) before the indexer starts,
// but the attention inputs q and kv (4.9 GB) only after it ends, and the ids
// are final before attention starts.  Enqueued on two caller streams:
//
//   copy:     H2D cu, qi, ki, w, sink --e_in--> H2D q, kv --e_att-->
//             ... D2H idx, topk_length (after e_sel) ... D2H out/lse chunk c
//             (after e_chunk[c]) ...
//   compute:  (wait e_in) metadata-free fused indexer + top-k --e_sel-->
//             (wait e_att) attention chunk 0 --e_chunk[0]--> chunk 1 ...
//             (wait the copy stream's end)
//
// so the query/KV upload runs under the indexer and each attention chunk's
// output download runs under the next chunk.  Attention chunks are token
// ranges of the same kernel (every row is independent given the full kv).
// Nothing is allocated: inputs, outputs and the workspace are the caller's;
// the events are created once per device and reused under a lock that is
// held while a call enqueues, so calls from several host threads serialise
// their enqueues and each wait binds to its own call's record.
#include <mutex>

#include "common.cuh"

namespace {

constexpr int kMaxChunks = 16;
constexpr int kMaxDevices = 64;

struct DeviceEvents {
  bool ready = false;
  cudaEvent_t in, att, sel, done;
  cudaEvent_t chunk[kMaxChunks];
};

std::mutex g_mutex;
DeviceEvents g_events[kMaxDevices];

int events_for_current_device(DeviceEvents** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return dsa::set_error(DSA_ERR_UNSUPPORTED, "dsa_forward_host: unusable device ordinal");
  }
  DeviceEvents& e = g_events[dev];
  if (!e.ready) {
    cudaEvent_t* all[4 + kMaxChunks] = {&e.in, &e.att, &e.sel, &e.done};
    for (int c = 0; c < kMaxChunks; ++c) all[4 + c] = &e.chunk[c];
    for (cudaEvent_t* p : all)
      if (cudaEventCreateWithFlags(p, cudaEventDisableTiming) != cudaSuccess)
        return dsa::launch_error("dsa_forward_host: event creation");
    e.ready = true;
  }
  *out = &e;
  return DSA_OK;
}

int h2d(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return DSA_OK;
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s) == cudaSuccess
             ? DSA_OK
             : dsa::launch_error("dsa_forward_host: host-to-device copy");
}

int d2h(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return DSA_OK;
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, s) == cudaSuccess
             ? DSA_OK
             : dsa::launch_error("dsa_forward_host: device-to-host copy");
}

}  // namespace

extern "C" int dsa_forward_host(const dsa_forward_buffers* b, int n_docs, int T, int Hi, int d, int k, int s_max,
                                int H, int Dqk, int Dv, float scale, int chunks, cudaStream_t compute,
                                cudaStream_t copy) {
  dsa::clear_error();
  if (!b) return dsa::set_error(DSA_ERR_VALUE, "dsa_forward_host: NULL buffers");
  if (n_docs < 1 || T < 1 || s_max < 1 || s_max > T)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_forward_host: need n_docs >= 1, T >= 1, 1 <= s_max <= T");
  if ((d != 64 && d != 128) || (Hi != 8 && Hi != 16 && Hi != 32 && Hi != 64) || k < 1 || k > DSA_MAX_TOPK)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_forward_host: need d in {64, 128}, Hi in {8, 16, 32, 64}, 1 <= k <= %d",
                          DSA_MAX_TOPK);
  if (!((Dqk == 576 || Dqk == 512) && Dv == 512) || H < 1 || H > 128 || !(scale > 0.f) || !(scale < INFINITY))
    return dsa::set_error(DSA_ERR_VALUE,
                          "dsa_forward_host: need (Dqk, Dv) in {(576, 512), (512, 512)}, 1 <= H <= 128, finite scale > 0");
  if (chunks < 1 || chunks > kMaxChunks || chunks > T)
    return dsa::set_error(DSA_ERR_VALUE, "dsa_forward_host: need 1 <= chunks <= min(%d, T)", kMaxChunks);
  const void* need[] = {b->qi, b->ki, b->w, b->cu_seqlens, b->q, b->kv, b->qi_d, b->ki_d, b->w_d, b->cu_seqlens_d,
                        b->q_d, b->kv_d, b->idx_d, b->topk_length_d, b->out_d, b->lse_d, b->workspace, b->idx,
                        b->topk_length, b->out, b->lse};
  for (const void* p : need)
    if (!p) return dsa::set_error(DSA_ERR_VALUE, "dsa_forward_host: NULL pointer");
  if ((b->sink == nullptr) != (b->sink_d == nullptr))
    return dsa::set_error(DSA_ERR_VALUE, "dsa_forward_host: sink and sink_d must both be given or both be NULL");
  if (!dsa::aligned(b->qi_d, 16) || !dsa::aligned(b->ki_d, 16) || !dsa::aligned(b->q_d, 16) ||
      !dsa::aligned(b->kv_d, 16) || !dsa::aligned(b->out_d, 16))
    return dsa::set_error(DSA_ERR_VALUE, "dsa_forward_host: qi_d, ki_d, q_d, kv_d and out_d must be 16-byte aligned");
  const size_t ws_need = dsa_indexer_topk_workspace_size(T, Hi, d, k, s_max);
  if (ws_need == 0 || b->ws_bytes < ws_need || !dsa::aligned(b->workspace, 256))
    return dsa::set_error(DSA_ERR_WORKSPACE, "dsa_forward_host: workspace needs %zu bytes, 256-byte aligned", ws_need);
  int rc = dsa::check_device(nullptr);
  if (rc != DSA_OK) return rc;

  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceEvents* ev = nullptr;
  rc = events_for_current_device(&ev);
  if (rc != DSA_OK) return rc;
  const size_t t = static_cast<size_t>(T);
  // ---- inputs of the indexer, then (under it) those of attention
  if ((rc = h2d(b->cu_seqlens_d, b->cu_seqlens, (n_docs + 1) * sizeof(int32_t), copy)) != DSA_OK ||
      (rc = h2d(b->qi_d, b->qi, t * Hi * d * 2, copy)) != DSA_OK || (rc = h2d(b->ki_d, b->ki, t * d * 2, copy)) != DSA_OK ||
      (rc = h2d(b->w_d, b->w, t * Hi * sizeof(float), copy)) != DSA_OK)
    return rc;
  if (b->sink && (rc = h2d(b->sink_d, b->sink, H * sizeof(float), copy)) != DSA_OK) return rc;
  if (cudaEventRecord(ev->in, copy) != cudaSuccess) return dsa::launch_error("dsa_forward_host: event record");
  if ((rc = h2d(b->q_d, b->q, t * H * Dqk * 2, copy)) != DSA_OK || (rc = h2d(b->kv_d, b->kv, t * Dqk * 2, copy)) != DSA_OK)
    return rc;
  if (cudaEventRecord(ev->att, copy) != cudaSuccess) return dsa::launch_error("dsa_forward_host: event record");
  // ---- indexer + top-k
  if (cudaStreamWaitEvent(compute, ev->in, 0) != cudaSuccess) return dsa::launch_error("dsa_forward_host: event wait");
  rc = dsa_indexer_topk(b->qi_d, b->ki_d, b->w_d, b->cu_seqlens_d, n_docs, T, Hi, d, k, s_max, b->idx_d,
                        b->topk_length_d, b->workspace, b->ws_bytes, compute);
  if (rc != DSA_OK) return rc;
  if (cudaEventRecord(ev->sel, compute) != cudaSuccess) return dsa::launch_error("dsa_forward_host: event record");
  if (cudaStreamWaitEvent(copy, ev->sel, 0) != cudaSuccess) return dsa::launch_error("dsa_forward_host: event wait");
  if ((rc = d2h(b->idx, b->idx_d, t * k * sizeof(int32_t), copy)) != DSA_OK ||
      (rc = d2h(b->topk_length, b->topk_length_d, t * sizeof(int32_t), copy)) != DSA_OK)
    return rc;
  // ---- attention in token chunks, each chunk's results downloaded under the next
  if (cudaStreamWaitEvent(compute, ev->att, 0) != cudaSuccess) return dsa::launch_error("dsa_forward_host: event wait");
  for (int c = 0; c < chunks; ++c) {
    const size_t t0 = t * c / chunks, t1 = t * (c + 1) / chunks;
    if (t1 == t0) continue;
    const uint8_t* q = static_cast<const uint8_t*>(b->q_d) + t0 * H * Dqk * 2;
    uint8_t* o = static_cast<uint8_t*>(b->out_d) + t0 * H * Dv * 2;
    rc = dsa_sparse_attn_fwd(q, b->kv_d, nullptr, b->idx_d + t0 * k, b->topk_length_d + t0, b->sink_d,
                             static_cast<int>(t1 - t0), T, H, Dqk, Dv, k, scale, o, b->lse_d + t0 * H, nullptr,
                             nullptr, compute);
    if (rc != DSA_OK) return rc;
    if (cudaEventRecord(ev->chunk[c], compute) != cudaSuccess ||
        cudaStreamWaitEvent(copy, ev->chunk[c], 0) != cudaSuccess)
      return dsa::launch_error("dsa_forward_host: event record/wait");
    if ((rc = d2h(static_cast<uint8_t*>(b->out) + t0 * H * Dv * 2, o, (t1 - t0) * H * Dv * 2, copy)) != DSA_OK ||
        (rc = d2h(b->lse + t0 * H, b->lse_d + t0 * H, (t1 - t0) * H * sizeof(float), copy)) != DSA_OK)
      return rc;
  }
  // the compute stream ends after the last download: waiting on it waits for the whole step
  if (cudaEventRecord(ev->done, copy) != cudaSuccess || cudaStreamWaitEvent(compute, ev->done, 0) != cudaSuccess)
    return dsa::launch_error("dsa_forward_host: event record/wait");
  return DSA_OK;
}
