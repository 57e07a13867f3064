// api.cu -- error reporting, device checks, the device status word and the
// tensor-map encoder shared by the entry points of libdsa.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace {

thread_local char g_last_error[512] = "";

// Control block of this library on each device: the status word (OR of
// DSA_STATUS_* bits) and the wait-limit override (0: the default).
__device__ dsa::DeviceControl g_ctl;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int g_dev_checked[kMaxDevices];        // 0 unknown, 1 ok, -1 unsupported
int g_dev_sm_count[kMaxDevices];
uint32_t* g_dev_status[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

}  // namespace

namespace dsa {

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_last_error[0] = '\0'; }

int launch_error(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return DSA_OK;
}

int check_device(int* sm_count) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return set_error(DSA_ERR_UNSUPPORTED, "no usable CUDA device: %s", cudaGetErrorString(e));
  }
  if (dev >= kMaxDevices) return set_error(DSA_ERR_UNSUPPORTED, "device ordinal %d not supported", dev);
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_dev_checked[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) {
      g_dev_checked[dev] = -1;
      g_dev_sm_count[dev] = major * 10 + minor;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_ctl) != cudaSuccess) {
        cudaGetLastError();
        return set_error(DSA_ERR_CUDA, "cannot resolve the device status word");
      }
      g_dev_status[dev] = static_cast<uint32_t*>(p);
      g_dev_sm_count[dev] = sms;
      g_dev_checked[dev] = 1;
    }
  }
  if (g_dev_checked[dev] < 0)
    return set_error(DSA_ERR_UNSUPPORTED, "device %d has compute capability %d.%d; libdsa is built for sm_103a only",
                     dev, g_dev_sm_count[dev] / 10, g_dev_sm_count[dev] % 10);
  if (sm_count) *sm_count = g_dev_sm_count[dev];
  return DSA_OK;
}

uint32_t* device_status_ptr() {
  int dev = 0;
  cudaGetDevice(&dev);
  return g_dev_status[dev];
}

int encode_tensor_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t inner,
                         uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                         CUtensorMapSwizzle swizzle) {
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return set_error(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(DSA_ERR_VALUE, "tensor map encode failed (%d): dims %llu x %llu, row %llu B, box %u x %u",
                     static_cast<int>(r), (unsigned long long)inner, (unsigned long long)outer,
                     (unsigned long long)row_bytes, box_inner, box_outer);
  return DSA_OK;
}

int encode_tensor_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t d0, uint64_t d1,
                         uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
                         uint32_t b2, CUtensorMapSwizzle swizzle) {
  CUtensorMap probe;
  int rc = encode_tensor_map_2d(&probe, base, dtype, d0, d1, stride1_bytes, b0, b1, swizzle);  // loads the encoder
  if (rc != DSA_OK) return rc;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(DSA_ERR_VALUE, "3-D tensor map encode failed (%d): dims %llu x %llu x %llu", static_cast<int>(r),
                     (unsigned long long)d0, (unsigned long long)d1, (unsigned long long)d2);
  return DSA_OK;
}

}  // namespace dsa

extern "C" const char* dsa_last_error(void) { return g_last_error; }

extern "C" int dsa_device_status(uint32_t* flags, int clear) {
  dsa::clear_error();
  if (!flags) return dsa::set_error(DSA_ERR_VALUE, "flags must not be NULL");
  int rc = dsa::check_device(nullptr);
  if (rc != DSA_OK) return rc;
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_ctl, sizeof(v), offsetof(dsa::DeviceControl, status)) != cudaSuccess)
    return dsa::launch_error("dsa_device_status read");
  if (clear) {
    uint32_t z = 0;
    if (cudaMemcpyToSymbol(g_ctl, &z, sizeof(z), offsetof(dsa::DeviceControl, status)) != cudaSuccess)
      return dsa::launch_error("dsa_device_status clear");
  }
  *flags = v;
  return DSA_OK;
}

extern "C" int dsa_set_wait_limit_ns(uint64_t limit_ns) {
  dsa::clear_error();
  int rc = dsa::check_device(nullptr);
  if (rc != DSA_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return dsa::launch_error("dsa_set_wait_limit_ns synchronize");
  if (cudaMemcpyToSymbol(g_ctl, &limit_ns, sizeof(limit_ns), offsetof(dsa::DeviceControl, wait_limit_ns)) !=
      cudaSuccess)
    return dsa::launch_error("dsa_set_wait_limit_ns write");
  if (cudaDeviceSynchronize() != cudaSuccess) return dsa::launch_error("dsa_set_wait_limit_ns synchronize");
  return DSA_OK;
}
