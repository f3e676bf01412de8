// Host runtime of libkvpop: status strings, thread-local error detail, the
// per-device status words, tensor-map creation and device queries.
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"

namespace kvpop {

// Four status words per device, in module memory (no allocation).
__device__ int g_device_status[4];

static thread_local char t_last_error[512] = "";

void set_last_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
}

kvpop_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return KVPOP_OK;
  set_last_error("%s: %s", what, cudaGetErrorString(e));
  return KVPOP_ERR_CUDA;
}

int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}

int* device_status_ptr() {
  static int* cache[64] = {nullptr};
  int d = current_device();
  if (d < 0 || d >= 64) return nullptr;
  if (cache[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    cache[d] = static_cast<int*>(p);
  }
  return cache[d];
}

int num_sms() {
  static int cache[64] = {0};
  int d = current_device();
  if (d < 0 || d >= 64) return 148;
  if (cache[d] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    cache[d] = n > 0 ? n : 148;
  }
  return cache[d];
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_tmap_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                  const uint64_t strides_bytes[3], const uint32_t box[4]) {
  auto fn = get_encode_fn();
  if (!fn) {
    set_last_error("cuTensorMapEncodeTiled is not available");
    return false;
  }
  cuuint64_t gdim[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t gstride[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
  cuuint32_t bdim[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gdim, gstride,
                  bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("cuTensorMapEncodeTiled failed (%d)", (int)r);
    return false;
  }
  return true;
}

bool make_tmap_4d_f32(CUtensorMap* map, const void* base, const uint64_t dims[4],
                      const uint64_t strides_bytes[3], const uint32_t box[4]) {
  auto fn = get_encode_fn();
  if (!fn) {
    set_last_error("cuTensorMapEncodeTiled is not available");
    return false;
  }
  cuuint64_t gdim[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t gstride[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
  cuuint32_t bdim[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), gdim, gstride, bdim, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("cuTensorMapEncodeTiled (fp32) failed (%d)", (int)r);
    return false;
  }
  return true;
}

bool make_tmap_rows(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                    uint32_t box_cols) {
  auto fn = get_encode_fn();
  if (!fn) {
    set_last_error("cuTensorMapEncodeTiled is not available");
    return false;
  }
  cuuint64_t gdim[2] = {cols, rows};
  cuuint64_t gstride[1] = {cols * 2};
  cuuint32_t bdim[2] = {box_cols, 1};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, bdim,
                  estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_last_error("cuTensorMapEncodeTiled (rows) failed (%d)", (int)r);
    return false;
  }
  return true;
}

}  // namespace kvpop

extern "C" {

const char* kvpop_status_string(kvpop_status s) {
  switch (s) {
    case KVPOP_OK: return "ok";
    case KVPOP_ERR_INVALID_ARG: return "invalid argument";
    case KVPOP_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVPOP_ERR_CUDA: return "CUDA error";
    case KVPOP_ERR_TIMEOUT: return "device wait timed out";
    case KVPOP_ERR_INTERNAL: return "internal consistency check failed";
  }
  return "unknown status";
}

const char* kvpop_last_error(void) { return kvpop::t_last_error; }

int kvpop_version(void) { return 1; }

kvpop_status kvpop_device_status(int32_t out[4], int reset) {
  if (out == nullptr) {
    kvpop::set_last_error("kvpop_device_status: out is NULL");
    return KVPOP_ERR_INVALID_ARG;
  }
  kvpop_status st = kvpop::cuda_check(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  if (st != KVPOP_OK) return st;
  int* p = kvpop::device_status_ptr();
  if (!p) {
    kvpop::set_last_error("status symbol unavailable");
    return KVPOP_ERR_CUDA;
  }
  int h[4];
  st = kvpop::cuda_check(cudaMemcpy(h, p, sizeof(h), cudaMemcpyDeviceToHost), "read status");
  if (st != KVPOP_OK) return st;
  for (int i = 0; i < 4; ++i) out[i] = h[i];
  if (reset) {
    st = kvpop::cuda_check(cudaMemset(p, 0, sizeof(h)), "reset status");
    if (st != KVPOP_OK) return st;
  }
  return static_cast<kvpop_status>(h[0]);
}

}  // extern "C"
