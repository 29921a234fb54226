// Device binding, SM count and the library's own device status word.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "dt_internal.h"
#include "gemm_plan.h"

namespace dt {

// Status word for calls made with d_status == NULL (static device memory:
// nothing is allocated at run time).
__device__ int32_t g_dt_status_word;

dt_status bind_device_of(const void* device_ptr) {
  if (!device_ptr) return DT_OK;
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, device_ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DT_ERR_CUDA, "cudaPointerGetAttributes: %s", cudaGetErrorString(e));
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return fail(DT_ERR_INVALID_ARG, "operand is not device memory");
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != attr.device) {
    e = cudaSetDevice(attr.device);
    if (e != cudaSuccess) return fail(DT_ERR_CUDA, "cudaSetDevice: %s", cudaGetErrorString(e));
  }
  return DT_OK;
}

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

static std::atomic<uint64_t> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int32_t* device_status_word(int32_t* user) {
  if (user) return user;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_dt_status_word) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<int32_t*>(p);
}

bool append_plan_key(std::string* k, const dt_dtensor* d) {
  if (!d) {
    k->push_back('\0');
    return true;
  }
  k->push_back('\1');
  if (d->nslots < 0 || d->nslots > DT_MAX_SLOTS || (d->nslots > 0 && !d->slots)) return false;
  const int nd = d->layout.ndim;
  if (nd < 0 || nd > DT_MAX_TENSOR_DIMS) return false;
  k->append(reinterpret_cast<const char*>(&d->layout), sizeof(d->layout));
  k->append(reinterpret_cast<const char*>(&d->nslots), sizeof(d->nslots));
  if (d->nslots > 0) k->append(reinterpret_cast<const char*>(d->slots), sizeof(void*) * d->nslots);
  const char has = d->strides ? 1 : 0;
  k->push_back(has);
  if (has) k->append(reinterpret_cast<const char*>(d->strides), sizeof(int64_t) * (size_t)d->nslots * nd);
  return true;
}

}  // namespace dt

using namespace dt;

extern "C" uint64_t dt_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" dt_status dt_read_device_status(int32_t* bits, int32_t clear) {
  if (!bits) return fail(DT_ERR_INVALID_ARG, "bits is NULL");
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_dt_status_word, sizeof(int32_t));
  if (e != cudaSuccess) return fail(DT_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  if (clear) {
    int32_t zero = 0;
    e = cudaMemcpyToSymbol(g_dt_status_word, &zero, sizeof(int32_t));
    if (e != cudaSuccess) return fail(DT_ERR_CUDA, "clearing the status word: %s", cudaGetErrorString(e));
  }
  return DT_OK;
}
