// dt_tp_mlp_static_workspace: the TP MLP for callers that cannot allocate
// device memory when they call it.
//
// dt_tp_mlp needs a scratch buffer for H = SiLU(X Wg) * (X Wu) between its
// two GEMMs, and expects the caller to pass one.  Some callers have no way
// to get one at call time: a serving loop that must not allocate once it is
// running (an allocation can block, fragment a fixed memory plan, or fail
// under memory pressure at the worst moment), or host code that does not
// own a device allocator at all and must not mix raw cudaMalloc with the
// pool its framework manages.  For them this entry point keeps H in a
// buffer that is part of the library image itself: a file-scope device
// array.  With CUDA's lazy module loading the array is reserved on a device
// when its address is first looked up there, i.e. by the first call on that
// device, which can therefore fail with an out-of-memory error
// (DT_ERR_CUDA); callers make one call at start-up, before memory is tight
// and before any stream capture.  From then on every GPU that has run the
// entry point holds the array until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "dt_internal.h"

namespace dt {
namespace {

// The library-resident scratch for H.  In host code this name is only a
// host-side handle for the symbol, not a device address: its device address
// is looked up once per device (cudaGetSymbolAddress, with that device
// current) and that address is what the kernels receive.
static __device__ __align__(256) unsigned char g_mlp_static_workspace[DT_TP_MLP_STATIC_WORKSPACE_BYTES];

std::mutex g_mu;
void* g_addr[64] = {};

// Device address of the array on the current device (set up on first use).
dt_status static_workspace_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return fail(DT_ERR_CUDA, "no current CUDA device");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_mlp_static_workspace);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return fail(DT_ERR_CUDA, "cudaGetSymbolAddress of the static workspace: %s", cudaGetErrorString(e));
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return DT_OK;
}

}  // namespace
}  // namespace dt

using namespace dt;

extern "C" dt_status dt_tp_mlp_static_workspace(const dt_dtensor* x, const dt_dtensor* w_gate,
                                                const dt_dtensor* w_up, const dt_dtensor* w_down,
                                                const dt_dtensor* y, int32_t mode, int32_t tp_mesh_dim,
                                                int32_t* d_status, dt_stream_t stream) {
  clear_error();
  size_t need = 0;
  dt_status st = mlp_hidden_bytes(x, w_gate, &need);
  if (st != DT_OK) return st;
  if (need > (size_t)DT_TP_MLP_STATIC_WORKSPACE_BYTES)
    return fail(DT_ERR_CAPACITY,
                "H needs %zu bytes but the library's static workspace holds %d; use dt_tp_mlp with a "
                "caller-owned workspace",
                need, DT_TP_MLP_STATIC_WORKSPACE_BYTES);
  // make the operands' device current before looking up the array there
  if (x && x->nslots > 0 && x->slots) {
    for (int s = 0; s < x->nslots; ++s) {
      if (x->slots[s]) {
        if ((st = bind_device_of(x->slots[s])) != DT_OK) return st;
        break;
      }
    }
  }
  void* ws = nullptr;
  if ((st = static_workspace_address(&ws)) != DT_OK) return st;
  // H is written in full by the gate/up GEMM before the down GEMM reads it,
  // so nothing in the array needs clearing between calls.  Only H's bytes
  // are offered as workspace, so the GEMMs run every tile whole and never
  // use split-tail scratch.
  return dt_tp_mlp(x, w_gate, w_up, w_down, y, mode, tp_mesh_dim, ws, need, d_status, stream);
}
