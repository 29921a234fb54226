// Internal host-side declarations of libdt: the layout engine and helpers
// shared by the entry points.  Not part of the ABI.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/dt.h"

namespace dt {

// Thread-local error message behind dt_last_error().
dt_status fail(dt_status s, const char* fmt, ...);
void clear_error();

inline int dtype_size(int dtype) {
  switch (dtype) {
    case DT_BF16: return 2;
    case DT_FP32: return 4;
    case DT_INT32: return 4;
    default: return 0;
  }
}

// torch.chunk-style block j of [0, n) split into p parts: width ceil(n/p),
// trailing blocks short or empty.
inline void chunk(int64_t n, int64_t p, int64_t j, int64_t* off, int64_t* size) {
  int64_t c = n > 0 ? (n + p - 1) / p : 0;
  int64_t start = j * c < n ? j * c : n;
  int64_t s = n - j * c;
  if (s > c) s = c;
  if (s < 0) s = 0;
  *off = start;
  *size = s;
}

struct Box {
  int64_t off[DT_MAX_TENSOR_DIMS];
  int64_t size[DT_MAX_TENSOR_DIMS];
  int64_t numel(int ndim) const {
    int64_t n = 1;
    for (int d = 0; d < ndim; ++d) n *= size[d];
    return n;
  }
};

// Normalised, validated copy of a dt_layout.
struct Layout {
  int mesh_ndim = 0;
  int mesh[DT_MAX_MESH_DIMS] = {1, 1, 1, 1};
  int mesh_size = 1;
  int kind[DT_MAX_MESH_DIMS] = {0, 0, 0, 0};
  int dim[DT_MAX_MESH_DIMS] = {0, 0, 0, 0};  // normalised shard dim
  int op[DT_MAX_MESH_DIMS] = {0, 0, 0, 0};   // dt_reduce_op of a Partial dim
  int partial_op() const {                     // the layout's one reduce op (SUM if none)
    for (int m = 0; m < mesh_ndim; ++m)
      if (kind[m] == DT_PARTIAL) return op[m];
    return DT_SUM;
  }
  int ndim = 0;
  int64_t gshape[DT_MAX_TENSOR_DIMS] = {1, 1, 1, 1};
  int dtype = 0;
  int esize = 0;
  bool materialize = false;
  int distinct[DT_MAX_MESH_DIMS];  // mesh dims that select different stored data
  int ndistinct = 0;
  int nslots = 1;

  void rank_coords(int rank, int* coords) const;
  int coords_rank(const int* coords) const;
  int slot_of_coords(const int* coords) const;
  void slot_coords(int slot, int* coords) const;  // 0 on shared (Replicate) dims
  Box box_of_coords(const int* coords) const;
  Box slot_box(int slot) const {
    int c[DT_MAX_MESH_DIMS];
    slot_coords(slot, c);
    return box_of_coords(c);
  }
  bool is_partial(int m) const { return kind[m] == DT_PARTIAL; }
  bool is_replicate(int m) const { return kind[m] == DT_REPLICATE; }
  bool is_shard(int m, int d) const { return kind[m] == DT_SHARD && dim[m] == d; }
};

dt_status parse_layout(const dt_layout* in, Layout* out);

// One slot of a dt_dtensor as the kernels see it.
struct SlotView {
  char* ptr = nullptr;
  int64_t shape[DT_MAX_TENSOR_DIMS] = {1, 1, 1, 1};
  int64_t stride[DT_MAX_TENSOR_DIMS] = {0, 0, 0, 0};  // elements
  int64_t goff[DT_MAX_TENSOR_DIMS] = {0, 0, 0, 0};    // global offset of element 0
  int64_t numel = 0;
};

struct DTensor {
  Layout layout;
  std::vector<SlotView> slots;
};

// Parse + validate a dt_dtensor: slot count, non-null non-empty slots,
// stride array.  `what` names the operand in error messages.
dt_status parse_dtensor(const dt_dtensor* in, DTensor* out, const char* what);

// Device/stream helpers (implemented in common.cu).
dt_status bind_device_of(const void* device_ptr);
int device_sm_count();
int32_t* device_status_word(int32_t* user);  // user if non-null, else the library word
void count_launch();
void clear_redistribute_plans();  // drop the redistribute plan cache (dt_clear_cache)
void clear_gemm_plans();          // drop the linears' plan cache (dt_clear_cache)

// Bytes of the TP MLP's H blocks for these operands (the least workspace
// dt_tp_mlp accepts; its split tail's scratch would come on top).
dt_status mlp_hidden_bytes(const dt_dtensor* x, const dt_dtensor* w_gate, size_t* bytes);

// Append the bytes that decide a launch plan for descriptor d (its layout,
// slot pointers and strides; a marker for NULL) to a cache key.  false: a
// malformed descriptor, left to the planning path's checks.
bool append_plan_key(std::string* key, const dt_dtensor* d);
template <class T>
void append_plan_scalar(std::string* key, const T& v) {
  key->append(reinterpret_cast<const char*>(&v), sizeof(T));
}

}  // namespace dt
