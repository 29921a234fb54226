// Host layout engine: mesh coordinates, slots and per-slot boxes.
//
// Hyper-Parallel DTensor API (MindSpore hyper-parallel PR 121): a DTensor is
// a local tensor per rank plus a DeviceMesh and one placement per mesh dim;
// _build_layout maps placements to tensor dims.  The distribute_tensor
// example fixes rank order (row-major over the mesh) and the split order.
// Model parallelism (wineandchord), "Tensor-parallel linear layers": shards
// are torch.chunk blocks.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "dt_internal.h"

namespace dt {

static thread_local std::string g_last_error;

dt_status fail(dt_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

void clear_error() { g_last_error.clear(); }

void Layout::rank_coords(int rank, int* coords) const {
  for (int m = mesh_ndim - 1; m >= 0; --m) {
    coords[m] = rank % mesh[m];
    rank /= mesh[m];
  }
}

int Layout::coords_rank(const int* coords) const {
  int r = 0;
  for (int m = 0; m < mesh_ndim; ++m) r = r * mesh[m] + coords[m];
  return r;
}

int Layout::slot_of_coords(const int* coords) const {
  int s = 0;
  for (int i = 0; i < ndistinct; ++i) s = s * mesh[distinct[i]] + coords[distinct[i]];
  return s;
}

void Layout::slot_coords(int slot, int* coords) const {
  for (int m = 0; m < DT_MAX_MESH_DIMS; ++m) coords[m] = 0;
  for (int i = ndistinct - 1; i >= 0; --i) {
    int m = distinct[i];
    coords[m] = slot % mesh[m];
    slot /= mesh[m];
  }
}

Box Layout::box_of_coords(const int* coords) const {
  Box b;
  for (int d = 0; d < DT_MAX_TENSOR_DIMS; ++d) {
    b.off[d] = 0;
    b.size[d] = d < ndim ? gshape[d] : 1;
  }
  // mesh-dim order: an outer mesh dim splits first, an inner one splits its block
  for (int m = 0; m < mesh_ndim; ++m) {
    if (kind[m] != DT_SHARD) continue;
    int d = dim[m];
    int64_t o, s;
    chunk(b.size[d], mesh[m], coords[m], &o, &s);
    b.off[d] += o;
    b.size[d] = s;
  }
  return b;
}

dt_status parse_layout(const dt_layout* in, Layout* out) {
  if (!in) return fail(DT_ERR_INVALID_ARG, "layout is NULL");
  Layout L;
  if (in->mesh_ndim < 1 || in->mesh_ndim > DT_MAX_MESH_DIMS)
    return fail(DT_ERR_INVALID_ARG, "mesh_ndim %d not in [1, %d]", in->mesh_ndim, DT_MAX_MESH_DIMS);
  if (in->ndim < 1 || in->ndim > DT_MAX_TENSOR_DIMS)
    return fail(DT_ERR_INVALID_ARG, "ndim %d not in [1, %d]", in->ndim, DT_MAX_TENSOR_DIMS);
  L.mesh_ndim = in->mesh_ndim;
  L.ndim = in->ndim;
  L.mesh_size = 1;
  for (int m = 0; m < L.mesh_ndim; ++m) {
    if (in->mesh_shape[m] < 1) return fail(DT_ERR_INVALID_ARG, "mesh_shape[%d] = %d", m, in->mesh_shape[m]);
    L.mesh[m] = in->mesh_shape[m];
    L.mesh_size *= L.mesh[m];
  }
  if (L.mesh_size > 4096) return fail(DT_ERR_CAPACITY, "mesh of %d ranks", L.mesh_size);
  for (int d = 0; d < L.ndim; ++d) {
    if (in->gshape[d] < 0) return fail(DT_ERR_INVALID_ARG, "gshape[%d] < 0", d);
    L.gshape[d] = in->gshape[d];
  }
  L.dtype = in->dtype;
  L.esize = dtype_size(in->dtype);
  if (!L.esize) return fail(DT_ERR_INVALID_ARG, "dtype %d", in->dtype);
  L.materialize = in->materialize_replicas != 0;
  for (int m = 0; m < L.mesh_ndim; ++m) {
    const dt_placement& p = in->placements[m];
    L.kind[m] = p.kind;
    if (p.kind == DT_SHARD) {
      int d = p.dim < 0 ? p.dim + L.ndim : p.dim;
      if (d < 0 || d >= L.ndim) return fail(DT_ERR_INVALID_ARG, "Shard(%d) on a rank-%d tensor", p.dim, L.ndim);
      L.dim[m] = d;
    } else if (p.kind == DT_PARTIAL) {
      if (p.op != DT_SUM && p.op != DT_AVG && p.op != DT_MAX)
        return fail(DT_ERR_INVALID_ARG, "Partial reduce op %d", p.op);
      for (int q = 0; q < m; ++q)
        if (L.kind[q] == DT_PARTIAL && L.op[q] != p.op)
          return fail(DT_ERR_UNSUPPORTED, "Partial dims of one layout must share one reduce op");
      L.dim[m] = 0;
      L.op[m] = p.op;
    } else if (p.kind == DT_REPLICATE) {
      L.dim[m] = 0;
    } else {
      return fail(DT_ERR_INVALID_ARG, "placement kind %d on mesh dim %d", p.kind, m);
    }
  }
  L.ndistinct = 0;
  L.nslots = 1;
  for (int m = 0; m < L.mesh_ndim; ++m) {
    if (L.materialize || L.kind[m] != DT_REPLICATE) {
      L.distinct[L.ndistinct++] = m;
      L.nslots *= L.mesh[m];
    }
  }
  if (L.nslots > DT_MAX_SLOTS) return fail(DT_ERR_CAPACITY, "%d slots (max %d)", L.nslots, DT_MAX_SLOTS);
  *out = L;
  return DT_OK;
}

dt_status parse_dtensor(const dt_dtensor* in, DTensor* out, const char* what) {
  if (!in) return fail(DT_ERR_INVALID_ARG, "%s is NULL", what);
  dt_status st = parse_layout(&in->layout, &out->layout);
  if (st != DT_OK) {
    std::string inner = dt_last_error();
    return fail(st, "%s: %s", what, inner.c_str());
  }
  const Layout& L = out->layout;
  if (in->nslots != L.nslots)
    return fail(DT_ERR_INVALID_ARG, "%s: nslots %d but the layout has %d slots", what, in->nslots, L.nslots);
  if (!in->slots) return fail(DT_ERR_INVALID_ARG, "%s: slot array is NULL", what);
  out->slots.assign(L.nslots, SlotView());
  for (int s = 0; s < L.nslots; ++s) {
    SlotView& v = out->slots[s];
    Box b = L.slot_box(s);
    v.numel = 1;
    for (int d = 0; d < DT_MAX_TENSOR_DIMS; ++d) {
      v.shape[d] = d < L.ndim ? b.size[d] : 1;
      v.goff[d] = d < L.ndim ? b.off[d] : 0;
    }
    for (int d = 0; d < L.ndim; ++d) v.numel *= v.shape[d];
    // contiguous row-major unless strides were given
    int64_t st_acc = 1;
    for (int d = L.ndim - 1; d >= 0; --d) {
      v.stride[d] = in->strides ? in->strides[(int64_t)s * L.ndim + d] : st_acc;
      st_acc *= v.shape[d] > 0 ? v.shape[d] : 1;
    }
    for (int d = L.ndim; d < DT_MAX_TENSOR_DIMS; ++d) v.stride[d] = 0;
    v.ptr = static_cast<char*>(in->slots[s]);
    if (v.numel > 0 && !v.ptr) return fail(DT_ERR_INVALID_ARG, "%s: slot %d is NULL", what, s);
    if (v.numel > 0 && (reinterpret_cast<uintptr_t>(v.ptr) % L.esize) != 0)
      return fail(DT_ERR_ALIGNMENT, "%s: slot %d not aligned to its element size", what, s);
    for (int d = 0; d < L.ndim; ++d)
      if (v.stride[d] < 0) return fail(DT_ERR_UNSUPPORTED, "%s: negative stride", what);
  }
  return DT_OK;
}

}  // namespace dt

using namespace dt;

extern "C" {

dt_status dt_layout_nslots(const dt_layout* layout, int32_t* nslots) {
  if (!nslots) return fail(DT_ERR_INVALID_ARG, "nslots is NULL");
  Layout L;
  dt_status st = parse_layout(layout, &L);
  if (st != DT_OK) return st;
  *nslots = L.nslots;
  return DT_OK;
}

dt_status dt_layout_slot_of_rank(const dt_layout* layout, int32_t rank, int32_t* slot) {
  if (!slot) return fail(DT_ERR_INVALID_ARG, "slot is NULL");
  Layout L;
  dt_status st = parse_layout(layout, &L);
  if (st != DT_OK) return st;
  if (rank < 0 || rank >= L.mesh_size) return fail(DT_ERR_INVALID_ARG, "rank %d outside the mesh", rank);
  int c[DT_MAX_MESH_DIMS];
  L.rank_coords(rank, c);
  *slot = L.slot_of_coords(c);
  return DT_OK;
}

dt_status dt_layout_slot_box(const dt_layout* layout, int32_t slot, int64_t* local_shape,
                             int64_t* global_offset) {
  Layout L;
  dt_status st = parse_layout(layout, &L);
  if (st != DT_OK) return st;
  if (slot < 0 || slot >= L.nslots) return fail(DT_ERR_INVALID_ARG, "slot %d of %d", slot, L.nslots);
  Box b = L.slot_box(slot);
  for (int d = 0; d < L.ndim; ++d) {
    if (local_shape) local_shape[d] = b.size[d];
    if (global_offset) global_offset[d] = b.off[d];
  }
  return DT_OK;
}

const char* dt_status_string(dt_status s) {
  switch (s) {
    case DT_OK: return "ok";
    case DT_ERR_INVALID_ARG: return "invalid argument";
    case DT_ERR_SHAPE: return "shape mismatch";
    case DT_ERR_PLACEMENT: return "placement check failed";
    case DT_ERR_UNSUPPORTED: return "unsupported";
    case DT_ERR_ALIGNMENT: return "alignment";
    case DT_ERR_CUDA: return "CUDA error";
    case DT_ERR_CAPACITY: return "capacity exceeded";
  }
  return "unknown status";
}

const char* dt_last_error(void) { return g_last_error.c_str(); }

int32_t dt_version(void) { return 100; }

}  // extern "C"
