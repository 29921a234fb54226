// redistribute(): placement changes between Shard(d), Replicate and Partial
// on one logical mesh whose slots all live in this GPU's HBM.
//
// Hyper-Parallel DTensor API (MindSpore hyper-parallel PR 121):
//   redistribute     -- build the destination layout, move the data
//                       (AllGather / AllReduce / AllToAll on a real mesh);
//   reduce_partial   -- Partial -> Replicate (AllReduce);
//   full_tensor      -- everything -> Replicate;
//   distribute_tensor-- Replicate -> Shard (slicing).
// nanotron tutorial ch. 5, 5.1: reduce_scatter of the row-parallel output.
//
// On one GPU every collective is a memory-bound pass: the host plans, for
// every destination slot, the boxes it takes from each source slot (the
// intersection of the two slots' global boxes) and, where the source is
// Partial, the list of partial slots to add in rank order.  One kernel then
// streams all boxes: pure copies move bytes untouched (bit-exact for any
// dtype), Partial sums widen bf16 to fp32, add in rank order with
// round-to-nearest adds, and round once to bf16.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "dt_internal.h"

namespace dt {
namespace {

constexpr int RD_MAX_TASKS = 64;
constexpr int RD_MAX_REFS = 256;
constexpr int RD_MAX_SRC = 16;
constexpr int RD_THREADS = 256;
constexpr int RD_WARPS = RD_THREADS / 32;

struct RdSlot {
  char* ptr;
  int64_t stride[4];  // elements; dims padded at the front
};

// One box: `ext` elements per (padded) dim, taken from `nsrc` sources (rank
// order) and written to one destination slot.  nsrc == 0 writes zeros.
struct RdTask {
  int64_t ext[4];
  int64_t dst_off;
  int64_t chunk_begin;
  int32_t dst_slot;
  int32_t nsrc;
  int32_t ref_begin;
  int32_t rows_per_chunk;
};

struct RdRef {
  int64_t off;
  int32_t slot;
  int32_t pad;
};

struct RdParams {
  RdSlot dst[DT_MAX_SLOTS];
  RdSlot src[DT_MAX_SLOTS];
  RdTask task[RD_MAX_TASKS];
  RdRef ref[RD_MAX_REFS];
  int64_t nchunks;
  int32_t ntasks;
  int32_t dtype;
  int32_t esize;
  int32_t pad;
};

// ---------------------------------------------------------------- device

__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) { __stcs(p, v); }

// Byte copy of one row with unit inner strides.  Both ends are moved in the
// widest unit U (16, 8, 4 or the element size) for which source and
// destination share their misalignment; the head up to the first U-aligned
// destination byte and the tail are moved element by element.
template <int U>
__device__ __forceinline__ void copy_body(char* d, const char* s, int64_t nunits, int lane) {
  if constexpr (U == 16) {
    uint4* dv = reinterpret_cast<uint4*>(d);
    const uint4* sv = reinterpret_cast<const uint4*>(s);
    int64_t i = lane;
    for (; i + 96 < nunits; i += 128) {
      uint4 a = ld_stream(sv + i), b = ld_stream(sv + i + 32), c = ld_stream(sv + i + 64), e = ld_stream(sv + i + 96);
      st_stream(dv + i, a);
      st_stream(dv + i + 32, b);
      st_stream(dv + i + 64, c);
      st_stream(dv + i + 96, e);
    }
    for (; i < nunits; i += 32) st_stream(dv + i, ld_stream(sv + i));
  } else {
    using T = typename std::conditional<U == 8, uint2, typename std::conditional<U == 4, uint32_t, uint16_t>::type>::type;
    T* dv = reinterpret_cast<T*>(d);
    const T* sv = reinterpret_cast<const T*>(s);
    int64_t i = lane;
    for (; i + 96 < nunits; i += 128) {
      T a = sv[i], b = sv[i + 32], c = sv[i + 64], e = sv[i + 96];
      dv[i] = a;
      dv[i + 32] = b;
      dv[i + 64] = c;
      dv[i + 96] = e;
    }
    for (; i < nunits; i += 32) dv[i] = sv[i];
  }
}

__device__ __forceinline__ void copy_elems(char* d, const char* s, int64_t n, int esize, int lane) {
  if (esize == 2) {
    for (int64_t i = lane; i < n; i += 32) reinterpret_cast<uint16_t*>(d)[i] = reinterpret_cast<const uint16_t*>(s)[i];
  } else {
    for (int64_t i = lane; i < n; i += 32) reinterpret_cast<uint32_t*>(d)[i] = reinterpret_cast<const uint32_t*>(s)[i];
  }
}

__device__ void copy_row(char* d, const char* s, int64_t n, int esize, int lane) {
  const int64_t nbytes = n * esize;
  const uintptr_t da = reinterpret_cast<uintptr_t>(d), sa = reinterpret_cast<uintptr_t>(s);
  int U = esize;
  if (((da ^ sa) & 15) == 0) U = 16;
  else if (((da ^ sa) & 7) == 0) U = 8;
  else if (((da ^ sa) & 3) == 0) U = 4;
  if (U < esize) U = esize;
  int64_t head = (int64_t)((U - (da % U)) % U);
  if (head > nbytes) head = nbytes;
  const int64_t units = (nbytes - head) / U;
  const int64_t tail = nbytes - head - units * U;
  copy_elems(d, s, head / esize, esize, lane);
  char* db = d + head;
  const char* sb = s + head;
  switch (U) {
    case 16: copy_body<16>(db, sb, units, lane); break;
    case 8: copy_body<8>(db, sb, units, lane); break;
    case 4: copy_body<4>(db, sb, units, lane); break;
    default: copy_body<2>(db, sb, units, lane); break;
  }
  copy_elems(db + units * U, sb + units * U, tail / esize, esize, lane);
}

__device__ void copy_row_strided(char* d, const char* s, int64_t n, int64_t dstr, int64_t sstr, int esize, int lane) {
  if (esize == 2) {
    for (int64_t i = lane; i < n; i += 32)
      reinterpret_cast<uint16_t*>(d)[i * dstr] = reinterpret_cast<const uint16_t*>(s)[i * sstr];
  } else {
    for (int64_t i = lane; i < n; i += 32)
      reinterpret_cast<uint32_t*>(d)[i * dstr] = reinterpret_cast<const uint32_t*>(s)[i * sstr];
  }
}

__device__ void zero_row(char* d, int64_t n, int64_t dstr, int esize, int lane) {
  const uintptr_t da = reinterpret_cast<uintptr_t>(d);
  if (dstr == 1) {
    const int64_t nbytes = n * esize;
    int64_t head = (int64_t)((16 - (da & 15)) & 15);
    if (head > nbytes) head = nbytes;
    const int64_t units = (nbytes - head) / 16;
    const int64_t tail = nbytes - head - units * 16;
    for (int64_t i = lane; i < head / esize; i += 32) {
      if (esize == 2) reinterpret_cast<uint16_t*>(d)[i] = 0;
      else reinterpret_cast<uint32_t*>(d)[i] = 0;
    }
    uint4* dv = reinterpret_cast<uint4*>(d + head);
    for (int64_t i = lane; i < units; i += 32) st_stream(dv + i, make_uint4(0, 0, 0, 0));
    char* t = d + head + units * 16;
    for (int64_t i = lane; i < tail / esize; i += 32) {
      if (esize == 2) reinterpret_cast<uint16_t*>(t)[i] = 0;
      else reinterpret_cast<uint32_t*>(t)[i] = 0;
    }
  } else {
    for (int64_t i = lane; i < n; i += 32) {
      if (esize == 2) reinterpret_cast<uint16_t*>(d)[i * dstr] = 0;
      else reinterpret_cast<uint32_t*>(d)[i * dstr] = 0;
    }
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float to_f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ uint16_t from_f(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// Sum of nsrc partial rows in rank order, fp32 accumulation.  The first value
// is taken as is; the rest are added with round-to-nearest fp32 adds.
__device__ void sum_row(char* d, const char* const* s, int nsrc, int64_t n, int64_t dstr, const int64_t* sstr,
                        int dtype, int lane) {
  bool vec = dstr == 1;
  const uintptr_t da = reinterpret_cast<uintptr_t>(d);
  for (int k = 0; k < nsrc; ++k) {
    vec = vec && sstr[k] == 1 && ((reinterpret_cast<uintptr_t>(s[k]) ^ da) & 15) == 0;
  }
  const int esize = dtype == DT_BF16 ? 2 : 4;
  int64_t head = 0, units = 0;
  if (vec) {
    head = (int64_t)(((16 - (da & 15)) & 15) / esize);
    if (head > n) head = n;
    units = (n - head) * esize / 16;
  }
  const int64_t vec_end = head + units * (16 / esize);
  auto scalar = [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo + lane; i < hi; i += 32) {
      if (dtype == DT_BF16) {
        float acc = to_f(reinterpret_cast<const uint16_t*>(s[0])[i * sstr[0]]);
        for (int k = 1; k < nsrc; ++k)
          acc = __fadd_rn(acc, to_f(reinterpret_cast<const uint16_t*>(s[k])[i * sstr[k]]));
        reinterpret_cast<uint16_t*>(d)[i * dstr] = from_f(acc);
      } else {
        float acc = reinterpret_cast<const float*>(s[0])[i * sstr[0]];
        for (int k = 1; k < nsrc; ++k) acc = __fadd_rn(acc, reinterpret_cast<const float*>(s[k])[i * sstr[k]]);
        reinterpret_cast<float*>(d)[i * dstr] = acc;
      }
    }
  };
  if (!vec) {
    scalar(0, n);
    return;
  }
  scalar(0, head);
  scalar(vec_end, n);
  const int64_t hb = head * esize;
  uint4* dv = reinterpret_cast<uint4*>(d + hb);
  for (int64_t u = lane; u < units; u += 64) {
    const bool two = u + 32 < units;
    float a0[8], a1[8];
    for (int k = 0; k < nsrc; ++k) {
      const uint4* sv = reinterpret_cast<const uint4*>(s[k] + hb);
      uint4 v0 = ld_stream(sv + u);
      uint4 v1 = two ? ld_stream(sv + u + 32) : make_uint4(0, 0, 0, 0);
      if (dtype == DT_BF16) {
        const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
        const uint32_t w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (k == 0) {
            a0[2 * j] = bf16_lo(w0[j]);
            a0[2 * j + 1] = bf16_hi(w0[j]);
            a1[2 * j] = bf16_lo(w1[j]);
            a1[2 * j + 1] = bf16_hi(w1[j]);
          } else {
            a0[2 * j] = __fadd_rn(a0[2 * j], bf16_lo(w0[j]));
            a0[2 * j + 1] = __fadd_rn(a0[2 * j + 1], bf16_hi(w0[j]));
            a1[2 * j] = __fadd_rn(a1[2 * j], bf16_lo(w1[j]));
            a1[2 * j + 1] = __fadd_rn(a1[2 * j + 1], bf16_hi(w1[j]));
          }
        }
      } else {
        const float f0[4] = {__uint_as_float(v0.x), __uint_as_float(v0.y), __uint_as_float(v0.z), __uint_as_float(v0.w)};
        const float f1[4] = {__uint_as_float(v1.x), __uint_as_float(v1.y), __uint_as_float(v1.z), __uint_as_float(v1.w)};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          a0[j] = k == 0 ? f0[j] : __fadd_rn(a0[j], f0[j]);
          a1[j] = k == 0 ? f1[j] : __fadd_rn(a1[j], f1[j]);
        }
      }
    }
    uint4 o0, o1;
    if (dtype == DT_BF16) {
      o0 = make_uint4(pack_bf16x2(a0[0], a0[1]), pack_bf16x2(a0[2], a0[3]), pack_bf16x2(a0[4], a0[5]),
                      pack_bf16x2(a0[6], a0[7]));
      o1 = make_uint4(pack_bf16x2(a1[0], a1[1]), pack_bf16x2(a1[2], a1[3]), pack_bf16x2(a1[4], a1[5]),
                      pack_bf16x2(a1[6], a1[7]));
    } else {
      o0 = make_uint4(__float_as_uint(a0[0]), __float_as_uint(a0[1]), __float_as_uint(a0[2]), __float_as_uint(a0[3]));
      o1 = make_uint4(__float_as_uint(a1[0]), __float_as_uint(a1[1]), __float_as_uint(a1[2]), __float_as_uint(a1[3]));
    }
    st_stream(dv + u, o0);
    if (two) st_stream(dv + u + 32, o1);
  }
}

// SUM = false: every task copies (nsrc <= 1) or zero-fills; SUM = true: every
// task adds nsrc >= 2 partial sources.  One instantiation per kind keeps the
// copy path's register use low.
template <bool SUM>
__global__ void __launch_bounds__(RD_THREADS) rd_kernel(const __grid_constant__ RdParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int esize = p.esize;
  for (int64_t c = blockIdx.x; c < p.nchunks; c += gridDim.x) {
    int t = 0;
    while (t + 1 < p.ntasks && p.task[t + 1].chunk_begin <= c) ++t;
    const RdTask& T = p.task[t];
    const int64_t rows = T.ext[0] * T.ext[1] * T.ext[2];
    const int64_t r0 = (c - T.chunk_begin) * T.rows_per_chunk;
    const int64_t r1 = min(rows, r0 + (int64_t)T.rows_per_chunk);
    const RdSlot& D = p.dst[T.dst_slot];
    for (int64_t r = r0 + warp; r < r1; r += RD_WARPS) {
      const int64_t i2 = r % T.ext[2];
      const int64_t q = r / T.ext[2];
      const int64_t i1 = q % T.ext[1];
      const int64_t i0 = q / T.ext[1];
      char* d = D.ptr + (T.dst_off + i0 * D.stride[0] + i1 * D.stride[1] + i2 * D.stride[2]) * esize;
      const int64_t n = T.ext[3];
      if (!SUM && T.nsrc == 0) {
        zero_row(d, n, D.stride[3], esize, lane);
      } else if (!SUM) {
        const RdRef& R = p.ref[T.ref_begin];
        const RdSlot& S = p.src[R.slot];
        const char* s = S.ptr + (R.off + i0 * S.stride[0] + i1 * S.stride[1] + i2 * S.stride[2]) * esize;
        if (D.stride[3] == 1 && S.stride[3] == 1) copy_row(d, s, n, esize, lane);
        else copy_row_strided(d, s, n, D.stride[3], S.stride[3], esize, lane);
      } else {
        const char* sp[RD_MAX_SRC];
        int64_t ss[RD_MAX_SRC];
        for (int k = 0; k < T.nsrc; ++k) {
          const RdRef& R = p.ref[T.ref_begin + k];
          const RdSlot& S = p.src[R.slot];
          sp[k] = S.ptr + (R.off + i0 * S.stride[0] + i1 * S.stride[1] + i2 * S.stride[2]) * esize;
          ss[k] = S.stride[3];
        }
        sum_row(d, sp, T.nsrc, n, D.stride[3], ss, p.dtype, lane);
      }
    }
  }
}

// ---------------------------------------------------------------- host

struct HostTask {
  Box box;  // global box moved
  int dst_slot;
  std::vector<int> src_slots;  // rank order; empty = zero fill
};

int64_t local_offset(const SlotView& v, const Box& b, int ndim) {
  int64_t off = 0;
  for (int d = 0; d < ndim; ++d) off += (b.off[d] - v.goff[d]) * v.stride[d];
  return off;
}

bool intersect(const Box& a, const Box& b, int ndim, Box* out) {
  for (int d = 0; d < DT_MAX_TENSOR_DIMS; ++d) {
    if (d >= ndim) {
      out->off[d] = 0;
      out->size[d] = 1;
      continue;
    }
    const int64_t lo = std::max(a.off[d], b.off[d]);
    const int64_t hi = std::min(a.off[d] + a.size[d], b.off[d] + b.size[d]);
    if (hi <= lo) return false;
    out->off[d] = lo;
    out->size[d] = hi - lo;
  }
  return true;
}

dt_status plan(const DTensor& S, const DTensor& D, std::vector<HostTask>* tasks) {
  const Layout& ls = S.layout;
  const Layout& ld = D.layout;
  const int nm = ls.mesh_ndim;
  const int nd = ls.ndim;
  bool kept[DT_MAX_MESH_DIMS] = {}, summed[DT_MAX_MESH_DIMS] = {}, zeroed[DT_MAX_MESH_DIMS] = {};
  for (int m = 0; m < nm; ++m) {
    if (ld.is_partial(m)) {
      if (ls.is_partial(m)) kept[m] = true;
      else if (ls.is_replicate(m)) zeroed[m] = true;
      else return fail(DT_ERR_UNSUPPORTED, "Shard -> Partial on mesh dim %d is not defined", m);
    } else if (ls.is_partial(m)) {
      summed[m] = true;
    }
  }
  if (ls.dtype == DT_INT32) {
    for (int m = 0; m < nm; ++m)
      if (summed[m]) return fail(DT_ERR_UNSUPPORTED, "Partial sums of int32 tensors");
  }
  int nsum = 1;
  for (int m = 0; m < nm; ++m)
    if (summed[m]) nsum *= ls.mesh[m];
  if (nsum > RD_MAX_SRC) return fail(DT_ERR_CAPACITY, "%d partial sources per element (max %d)", nsum, RD_MAX_SRC);

  int shard_dims[DT_MAX_MESH_DIMS], nshard = 0;
  for (int m = 0; m < nm; ++m)
    if (ls.kind[m] == DT_SHARD) shard_dims[nshard++] = m;
  int nshard_combos = 1;
  for (int i = 0; i < nshard; ++i) nshard_combos *= ls.mesh[shard_dims[i]];
  int sum_dims[DT_MAX_MESH_DIMS], nsd = 0;
  for (int m = 0; m < nm; ++m)
    if (summed[m]) sum_dims[nsd++] = m;

  for (int ds = 0; ds < ld.nslots; ++ds) {
    int cd[DT_MAX_MESH_DIMS];
    ld.slot_coords(ds, cd);
    const Box bd = ld.box_of_coords(cd);
    if (bd.numel(nd) == 0) continue;
    bool zero = false;
    for (int m = 0; m < nm; ++m)
      if (zeroed[m] && cd[m] != 0) zero = true;
    if (zero) {
      tasks->push_back(HostTask{bd, ds, {}});
      continue;
    }
    for (int sc = 0; sc < nshard_combos; ++sc) {
      int cs[DT_MAX_MESH_DIMS] = {0, 0, 0, 0};
      // kept Partial dims follow the destination; materialised source
      // replicas are read at Replicate coordinate 0
      for (int m = 0; m < nm; ++m)
        if (kept[m]) cs[m] = cd[m];
      int rem = sc;
      for (int i = nshard - 1; i >= 0; --i) {
        const int m = shard_dims[i];
        cs[m] = rem % ls.mesh[m];
        rem /= ls.mesh[m];
      }
      const Box bs = ls.box_of_coords(cs);
      Box inter;
      if (!intersect(bd, bs, nd, &inter)) continue;
      HostTask t{inter, ds, {}};
      for (int pc = 0; pc < nsum; ++pc) {  // row-major over the summed mesh dims
        int r = pc;
        for (int i = nsd - 1; i >= 0; --i) {
          cs[sum_dims[i]] = r % ls.mesh[sum_dims[i]];
          r /= ls.mesh[sum_dims[i]];
        }
        t.src_slots.push_back(ls.slot_of_coords(cs));
      }
      tasks->push_back(std::move(t));
    }
  }
  return DT_OK;
}

void fill_slot(RdSlot* out, const SlotView& v, int ndim) {
  out->ptr = v.ptr;
  // pad dims at the front so the innermost tensor dim is padded dim 3
  const int pad = 4 - ndim;
  for (int d = 0; d < 4; ++d) out->stride[d] = d < pad ? 0 : v.stride[d - pad];
}

}  // namespace
}  // namespace dt

using namespace dt;

extern "C" dt_status dt_redistribute(const dt_dtensor* src, const dt_dtensor* dst, int32_t* d_status,
                                     dt_stream_t stream) {
  clear_error();
  (void)d_status;  // data movement reports no device-side errors
  DTensor S, D;
  dt_status st = parse_dtensor(src, &S, "src");
  if (st != DT_OK) return st;
  st = parse_dtensor(dst, &D, "dst");
  if (st != DT_OK) return st;
  const Layout& ls = S.layout;
  const Layout& ld = D.layout;
  if (ls.mesh_ndim != ld.mesh_ndim) return fail(DT_ERR_SHAPE, "src and dst meshes differ");
  for (int m = 0; m < ls.mesh_ndim; ++m)
    if (ls.mesh[m] != ld.mesh[m]) return fail(DT_ERR_SHAPE, "src and dst meshes differ");
  if (ls.ndim != ld.ndim) return fail(DT_ERR_SHAPE, "src and dst ranks differ");
  for (int d = 0; d < ls.ndim; ++d)
    if (ls.gshape[d] != ld.gshape[d]) return fail(DT_ERR_SHAPE, "global shapes differ on dim %d", d);
  if (ls.dtype != ld.dtype) return fail(DT_ERR_INVALID_ARG, "src and dst dtypes differ");

  std::vector<HostTask> tasks;
  st = plan(S, D, &tasks);
  if (st != DT_OK) return st;
  if (tasks.empty()) return DT_OK;
  // a plan either sums (every non-zero-fill task has the same >= 2 sources)
  // or copies; zero-fill tasks of a summing plan go to a copy launch
  std::vector<HostTask> sums, copies;
  for (auto& t : tasks) (t.src_slots.size() >= 2 ? sums : copies).push_back(std::move(t));

  const void* any = nullptr;
  for (auto& v : D.slots)
    if (v.numel) { any = v.ptr; break; }
  st = bind_device_of(any);
  if (st != DT_OK) return st;

  const int nd = ls.ndim;
  const int pad = 4 - nd;
  static thread_local RdParams p;  // ~13 KB: keep it off the stack
  for (int s = 0; s < ld.nslots; ++s) fill_slot(&p.dst[s], D.slots[s], nd);
  for (int s = 0; s < ls.nslots; ++s) fill_slot(&p.src[s], S.slots[s], nd);
  p.dtype = ls.dtype;
  p.esize = ls.esize;
  const int grid_cap = device_sm_count() * 8;

  auto launch_all = [&](const std::vector<HostTask>& tasks, bool sum) -> dt_status {
  size_t i = 0;
  while (i < tasks.size()) {
    int nt = 0, nref = 0;
    int64_t chunks = 0;
    for (; i < tasks.size() && nt < RD_MAX_TASKS; ++i) {
      const HostTask& ht = tasks[i];
      if (nref + (int)ht.src_slots.size() > RD_MAX_REFS) break;
      RdTask& t = p.task[nt];
      for (int d = 0; d < 4; ++d) t.ext[d] = d < pad ? 1 : ht.box.size[d - pad];
      t.dst_slot = ht.dst_slot;
      t.dst_off = local_offset(D.slots[ht.dst_slot], ht.box, nd);
      t.nsrc = (int)ht.src_slots.size();
      t.ref_begin = nref;
      for (int k = 0; k < t.nsrc; ++k) {
        p.ref[nref].slot = ht.src_slots[k];
        p.ref[nref].off = local_offset(S.slots[ht.src_slots[k]], ht.box, nd);
        ++nref;
      }
      const int64_t row_bytes = std::max<int64_t>(1, t.ext[3] * ls.esize);
      const int64_t rows = t.ext[0] * t.ext[1] * t.ext[2];
      int64_t rpc = std::max<int64_t>(1, (32 * 1024) / row_bytes);
      rpc = std::min<int64_t>(rpc, 1 << 20);
      t.rows_per_chunk = (int32_t)rpc;
      t.chunk_begin = chunks;
      chunks += (rows + rpc - 1) / rpc;
      ++nt;
    }
    p.ntasks = nt;
    p.nchunks = chunks;
    const int grid = (int)std::min<int64_t>(chunks, grid_cap);
    if (sum)
      rd_kernel<true><<<grid, RD_THREADS, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    else
      rd_kernel<false><<<grid, RD_THREADS, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(DT_ERR_CUDA, "redistribute launch: %s", cudaGetErrorString(e));
    count_launch();
  }
  return DT_OK;
  };
  if ((st = launch_all(copies, false)) != DT_OK) return st;
  if ((st = launch_all(sums, true)) != DT_OK) return st;
  return DT_OK;
}
