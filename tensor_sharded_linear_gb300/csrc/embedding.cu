// EmbeddingWithReplicateOutput: per-shard row gather written straight into
// the Replicate output.
//
// DTorch user guide, "Module parallel", section 2 (tensor parallel): the
// table is Shard(1) on tp (each rank holds every vocabulary row for a slice
// of the embedding dim), token ids are Replicate on tp, and the layer makes
// its output Replicate with an all-gather along the embedding dim.  Here the
// gather and the all-gather are one pass: the warp that reads row id_t of
// shard i writes it at columns [o_i, o_i + d_i) of output row t.
#include <cuda_runtime.h>

#include <algorithm>

#include "dt_internal.h"

namespace dt {
namespace {

constexpr int EMB_THREADS = 256;

struct EmbShard {
  const char* ptr;
  int64_t row_stride;  // elements
  int64_t width;       // elements (d_i)
  int64_t col_off;     // o_i
};

struct EmbOut {
  char* ptr;
  int64_t row_stride;  // elements between consecutive tokens
};

struct EmbParams {
  EmbShard shard[DT_MAX_SLOTS];
  EmbOut out[DT_MAX_SLOTS];
  const int32_t* ids;
  int64_t ntok;
  int64_t vocab;
  int32_t nshard;
  int32_t nout;
  int32_t esize;
  int32_t vec16;  // every row start and width is a multiple of 16 bytes
  int32_t* status;
};

// One warp per (token, shard) row copy, in a grid-stride loop.  The ids of
// a warp's next 32 items are loaded together, one per lane, and handed out
// by shuffle, so a row's loads never wait behind its id's load.  The items
// go two at a time: for 1 KiB rows (16-byte aligned, one output) both rows'
// loads are issued before either row's stores, two rows in flight per warp
// (measured alone: 51.2 -> 49.5 us for the [4, 4096] x 8-shard gather; four
// rows in flight took 51.0).
__device__ __forceinline__ void emb_item(const EmbParams& p, int64_t w, int32_t id, int lane) {
  const int64_t t = w / p.nshard;
  const int i = (int)(w - t * p.nshard);
  const EmbShard& S = p.shard[i];
  const bool ok = id >= 0 && id < p.vocab;
  if (!ok && lane == 0 && i == 0) atomicOr(p.status, DT_DEV_ERR_INDEX);
  const char* src = S.ptr + (int64_t)(ok ? id : 0) * S.row_stride * p.esize;
  const int64_t nbytes = S.width * p.esize;
  for (int o = 0; o < p.nout; ++o) {
    char* dst = p.out[o].ptr + (t * p.out[o].row_stride + S.col_off) * p.esize;
    if (p.vec16) {
      const uint4* sv = reinterpret_cast<const uint4*>(src);
      uint4* dv = reinterpret_cast<uint4*>(dst);
      const int64_t n = nbytes / 16;
      int64_t u = lane;
      for (; u + 32 < n; u += 64) {
        uint4 a = ok ? __ldg(sv + u) : make_uint4(0, 0, 0, 0);
        uint4 b = ok ? __ldg(sv + u + 32) : make_uint4(0, 0, 0, 0);
        __stcs(dv + u, a);
        __stcs(dv + u + 32, b);
      }
      for (; u < n; u += 32) __stcs(dv + u, ok ? __ldg(sv + u) : make_uint4(0, 0, 0, 0));
    } else if (p.esize == 2) {
      const uint16_t* sv = reinterpret_cast<const uint16_t*>(src);
      uint16_t* dv = reinterpret_cast<uint16_t*>(dst);
      for (int64_t e = lane; e < S.width; e += 32) dv[e] = ok ? sv[e] : (uint16_t)0;
    } else {
      const uint32_t* sv = reinterpret_cast<const uint32_t*>(src);
      uint32_t* dv = reinterpret_cast<uint32_t*>(dst);
      for (int64_t e = lane; e < S.width; e += 32) dv[e] = ok ? sv[e] : 0u;
    }
  }
}

__global__ void __launch_bounds__(EMB_THREADS) embedding_kernel(const __grid_constant__ EmbParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (int64_t)blockIdx.x * (EMB_THREADS / 32) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (EMB_THREADS / 32);
  const int64_t pairs = p.ntok * p.nshard;
  for (int64_t w0 = warp_global; w0 < pairs; w0 += 32 * nwarps) {
    // lane k holds the id of item w0 + k * nwarps
    const int64_t mine = w0 + lane * nwarps;
    const int32_t my_id = mine < pairs ? __ldg(p.ids + mine / p.nshard) : 0;
    for (int k = 0; k < 32; k += 2) {
      const int64_t w = w0 + k * nwarps;
      if (w >= pairs) break;  // warp-uniform
      const int64_t w2 = w + nwarps;
      const int32_t id1 = __shfl_sync(0xffffffffu, my_id, k), id2 = __shfl_sync(0xffffffffu, my_id, k + 1);
      if (p.vec16 && p.nout == 1 && w2 < pairs) {
        const int64_t t1 = w / p.nshard, t2 = w2 / p.nshard;
        const int i1 = (int)(w - t1 * p.nshard), i2 = (int)(w2 - t2 * p.nshard);
        const EmbShard& S1 = p.shard[i1];
        const EmbShard& S2 = p.shard[i2];
        const bool ok1 = id1 >= 0 && id1 < p.vocab, ok2 = id2 >= 0 && id2 < p.vocab;
        if (!ok1 && lane == 0 && i1 == 0) atomicOr(p.status, DT_DEV_ERR_INDEX);
        if (!ok2 && lane == 0 && i2 == 0) atomicOr(p.status, DT_DEV_ERR_INDEX);
        const uint4* s1 = reinterpret_cast<const uint4*>(S1.ptr + (int64_t)(ok1 ? id1 : 0) * S1.row_stride * p.esize);
        const uint4* s2 = reinterpret_cast<const uint4*>(S2.ptr + (int64_t)(ok2 ? id2 : 0) * S2.row_stride * p.esize);
        uint4* d1 = reinterpret_cast<uint4*>(p.out[0].ptr + (t1 * p.out[0].row_stride + S1.col_off) * p.esize);
        uint4* d2 = reinterpret_cast<uint4*>(p.out[0].ptr + (t2 * p.out[0].row_stride + S2.col_off) * p.esize);
        const int64_t n1 = S1.width * p.esize / 16, n2 = S2.width * p.esize / 16;
        if (n1 == 64 && n2 == 64) {
          const uint4 z = make_uint4(0, 0, 0, 0);
          const uint4 a1 = ok1 ? __ldg(s1 + lane) : z, b1 = ok1 ? __ldg(s1 + lane + 32) : z;
          const uint4 a2 = ok2 ? __ldg(s2 + lane) : z, b2 = ok2 ? __ldg(s2 + lane + 32) : z;
          __stcs(d1 + lane, a1);
          __stcs(d1 + lane + 32, b1);
          __stcs(d2 + lane, a2);
          __stcs(d2 + lane + 32, b2);
          continue;
        }
      }
      emb_item(p, w, id1, lane);
      if (w2 < pairs) emb_item(p, w2, id2, lane);
    }
  }
}

}  // namespace
}  // namespace dt

using namespace dt;

extern "C" dt_status dt_tp_embedding(const dt_dtensor* ids, const dt_dtensor* table, const dt_dtensor* out,
                                     int32_t tp_mesh_dim, int32_t* d_status, dt_stream_t stream) {
  clear_error();
  DTensor I, T, O;
  dt_status st = parse_dtensor(ids, &I, "ids");
  if (st != DT_OK) return st;
  st = parse_dtensor(table, &T, "table");
  if (st != DT_OK) return st;
  st = parse_dtensor(out, &O, "out");
  if (st != DT_OK) return st;
  const Layout &li = I.layout, &lt = T.layout, &lo = O.layout;
  if (li.dtype != DT_INT32) return fail(DT_ERR_INVALID_ARG, "ids must be int32");
  if (lt.dtype != lo.dtype || lt.dtype == DT_INT32) return fail(DT_ERR_INVALID_ARG, "table/out dtype");
  if (lt.ndim != 2) return fail(DT_ERR_SHAPE, "table must be [vocab, dim]");
  if (lo.ndim != li.ndim + 1) return fail(DT_ERR_SHAPE, "out must have rank ids.ndim + 1");
  if (li.mesh_ndim != lt.mesh_ndim || lo.mesh_ndim != lt.mesh_ndim) return fail(DT_ERR_SHAPE, "meshes differ");
  for (int m = 0; m < lt.mesh_ndim; ++m)
    if (li.mesh[m] != lt.mesh[m] || lo.mesh[m] != lt.mesh[m]) return fail(DT_ERR_SHAPE, "meshes differ");
  if (tp_mesh_dim >= lt.mesh_ndim) return fail(DT_ERR_INVALID_ARG, "tp_mesh_dim %d", tp_mesh_dim);
  for (int m = 0; m < lt.mesh_ndim; ++m) {
    if (m == tp_mesh_dim) {
      if (!lt.is_shard(m, 1)) return fail(DT_ERR_PLACEMENT, "table must be Shard(1) on tp");
    } else if (!lt.is_replicate(m)) {
      return fail(DT_ERR_PLACEMENT, "table must be Replicate off tp");
    }
    if (!li.is_replicate(m)) return fail(DT_ERR_PLACEMENT, "ids must be Replicate");
    if (!lo.is_replicate(m)) return fail(DT_ERR_PLACEMENT, "out must be Replicate");
  }
  for (int d = 0; d < li.ndim; ++d)
    if (lo.gshape[d] != li.gshape[d]) return fail(DT_ERR_SHAPE, "out leading dims must equal ids dims");
  if (lo.gshape[lo.ndim - 1] != lt.gshape[1]) return fail(DT_ERR_SHAPE, "out last dim must be the embedding dim");
  // no tokens or an empty embedding dim: nothing to gather (and the slots'
  // strides, which torch leaves arbitrary on empty dims, are not checked)
  int64_t ntok = 1;
  for (int d = 0; d < li.ndim; ++d) ntok *= li.gshape[d];
  if (ntok == 0 || lt.gshape[1] == 0) return DT_OK;
  // an empty vocabulary has no row to gather for any id: refused here rather
  // than launched on slots without memory
  if (lt.gshape[0] == 0) return fail(DT_ERR_SHAPE, "table has no rows: every id would be out of range");

  // ids: one contiguous slot (replica 0)
  const SlotView& iv = I.slots[0];
  for (int d = 0; d < li.ndim; ++d) {
    int64_t expect = 1;
    for (int e = d + 1; e < li.ndim; ++e) expect *= iv.shape[e];
    if (iv.shape[d] > 1 && iv.stride[d] != expect) return fail(DT_ERR_UNSUPPORTED, "ids must be contiguous");
  }
  static thread_local EmbParams p;
  p.ids = reinterpret_cast<const int32_t*>(iv.ptr);
  p.ntok = iv.numel;
  p.vocab = lt.gshape[0];
  p.esize = lt.esize;
  bool vec = true;
  // the tp shards, in tp order (other mesh dims are Replicate: slots == tp shards,
  // or, with materialised replicas, pick those at coordinate 0)
  const int P = tp_mesh_dim >= 0 ? lt.mesh[tp_mesh_dim] : 1;
  p.nshard = 0;
  for (int j = 0; j < P; ++j) {
    int c[DT_MAX_MESH_DIMS] = {0, 0, 0, 0};
    if (tp_mesh_dim >= 0) c[tp_mesh_dim] = j;
    const SlotView& v = T.slots[lt.slot_of_coords(c)];
    if (v.shape[1] == 0) continue;
    if (v.stride[1] != 1) return fail(DT_ERR_UNSUPPORTED, "table rows must have unit inner stride");
    EmbShard& s = p.shard[p.nshard++];
    s.ptr = v.ptr;
    s.row_stride = v.stride[0];
    s.width = v.shape[1];
    s.col_off = v.goff[1];
    vec = vec && (reinterpret_cast<uintptr_t>(v.ptr) % 16 == 0) && (s.row_stride * p.esize) % 16 == 0 &&
          (s.width * p.esize) % 16 == 0 && (s.col_off * p.esize) % 16 == 0;
  }
  p.nout = 0;
  for (int s = 0; s < lo.nslots; ++s) {
    const SlotView& v = O.slots[s];
    const int nd = lo.ndim;
    if (v.stride[nd - 1] != 1) return fail(DT_ERR_UNSUPPORTED, "out must have unit inner stride");
    // tokens must be evenly spaced (collapsible leading dims)
    int64_t rs = v.stride[nd - 2 >= 0 ? nd - 2 : 0];
    for (int d = nd - 3; d >= 0; --d)
      if (v.shape[d] > 1 && v.stride[d] != v.stride[d + 1] * v.shape[d + 1])
        return fail(DT_ERR_UNSUPPORTED, "out leading dims must be collapsible");
    EmbOut& o = p.out[p.nout++];
    o.ptr = v.ptr;
    o.row_stride = rs;
    vec = vec && (reinterpret_cast<uintptr_t>(v.ptr) % 16 == 0) && (rs * p.esize) % 16 == 0;
  }
  p.vec16 = vec ? 1 : 0;
  if (p.ntok == 0 || p.nshard == 0) return DT_OK;
  st = bind_device_of(p.out[0].ptr);
  if (st != DT_OK) return st;
  p.status = device_status_word(d_status);
  if (!p.status) return fail(DT_ERR_CUDA, "no device status word");
  const int64_t warps_needed = p.ntok * p.nshard;
  const int64_t blocks = std::min<int64_t>((warps_needed + 7) / 8, (int64_t)device_sm_count() * 8);
  embedding_kernel<<<(int)blocks, EMB_THREADS, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(DT_ERR_CUDA, "embedding launch: %s", cudaGetErrorString(e));
  count_launch();
  return DT_OK;
}
