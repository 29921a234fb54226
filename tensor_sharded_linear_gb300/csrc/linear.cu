// Tensor-parallel linear entry points: placement checks and the lowering of
// every rank's local product to GEMM groups.
//
// DTorch user guide, "Module parallel", section 3: tp_shard_type "col" keeps
// the weight sharded on output features and requires a Replicate input on
// tp; "row" shards the weight on input features and requires a
// Shard(ndim - 1) input; the row bias is Partial so it is added once; every
// mesh dim other than tp keeps weights and biases Replicate.
// Model parallelism (wineandchord), "Tensor Parallel": Y_i = X W_i and
// Y = sum_i X_i W_i, weights [in, out].
// nanotron tutorial ch. 5, 5.1: ALL_REDUCE / REDUCE_SCATTER row outputs.
#include <algorithm>
#include <cstring>
#include <memory>
#include <mutex>
#include <set>
#include <string>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "gemm_plan.h"

namespace dt {
namespace {

using gemm::HostGroup;
using gemm::HostSeg;
using gemm::Mat;

// A [K, N] weight slot: row-major ([in, out] storage), or a transposed view
// of [N, K] storage (unit stride along K: the [out, in] convention of
// nn.Linear), which the GEMM reads as a K-major B operand.
dt_status weight_matrix(const SlotView& v, int dtype, Mat* out, const char* what);

// Matrix view of a slot: leading dims flattened to rows, last dim = cols.
dt_status slot_matrix(const SlotView& v, int ndim, int dtype, Mat* out, const char* what) {
  Mat m;
  m.ptr = v.ptr;
  m.dtype = dtype;
  m.cols = v.shape[ndim - 1];
  m.rows = 1;
  for (int d = 0; d < ndim - 1; ++d) m.rows *= v.shape[d];
  if (m.rows == 0 || m.cols == 0) {  // no elements: strides mean nothing (torch leaves them arbitrary)
    m.ld = m.cols;
    *out = m;
    return DT_OK;
  }
  if (m.cols > 1 && v.stride[ndim - 1] != 1) return fail(DT_ERR_UNSUPPORTED, "%s: inner stride must be 1", what);
  if (ndim >= 2) {
    m.ld = v.stride[ndim - 2];
    for (int d = ndim - 3; d >= 0; --d)
      if (v.shape[d] > 1 && v.stride[d] != v.stride[d + 1] * v.shape[d + 1])
        return fail(DT_ERR_UNSUPPORTED, "%s: leading dims must be collapsible", what);
    if (m.rows <= 1) m.ld = std::max<int64_t>(m.ld, m.cols);
  } else {
    m.ld = m.cols;
  }
  if (m.rows > 1 && m.ld < m.cols) return fail(DT_ERR_UNSUPPORTED, "%s: rows overlap", what);
  *out = m;
  return DT_OK;
}

dt_status weight_matrix(const SlotView& v, int dtype, Mat* out, const char* what) {
  const int64_t K = v.shape[0], N = v.shape[1];
  if (N > 1 && K > 1 && v.stride[1] != 1 && v.stride[0] == 1) {
    if (v.stride[1] < K) return fail(DT_ERR_UNSUPPORTED, "%s: columns overlap", what);
    Mat m;
    m.ptr = v.ptr;
    m.dtype = dtype;
    m.rows = K;
    m.cols = N;
    m.ld = v.stride[1];
    m.kmajor = true;
    *out = m;
    return DT_OK;
  }
  return slot_matrix(v, 2, dtype, out, what);
}

bool same_mesh(const Layout& a, const Layout& b) {
  if (a.mesh_ndim != b.mesh_ndim) return false;
  for (int m = 0; m < a.mesh_ndim; ++m)
    if (a.mesh[m] != b.mesh[m]) return false;
  return true;
}

bool same_placement(const Layout& a, int ma, const Layout& b, int mb) {
  if (a.kind[ma] != b.kind[mb]) return false;
  return a.kind[ma] != DT_SHARD || a.dim[ma] == b.dim[mb];
}

const char* pname(const Layout& l, int m) {
  switch (l.kind[m]) {
    case DT_REPLICATE: return "Replicate";
    case DT_SHARD: return "Shard";
    default: return "Partial";
  }
}

dt_status check_tp(int tp, const Layout& l) {
  if (tp >= l.mesh_ndim) return fail(DT_ERR_INVALID_ARG, "tp_mesh_dim %d outside a %d-D mesh", tp, l.mesh_ndim);
  return DT_OK;
}

int tp_size(const Layout& l, int tp) { return tp >= 0 ? l.mesh[tp] : 1; }

// Rows of the first local dim, scaled to flattened rows.
int64_t rows_per_dim0(const SlotView& v, int ndim) {
  int64_t r = 1;
  for (int d = 1; d < ndim - 1; ++d) r *= v.shape[d];
  return r;
}

struct ColumnSpec {
  const DTensor* w;
  const DTensor* bias;  // nullptr: none
  const DTensor* y;
};

// The GEMM kernels keep M, N and their TMA and tile coordinates in 32 bits:
// a dimension that would not fit is refused before anything touches the
// device (an [8, 2^31] bf16 activation is only 32 GB).
constexpr int64_t GEMM_DIM_LIMIT = (1ll << 31) - 512;
// The first output of a group that writes anything, or nullptr when none
// does (no tokens, or no output columns): the device the call binds to.
// A REDUCE_SCATTER group over no rows has no output blocks at all.
const void* first_output(const std::vector<HostGroup>& groups) {
  for (const auto& g : groups)
    if (g.m > 0 && g.n > 0 && !g.out_ptr.empty()) return g.out_ptr[0];
  return nullptr;
}

dt_status check_gemm_dims(const Layout& lx, int64_t k, int64_t n) {
  int64_t m = 1;
  for (int d = 0; d + 1 < lx.ndim; ++d) m *= lx.gshape[d];
  if (m > GEMM_DIM_LIMIT || k > GEMM_DIM_LIMIT || n > GEMM_DIM_LIMIT)
    return fail(DT_ERR_CAPACITY, "GEMM of M=%lld, K=%lld, N=%lld: each must be below 2^31 - 512", (long long)m,
                (long long)k, (long long)n);
  return DT_OK;
}

// Checks shared by the column layers: x [.., K] Replicate on tp, w [K, N]
// Shard(1) on tp, bias [N] Shard(0) on tp, y [.., N] Shard(-1) on tp; off tp
// weights/bias Replicate and x, y placed alike.
dt_status check_column(const DTensor& X, const ColumnSpec& c, int tp, bool allow_partial_x) {
  const Layout& lx = X.layout;
  const Layout& lw = c.w->layout;
  const Layout& ly = c.y->layout;
  if (!same_mesh(lx, lw) || !same_mesh(lx, ly) || (c.bias && !same_mesh(lx, c.bias->layout)))
    return fail(DT_ERR_SHAPE, "operands live on different meshes");
  if (lw.ndim != 2) return fail(DT_ERR_SHAPE, "weight must be 2-D [in, out]");
  if (lx.dtype != lw.dtype) return fail(DT_ERR_INVALID_ARG, "x and w dtypes differ");
  if (lx.dtype == DT_INT32 || ly.dtype == DT_INT32) return fail(DT_ERR_INVALID_ARG, "int32 linear");
  if (ly.ndim != lx.ndim) return fail(DT_ERR_SHAPE, "y rank must equal x rank");
  const int nd = lx.ndim;
  if (lx.gshape[nd - 1] != lw.gshape[0]) return fail(DT_ERR_SHAPE, "x last dim %lld != w rows %lld",
                                                     (long long)lx.gshape[nd - 1], (long long)lw.gshape[0]);
  for (int d = 0; d < nd - 1; ++d)
    if (ly.gshape[d] != lx.gshape[d]) return fail(DT_ERR_SHAPE, "y leading dims differ from x");
  if (ly.gshape[nd - 1] != lw.gshape[1]) return fail(DT_ERR_SHAPE, "y last dim != w cols");
  if (dt_status st = check_gemm_dims(lx, lw.gshape[0], lw.gshape[1]); st != DT_OK) return st;
  if (c.bias) {
    const Layout& lb = c.bias->layout;
    if (lb.ndim != 1 || lb.gshape[0] != lw.gshape[1]) return fail(DT_ERR_SHAPE, "bias must be [out]");
    if (lb.dtype == DT_INT32) return fail(DT_ERR_INVALID_ARG, "bias dtype");
  }
  for (int m = 0; m < lx.mesh_ndim; ++m) {
    if (m == tp) {
      // input: Replicate (DTorch's rule), or sharded on a leading (token) dim:
      // the sequence-parallel entry, whose all-gather is read in place
      const bool x_rep = lx.is_replicate(m);
      const bool x_seq = lx.kind[m] == DT_SHARD && lx.dim[m] < nd - 1;
      if (!x_rep && !x_seq)
        return fail(DT_ERR_PLACEMENT, "column-parallel input must be Replicate (or token-sharded) on tp, got %s%s",
                    pname(lx, m), lx.kind[m] == DT_SHARD && lx.dim[m] == nd - 1 ? "(-1)" : "");
      if (!lw.is_shard(m, 1)) return fail(DT_ERR_PLACEMENT, "column-parallel weight [in, out] must be Shard(1) on tp");
      // output: Shard(-1) (ColumnParallelLinear) or Replicate (the
      // ...WithReplicateOutput layers: each shard writes its column block)
      if (!ly.is_shard(m, nd - 1) && !ly.is_replicate(m))
        return fail(DT_ERR_PLACEMENT, "column-parallel output must be Shard(-1) or Replicate on tp");
      if (c.bias && !c.bias->layout.is_shard(m, 0)) return fail(DT_ERR_PLACEMENT, "column-parallel bias must be Shard(0) on tp");
    } else {
      if (!lw.is_replicate(m)) return fail(DT_ERR_PLACEMENT, "weight must be Replicate off tp");
      if (c.bias && !c.bias->layout.is_replicate(m)) return fail(DT_ERR_PLACEMENT, "bias must be Replicate off tp");
      if (!same_placement(lx, m, ly, m)) return fail(DT_ERR_PLACEMENT, "x and y must be placed alike off tp");
      if (lx.kind[m] == DT_SHARD && lx.dim[m] == nd - 1) return fail(DT_ERR_PLACEMENT, "x may not be sharded on its last dim off tp");
      if (lx.is_partial(m) && (!allow_partial_x || c.bias)) return fail(DT_ERR_PLACEMENT, "Partial input with a bias");
    }
  }
  return DT_OK;
}

dt_status add_column_groups(const DTensor& X, const ColumnSpec& c, int tp, std::vector<HostGroup>* groups,
                            std::set<std::tuple<const void*, int, int, int>>* done) {
  const Layout& lx = X.layout;
  const Layout& ly = c.y->layout;
  const int nd = lx.ndim;
  const bool x_seq = tp >= 0 && lx.kind[tp] == DT_SHARD;        // token-sharded input
  const bool y_rep = tp >= 0 && ly.is_replicate(tp);             // Replicate output
  const int P = tp >= 0 ? lx.mesh[tp] : 1;
  int coords[DT_MAX_MESH_DIMS], cj[DT_MAX_MESH_DIMS];
  for (int r = 0; r < lx.mesh_size; ++r) {
    lx.rank_coords(r, coords);
    const int ys = ly.slot_of_coords(coords);
    const int ws = c.w->layout.slot_of_coords(coords);
    const SlotView& wv = c.w->slots[ws];
    const SlotView& yv = c.y->slots[ys];
    Mat b, y;
    dt_status st = weight_matrix(wv, c.w->layout.dtype, &b, "w");
    if (st != DT_OK) return st;
    st = slot_matrix(yv, nd, ly.dtype, &y, "y");
    if (st != DT_OK) return st;
    // the weight shard's columns inside y: all of y (Shard(-1) output) or
    // its column block of the Replicate output
    const int64_t col0 = y_rep ? wv.goff[1] : 0;
    if (y_rep) {
      if (col0 + b.cols > y.cols) return fail(DT_ERR_SHAPE, "weight shard columns exceed the output");
    } else if (y.cols != b.cols) {
      return fail(DT_ERR_SHAPE, "output shard width %lld != weight shard width %lld", (long long)y.cols, (long long)b.cols);
    }
    // the x slots feeding this output: one (Replicate on tp) or the P token
    // shards, each writing its own block of rows
    const int nx = x_seq ? P : 1;
    for (int j = 0; j < nx; ++j) {
      std::copy(coords, coords + DT_MAX_MESH_DIMS, cj);
      if (x_seq) cj[tp] = j;
      const int xs = lx.slot_of_coords(cj);
      if (!done->insert(std::make_tuple((const void*)c.y, ys, ws, xs)).second) continue;
      const SlotView& xv = X.slots[xs];
      Mat a;
      if ((st = slot_matrix(xv, nd, lx.dtype, &a, "x")) != DT_OK) return st;
      if (a.cols != b.rows) return fail(DT_ERR_SHAPE, "x width %lld != w rows %lld", (long long)a.cols, (long long)b.rows);
      if (a.rows == 0) continue;
      int64_t row0 = 0;
      if (x_seq) {
        // x slot j holds dim-0 entries [goff, goff + n) of the y slot's, i.e.
        // a contiguous block of the flattened rows
        if (lx.dim[tp] != 0) return fail(DT_ERR_UNSUPPORTED, "a token-sharded input must be sharded on dim 0");
        int64_t inner = 1;
        for (int e = 1; e < nd - 1; ++e) inner *= xv.shape[e];
        row0 = (xv.goff[0] - yv.goff[0]) * inner;
        if (row0 < 0 || row0 + a.rows > y.rows) return fail(DT_ERR_SHAPE, "token shard rows outside the output");
      } else if (y.rows != a.rows) {
        return fail(DT_ERR_SHAPE, "x rows %lld != y rows %lld", (long long)a.rows, (long long)y.rows);
      }
      HostGroup g;
      g.m = a.rows;
      g.n = b.cols;
      g.m_block = x_seq ? j : 0;
      g.segs.push_back(HostSeg{a, b, Mat()});
      g.out_dtype = ly.dtype;
      const int esize = dtype_size(ly.dtype);
      g.row_begin = {0};
      g.out_ptr = {y.ptr + (row0 * y.ld + col0) * esize};
      g.out_ld = {y.ld};
      if (c.bias) {
        const SlotView& bv = c.bias->slots[c.bias->layout.slot_of_coords(coords)];
        if (bv.shape[0] != b.cols) return fail(DT_ERR_SHAPE, "bias shard width differs from the weight shard");
        if (bv.shape[0] > 1 && bv.stride[0] != 1) return fail(DT_ERR_UNSUPPORTED, "bias must be contiguous");
        g.bias = bv.ptr;
        g.bias_dtype = c.bias->layout.dtype;
      }
      groups->push_back(std::move(g));
    }
  }
  return DT_OK;
}

// Parse and check a (multi-)column call and lower every shard's product
// to GEMM groups.
dt_status column_build(const dt_dtensor* x, int32_t n, const dt_dtensor* w, const dt_dtensor* bias,
                       const dt_dtensor* y, int32_t tp, std::vector<HostGroup>* groups) {
  if (n < 1 || !w || !y) return fail(DT_ERR_INVALID_ARG, "need n >= 1 weights and outputs");
  DTensor X;
  dt_status st = parse_dtensor(x, &X, "x");
  if (st != DT_OK) return st;
  st = check_tp(tp, X.layout);
  if (st != DT_OK) return st;
  std::vector<DTensor> W(n), Y(n), B(n);
  std::vector<bool> has_bias(n, false);
  for (int j = 0; j < n; ++j) {
    if ((st = parse_dtensor(&w[j], &W[j], "w")) != DT_OK) return st;
    if ((st = parse_dtensor(&y[j], &Y[j], "y")) != DT_OK) return st;
    if (bias && bias[j].nslots > 0) {
      if ((st = parse_dtensor(&bias[j], &B[j], "bias")) != DT_OK) return st;
      has_bias[j] = true;
    }
    ColumnSpec c{&W[j], has_bias[j] ? &B[j] : nullptr, &Y[j]};
    if ((st = check_column(X, c, tp, true)) != DT_OK) return st;
  }
  std::set<std::tuple<const void*, int, int, int>> done;
  for (int j = 0; j < n; ++j) {
    ColumnSpec c{&W[j], has_bias[j] ? &B[j] : nullptr, &Y[j]};
    if ((st = add_column_groups(X, c, tp, groups, &done)) != DT_OK) return st;
  }
  // a token-sharded x: each token shard's groups together, in weight order,
  // so a launch can order its tiles as the one GEMM of which they are parts
  std::stable_sort(groups->begin(), groups->end(),
                   [](const HostGroup& a, const HostGroup& b) { return a.m_block < b.m_block; });
  return DT_OK;
}

dt_status column_multi(const dt_dtensor* x, int32_t n, const dt_dtensor* w, const dt_dtensor* bias,
                       const dt_dtensor* y, int32_t tp, gemm::Workspace ws, int32_t* d_status, dt_stream_t stream) {
  clear_error();
  std::vector<HostGroup> groups;
  dt_status st = column_build(x, n, w, bias, y, tp, &groups);
  if (st != DT_OK) return st;
  const void* out = first_output(groups);
  if (!out) return DT_OK;
  if ((st = bind_device_of(out)) != DT_OK) return st;
  return gemm::run_groups(groups, d_status, reinterpret_cast<cudaStream_t>(stream), ws);
}

// Row-parallel groups for one (x, w, y) triple; `x_override` replaces the x
// slots by explicit matrices (the MLP's H views) when non-null.
dt_status row_groups(const Layout& lx, const std::vector<Mat>* x_mats, const DTensor* X, const DTensor& W,
                     const DTensor* Bias, const DTensor& Y, int mode, int tp, std::vector<HostGroup>* groups) {
  const Layout& lw = W.layout;
  const Layout& ly = Y.layout;
  const int nd = lx.ndim;
  const int P = tp_size(lx, tp);
  std::set<int> done;
  int c0[DT_MAX_MESH_DIMS], cj[DT_MAX_MESH_DIMS];
  for (int r = 0; r < lx.mesh_size; ++r) {
    lx.rank_coords(r, c0);
    if (tp >= 0 && c0[tp] != 0) continue;
    // the P ranks of this tp group, in tp order
    std::vector<HostSeg> segs;
    std::vector<int> yslots;
    Mat xm0;
    int64_t x_row0 = 0;
    for (int j = 0; j < P; ++j) {
      std::copy(c0, c0 + DT_MAX_MESH_DIMS, cj);
      if (tp >= 0) cj[tp] = j;
      Mat a, b;
      dt_status st;
      const int xs = lx.slot_of_coords(cj);
      if (x_mats) {
        a = (*x_mats)[xs];
      } else {
        const SlotView& xv = X->slots[xs];
        if ((st = slot_matrix(xv, nd, lx.dtype, &a, "x")) != DT_OK) return st;
      }
      x_row0 = lx.slot_box(xs).off[0];
      const SlotView& wv = W.slots[lw.slot_of_coords(cj)];
      if ((st = weight_matrix(wv, lw.dtype, &b, "w")) != DT_OK) return st;
      if (a.cols != b.rows) return fail(DT_ERR_SHAPE, "x shard width %lld != w shard rows %lld", (long long)a.cols, (long long)b.rows);
      if (j == 0) xm0 = a;
      if (a.rows != xm0.rows) return fail(DT_ERR_SHAPE, "x shards have different row counts");
      segs.push_back(HostSeg{a, b, Mat()});
      yslots.push_back(ly.slot_of_coords(cj));
    }
    const int64_t M = xm0.rows, N = lw.gshape[1];
    const void* bias_ptr = nullptr;
    int bias_dtype = -1;
    if (Bias) {
      const SlotView& bv = Bias->slots[Bias->layout.slot_of_coords(c0)];
      if (bv.shape[0] > 1 && bv.stride[0] != 1) return fail(DT_ERR_UNSUPPORTED, "bias must be contiguous");
      bias_ptr = bv.ptr;
      bias_dtype = Bias->layout.dtype;
    }
    if (mode == DT_TP_ALL_REDUCE) {
      for (int j = 0; j < P; ++j) {
        if (!done.insert(yslots[j]).second) continue;
        Mat y;
        dt_status st = slot_matrix(Y.slots[yslots[j]], nd, ly.dtype, &y, "y");
        if (st != DT_OK) return st;
        if (y.rows != M || y.cols != N) return fail(DT_ERR_SHAPE, "ALL_REDUCE output slot shape");
        HostGroup g;
        g.m = M;
        g.n = N;
        g.segs = segs;
        g.out_dtype = ly.dtype;
        g.row_begin = {0};
        g.out_ptr = {y.ptr};
        g.out_ld = {y.ld};
        g.bias = bias_ptr;
        g.bias_dtype = bias_dtype;
        groups->push_back(std::move(g));
      }
    } else if (mode == DT_TP_REDUCE_SCATTER) {
      if (!done.insert(yslots[0]).second) continue;
      HostGroup g;
      g.m = M;
      g.n = N;
      g.segs = segs;
      g.out_dtype = ly.dtype;
      g.bias = bias_ptr;
      g.bias_dtype = bias_dtype;
      int64_t next = 0;
      for (int j = 0; j < P; ++j) {
        const SlotView& yv = Y.slots[yslots[j]];
        Mat y;
        dt_status st = slot_matrix(yv, nd, ly.dtype, &y, "y");
        if (st != DT_OK) return st;
        if (y.rows == 0) continue;
        const int64_t begin = (yv.goff[0] - x_row0) * rows_per_dim0(yv, nd);
        if (begin != next || y.cols != N) return fail(DT_ERR_SHAPE, "REDUCE_SCATTER output blocks do not tile the rows");
        g.row_begin.push_back(begin);
        g.out_ptr.push_back(y.ptr);
        g.out_ld.push_back(y.ld);
        next = begin + y.rows;
      }
      if (next != M) return fail(DT_ERR_SHAPE, "REDUCE_SCATTER output blocks cover %lld of %lld rows", (long long)next, (long long)M);
      groups->push_back(std::move(g));
    } else {  // DT_TP_PARTIAL
      for (int j = 0; j < P; ++j) {
        if (!done.insert(yslots[j]).second) continue;
        Mat y;
        dt_status st = slot_matrix(Y.slots[yslots[j]], nd, ly.dtype, &y, "y");
        if (st != DT_OK) return st;
        if (y.rows != M || y.cols != N) return fail(DT_ERR_SHAPE, "PARTIAL output slot shape");
        HostGroup g;
        g.m = M;
        g.n = N;
        g.segs = {segs[j]};
        g.out_dtype = ly.dtype;
        g.row_begin = {0};
        g.out_ptr = {y.ptr};
        g.out_ld = {y.ld};
        if (j == 0) {  // the parts sum to X W + b: the bias rides on part 0
          g.bias = bias_ptr;
          g.bias_dtype = bias_dtype;
        }
        groups->push_back(std::move(g));
      }
    }
  }
  return DT_OK;
}

// Checks of the row layer: x [.., K] Shard(-1) on tp, w [K, N] Shard(0) on
// tp, bias [N] Replicate, y per mode; off tp weights/bias Replicate and x, y
// placed alike.
dt_status check_row(const Layout& lx, const Layout& lw, const Layout* lb, const Layout& ly, int mode, int tp) {
  if (!same_mesh(lx, lw) || !same_mesh(lx, ly) || (lb && !same_mesh(lx, *lb)))
    return fail(DT_ERR_SHAPE, "operands live on different meshes");
  if (mode != DT_TP_ALL_REDUCE && mode != DT_TP_REDUCE_SCATTER && mode != DT_TP_PARTIAL)
    return fail(DT_ERR_INVALID_ARG, "mode %d", mode);
  if (lw.ndim != 2) return fail(DT_ERR_SHAPE, "weight must be 2-D [in, out]");
  if (lx.dtype != lw.dtype) return fail(DT_ERR_INVALID_ARG, "x and w dtypes differ");
  if (lx.dtype == DT_INT32 || ly.dtype == DT_INT32) return fail(DT_ERR_INVALID_ARG, "int32 linear");
  const int nd = lx.ndim;
  if (ly.ndim != nd) return fail(DT_ERR_SHAPE, "y rank must equal x rank");
  if (lx.gshape[nd - 1] != lw.gshape[0]) return fail(DT_ERR_SHAPE, "x last dim != w rows");
  for (int d = 0; d < nd - 1; ++d)
    if (ly.gshape[d] != lx.gshape[d]) return fail(DT_ERR_SHAPE, "y leading dims differ from x");
  if (ly.gshape[nd - 1] != lw.gshape[1]) return fail(DT_ERR_SHAPE, "y last dim != w cols");
  if (dt_status st = check_gemm_dims(lx, lw.gshape[0], lw.gshape[1]); st != DT_OK) return st;
  if (lb) {
    if (lb->ndim != 1 || lb->gshape[0] != lw.gshape[1]) return fail(DT_ERR_SHAPE, "bias must be [out]");
    if (lb->dtype == DT_INT32) return fail(DT_ERR_INVALID_ARG, "bias dtype");
  }
  for (int m = 0; m < lx.mesh_ndim; ++m) {
    if (m == tp) {
      if (!lx.is_shard(m, nd - 1)) return fail(DT_ERR_PLACEMENT, "row-parallel input must be Shard(-1) on tp, got %s", pname(lx, m));
      if (!lw.is_shard(m, 0)) return fail(DT_ERR_PLACEMENT, "row-parallel weight [in, out] must be Shard(0) on tp");
      if (lb && !lb->is_replicate(m)) return fail(DT_ERR_PLACEMENT, "row-parallel bias is passed reduced (Replicate)");
      if (mode == DT_TP_ALL_REDUCE && !ly.is_replicate(m)) return fail(DT_ERR_PLACEMENT, "ALL_REDUCE output must be Replicate on tp");
      if (mode == DT_TP_REDUCE_SCATTER && !ly.is_shard(m, 0)) return fail(DT_ERR_PLACEMENT, "REDUCE_SCATTER output must be Shard(0) on tp");
      if (mode == DT_TP_REDUCE_SCATTER && nd < 2) return fail(DT_ERR_SHAPE, "REDUCE_SCATTER needs a leading dim");
      if (mode == DT_TP_PARTIAL && !ly.is_partial(m)) return fail(DT_ERR_PLACEMENT, "PARTIAL output must be Partial on tp");
      if (mode == DT_TP_PARTIAL && ly.op[m] != DT_SUM) return fail(DT_ERR_UNSUPPORTED, "a linear's partial products are summed: Partial(sum) only");
    } else {
      if (!lw.is_replicate(m)) return fail(DT_ERR_PLACEMENT, "weight must be Replicate off tp");
      if (lb && !lb->is_replicate(m)) return fail(DT_ERR_PLACEMENT, "bias must be Replicate off tp");
      if (!same_placement(lx, m, ly, m)) return fail(DT_ERR_PLACEMENT, "x and y must be placed alike off tp");
      if (lx.kind[m] == DT_SHARD && lx.dim[m] == nd - 1) return fail(DT_ERR_PLACEMENT, "x may be sharded on its last dim only on tp");
      if (lx.is_partial(m) && lb) return fail(DT_ERR_PLACEMENT, "Partial input with a bias");
      if (mode == DT_TP_REDUCE_SCATTER && lx.kind[m] == DT_SHARD && lx.dim[m] == 0 && m > tp)
        return fail(DT_ERR_UNSUPPORTED, "dim 0 sharded by a mesh dim inside tp");
    }
  }
  return DT_OK;
}

// Plans of the linears by operands (and stream, status word, workspace and
// allocation scope, which the launches' parameters also hold).  A hit
// replays the recorded launches; bounded, dropped whole when full.
std::mutex g_gemm_plan_mu;
std::unordered_map<std::string, std::shared_ptr<const gemm::GemmRecord>> g_gemm_plans;
std::unordered_map<std::string, int> g_gemm_plan_device;
constexpr size_t GEMM_PLAN_CACHE = 128;

template <class F>
dt_status with_gemm_plan(const std::string* key, dt_stream_t stream, F&& plan_and_launch) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (key) {
    std::shared_ptr<const gemm::GemmRecord> hit;
    int dev = -1;
    {
      std::lock_guard<std::mutex> lk(g_gemm_plan_mu);
      auto it = g_gemm_plans.find(*key);
      if (it != g_gemm_plans.end()) {
        hit = it->second;
        dev = g_gemm_plan_device[*key];
      }
    }
    if (hit) {
      clear_error();
      int cur = -1;
      cudaGetDevice(&cur);
      if (dev >= 0 && cur != dev && cudaSetDevice(dev) != cudaSuccess)
        return fail(DT_ERR_CUDA, "cudaSetDevice(%d)", dev);
      return gemm::replay_gemm(*hit, s);
    }
  }
  std::shared_ptr<gemm::GemmRecord> rec = gemm::new_gemm_record();
  dt_status st;
  {
    gemm::GemmRecordScope scope(rec.get());
    st = plan_and_launch();
  }
  if (st == DT_OK && key) {
    int dev = -1;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_gemm_plan_mu);
    if (g_gemm_plans.size() >= GEMM_PLAN_CACHE) {
      g_gemm_plans.clear();
      g_gemm_plan_device.clear();
    }
    g_gemm_plans[*key] = rec;
    g_gemm_plan_device[*key] = dev;
  }
  return st;
}

// The key's common tail: what the recorded parameters hold besides the operands.
void finish_key(std::string* k, void* workspace, size_t workspace_bytes, int32_t* d_status, dt_stream_t stream) {
  append_plan_scalar(k, workspace);
  append_plan_scalar(k, workspace_bytes);
  append_plan_scalar(k, d_status);
  append_plan_scalar(k, stream);
}

// A linear's workspace: null (size ignored), or 256-byte aligned device memory.
dt_status check_workspace(void* workspace, size_t workspace_bytes, gemm::Workspace* ws) {
  if (!workspace) return DT_OK;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(DT_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  ws->ptr = static_cast<char*>(workspace);
  ws->bytes = workspace_bytes;
  return DT_OK;
}

}  // namespace

void clear_gemm_plans() {
  std::lock_guard<std::mutex> lk(g_gemm_plan_mu);
  g_gemm_plans.clear();
  g_gemm_plan_device.clear();
}

}  // namespace dt

using namespace dt;

extern "C" {

dt_status dt_column_parallel_linear_multi(const dt_dtensor* x, int32_t n, const dt_dtensor* w,
                                          const dt_dtensor* bias, const dt_dtensor* y, int32_t tp_mesh_dim,
                                          void* workspace, size_t workspace_bytes, int32_t* d_status,
                                          dt_stream_t stream) {
  clear_error();
  gemm::Workspace ws;
  if (dt_status st = check_workspace(workspace, workspace_bytes, &ws); st != DT_OK) return st;
  std::string key(1, 'c');
  bool keyed = n >= 0 && n <= 64 && (n == 0 || (w && y)) && append_plan_key(&key, x);
  for (int j = 0; j < n && keyed; ++j)
    keyed = append_plan_key(&key, &w[j]) && append_plan_key(&key, &y[j]) &&
            append_plan_key(&key, bias ? &bias[j] : nullptr);
  append_plan_scalar(&key, tp_mesh_dim);
  finish_key(&key, workspace, workspace_bytes, d_status, stream);
  return with_gemm_plan(keyed ? &key : nullptr, stream,
                        [&] { return column_multi(x, n, w, bias, y, tp_mesh_dim, ws, d_status, stream); });
}

dt_status dt_column_parallel_linear(const dt_dtensor* x, const dt_dtensor* w, const dt_dtensor* bias,
                                    const dt_dtensor* y, int32_t tp_mesh_dim, void* workspace,
                                    size_t workspace_bytes, int32_t* d_status, dt_stream_t stream) {
  return dt_column_parallel_linear_multi(x, 1, w, bias, y, tp_mesh_dim, workspace, workspace_bytes, d_status,
                                         stream);
}

dt_status dt_column_parallel_linear_workspace_size(const dt_dtensor* x, int32_t n, const dt_dtensor* w,
                                                   const dt_dtensor* y, int32_t tp_mesh_dim, size_t* bytes) {
  clear_error();
  if (!bytes) return fail(DT_ERR_INVALID_ARG, "bytes is NULL");
  std::vector<HostGroup> groups;
  dt_status st = column_build(x, n, w, nullptr, y, tp_mesh_dim, &groups);
  if (st != DT_OK) return st;
  return gemm::workspace_bytes(groups, bytes);
}

}  // extern "C"

namespace dt {
namespace {

// Parse and check a row call and lower it to GEMM groups.
dt_status row_build(const dt_dtensor* x, const dt_dtensor* w, const dt_dtensor* bias, const dt_dtensor* y,
                    int32_t mode, int32_t tp, std::vector<HostGroup>* groups) {
  DTensor X, W, B, Y;
  dt_status st;
  if ((st = parse_dtensor(x, &X, "x")) != DT_OK) return st;
  if ((st = parse_dtensor(w, &W, "w")) != DT_OK) return st;
  if ((st = parse_dtensor(y, &Y, "y")) != DT_OK) return st;
  const bool has_bias = bias && bias->nslots > 0;
  if (has_bias && (st = parse_dtensor(bias, &B, "bias")) != DT_OK) return st;
  if ((st = check_tp(tp, X.layout)) != DT_OK) return st;
  if (tp < 0 && mode != DT_TP_ALL_REDUCE)
    return fail(DT_ERR_INVALID_ARG, "without tp only ALL_REDUCE (a plain linear) is defined");
  if ((st = check_row(X.layout, W.layout, has_bias ? &B.layout : nullptr, Y.layout, mode, tp)) != DT_OK) return st;
  return row_groups(X.layout, nullptr, &X, W, has_bias ? &B : nullptr, Y, mode, tp, groups);
}

dt_status row_parallel_planned(const dt_dtensor* x, const dt_dtensor* w, const dt_dtensor* bias, const dt_dtensor* y,
                               int32_t mode, int32_t tp, gemm::Workspace ws, int32_t* d_status, dt_stream_t stream) {
  clear_error();
  std::vector<HostGroup> groups;
  dt_status st = row_build(x, w, bias, y, mode, tp, &groups);
  if (st != DT_OK) return st;
  const void* out = first_output(groups);
  if (!out) return DT_OK;
  if ((st = bind_device_of(out)) != DT_OK) return st;
  return gemm::run_groups(groups, d_status, reinterpret_cast<cudaStream_t>(stream), ws);
}

}  // namespace
}  // namespace dt

extern "C" {

dt_status dt_row_parallel_linear(const dt_dtensor* x, const dt_dtensor* w, const dt_dtensor* bias,
                                 const dt_dtensor* y, int32_t mode, int32_t tp_mesh_dim, void* workspace,
                                 size_t workspace_bytes, int32_t* d_status, dt_stream_t stream) {
  clear_error();
  gemm::Workspace ws;
  if (dt_status st = check_workspace(workspace, workspace_bytes, &ws); st != DT_OK) return st;
  std::string key(1, 'r');
  const bool keyed = append_plan_key(&key, x) && append_plan_key(&key, w) && append_plan_key(&key, bias) &&
                     append_plan_key(&key, y);
  append_plan_scalar(&key, mode);
  append_plan_scalar(&key, tp_mesh_dim);
  finish_key(&key, workspace, workspace_bytes, d_status, stream);
  return with_gemm_plan(keyed ? &key : nullptr, stream, [&] {
    return row_parallel_planned(x, w, bias, y, mode, tp_mesh_dim, ws, d_status, stream);
  });
}

dt_status dt_row_parallel_linear_workspace_size(const dt_dtensor* x, const dt_dtensor* w, const dt_dtensor* y,
                                                int32_t mode, int32_t tp_mesh_dim, size_t* bytes) {
  clear_error();
  if (!bytes) return fail(DT_ERR_INVALID_ARG, "bytes is NULL");
  std::vector<HostGroup> groups;
  dt_status st = row_build(x, w, nullptr, y, mode, tp_mesh_dim, &groups);
  if (st != DT_OK) return st;
  return gemm::workspace_bytes(groups, bytes);
}

// ---- TP MLP -------------------------------------------------------------

}  // extern "C"

namespace dt {
namespace {

struct MlpPlan {
  std::vector<int> x_slots;        // distinct x slots (one H block each)
  std::vector<int64_t> h_offset;   // byte offset of each H block
  std::vector<int64_t> h_rows;
  int64_t F = 0;
  size_t bytes = 0;                // every H block, 256-byte aligned
};

dt_status mlp_plan(const DTensor& X, const DTensor& Wg, MlpPlan* plan) {
  const Layout& lx = X.layout;
  if (lx.ndim < 1) return fail(DT_ERR_SHAPE, "x rank");
  if (Wg.layout.ndim != 2) return fail(DT_ERR_SHAPE, "w_gate must be 2-D [in, ffn]");
  plan->F = Wg.layout.gshape[1];
  std::set<int> seen;
  int c[DT_MAX_MESH_DIMS];
  size_t off = 0;
  for (int r = 0; r < lx.mesh_size; ++r) {
    lx.rank_coords(r, c);
    const int s = lx.slot_of_coords(c);
    if (!seen.insert(s).second) continue;
    const SlotView& v = X.slots[s];
    int64_t rows = 1;
    for (int d = 0; d < lx.ndim - 1; ++d) rows *= v.shape[d];
    plan->x_slots.push_back(s);
    plan->h_offset.push_back((int64_t)off);
    plan->h_rows.push_back(rows);
    off += ((size_t)rows * (size_t)plan->F * 2 + 255) & ~size_t(255);
  }
  plan->bytes = off;
  return DT_OK;
}

// Parse and check an MLP call and lower it to its two GEMM launches' groups,
// with H at `h_base` (256-byte aligned device memory of plan->bytes).
dt_status mlp_build(const dt_dtensor* x, const dt_dtensor* w_gate, const dt_dtensor* w_up, const dt_dtensor* w_down,
                    const dt_dtensor* y, int32_t mode, int32_t tp, char* h_base, MlpPlan* plan,
                    std::vector<HostGroup>* up_groups, std::vector<HostGroup>* down_groups) {
  DTensor X, Wg, Wu, Wd, Y;
  dt_status st;
  if ((st = parse_dtensor(x, &X, "x")) != DT_OK) return st;
  if ((st = parse_dtensor(w_gate, &Wg, "w_gate")) != DT_OK) return st;
  if ((st = parse_dtensor(w_up, &Wu, "w_up")) != DT_OK) return st;
  if ((st = parse_dtensor(w_down, &Wd, "w_down")) != DT_OK) return st;
  if ((st = parse_dtensor(y, &Y, "y")) != DT_OK) return st;
  if ((st = check_tp(tp, X.layout)) != DT_OK) return st;
  const Layout& lx = X.layout;
  if (lx.dtype != DT_BF16 || Wg.layout.dtype != DT_BF16 || Wu.layout.dtype != DT_BF16 || Wd.layout.dtype != DT_BF16)
    return fail(DT_ERR_INVALID_ARG, "the TP MLP runs bf16 operands");
  // gate and up: column-parallel with the same placement and shape
  if (Wg.layout.ndim != 2 || Wu.layout.ndim != 2 || Wg.layout.gshape[0] != Wu.layout.gshape[0] ||
      Wg.layout.gshape[1] != Wu.layout.gshape[1])
    return fail(DT_ERR_SHAPE, "gate and up weights must have one shape");
  for (int m = 0; m < lx.mesh_ndim; ++m)
    if (!same_placement(Wg.layout, m, Wu.layout, m)) return fail(DT_ERR_PLACEMENT, "gate and up weights placed differently");
  for (int m = 0; m < lx.mesh_ndim; ++m) {
    if (m == tp) {
      if (!lx.is_replicate(m)) return fail(DT_ERR_PLACEMENT, "MLP input must be Replicate on tp");
      if (!Wg.layout.is_shard(m, 1)) return fail(DT_ERR_PLACEMENT, "gate/up weights [in, out] must be Shard(1) on tp");
    } else if (!Wg.layout.is_replicate(m)) {
      return fail(DT_ERR_PLACEMENT, "weights must be Replicate off tp");
    } else if (lx.is_partial(m)) {
      return fail(DT_ERR_PLACEMENT, "the MLP is not linear in a Partial input");
    } else if (lx.kind[m] == DT_SHARD && lx.dim[m] == lx.ndim - 1) {
      return fail(DT_ERR_PLACEMENT, "x may not be sharded on its last dim");
    }
  }
  const int nd = lx.ndim;
  if (lx.gshape[nd - 1] != Wg.layout.gshape[0]) return fail(DT_ERR_SHAPE, "x last dim != w_gate rows");
  if (Wd.layout.ndim != 2 || Wd.layout.gshape[0] != Wg.layout.gshape[1]) return fail(DT_ERR_SHAPE, "w_down must be [ffn, out]");
  if ((st = check_gemm_dims(lx, Wg.layout.gshape[0], 2 * Wg.layout.gshape[1])) != DT_OK) return st;
  if ((st = mlp_plan(X, Wg, plan)) != DT_OK) return st;
  const int64_t F = plan->F;
  if ((F * 2) % 16) return fail(DT_ERR_ALIGNMENT, "ffn width must be a multiple of 8");

  // H as a layout: x's placements with the last dim of size F, Shard(-1) on tp.
  dt_layout hl;
  std::memset(&hl, 0, sizeof(hl));
  hl.mesh_ndim = lx.mesh_ndim;
  for (int m = 0; m < lx.mesh_ndim; ++m) {
    hl.mesh_shape[m] = lx.mesh[m];
    hl.placements[m].kind = lx.kind[m];
    hl.placements[m].dim = lx.dim[m];
    if (m == tp) {
      hl.placements[m].kind = DT_SHARD;
      hl.placements[m].dim = nd - 1;
    }
  }
  hl.ndim = nd;
  for (int d = 0; d < nd; ++d) hl.gshape[d] = lx.gshape[d];
  hl.gshape[nd - 1] = F;
  hl.dtype = DT_BF16;
  Layout LH;
  if ((st = parse_layout(&hl, &LH)) != DT_OK) return st;
  // every H slot is a column block of its x slot's [rows, F] H block
  std::vector<Mat> hmats(LH.nslots);
  int c[DT_MAX_MESH_DIMS];
  for (int s = 0; s < LH.nslots; ++s) {
    LH.slot_coords(s, c);
    const int xs = lx.slot_of_coords(c);
    size_t bi = 0;
    while (bi < plan->x_slots.size() && plan->x_slots[bi] != xs) ++bi;
    const Box hb = LH.slot_box(s);
    Mat m;
    m.ptr = h_base + plan->h_offset[bi] + hb.off[nd - 1] * 2;
    m.rows = plan->h_rows[bi];
    m.cols = hb.size[nd - 1];
    m.ld = F;
    m.dtype = DT_BF16;
    hmats[s] = m;
  }
  // 1) gate/up: one dual group per (x slot, tp shard)
  std::set<int> done;
  for (int r = 0; r < lx.mesh_size; ++r) {
    lx.rank_coords(r, c);
    const int hs = LH.slot_of_coords(c);
    if (!done.insert(hs).second) continue;
    Mat a, bg, bu;
    if ((st = slot_matrix(X.slots[lx.slot_of_coords(c)], nd, DT_BF16, &a, "x")) != DT_OK) return st;
    if ((st = weight_matrix(Wg.slots[Wg.layout.slot_of_coords(c)], DT_BF16, &bg, "w_gate")) != DT_OK) return st;
    if ((st = weight_matrix(Wu.slots[Wu.layout.slot_of_coords(c)], DT_BF16, &bu, "w_up")) != DT_OK) return st;
    const Mat& h = hmats[hs];
    if (bg.cols != h.cols || bu.cols != h.cols || a.cols != bg.rows || a.rows != h.rows)
      return fail(DT_ERR_SHAPE, "gate/up local shapes disagree");
    HostGroup g;
    g.m = h.rows;
    g.n = h.cols;
    g.dual = true;
    g.segs.push_back(HostSeg{a, bg, bu});
    g.out_dtype = DT_BF16;
    g.row_begin = {0};
    g.out_ptr = {h.ptr};
    g.out_ld = {h.ld};
    up_groups->push_back(std::move(g));
  }
  // 2) down: row-parallel over the H shards
  if ((st = check_row(LH, Wd.layout, nullptr, Y.layout, mode, tp)) != DT_OK) return st;
  return row_groups(LH, &hmats, nullptr, Wd, nullptr, Y, mode, tp, down_groups);
}

dt_status tp_mlp_planned(const dt_dtensor* x, const dt_dtensor* w_gate, const dt_dtensor* w_up,
                         const dt_dtensor* w_down, const dt_dtensor* y, int32_t mode, int32_t tp_mesh_dim,
                         void* workspace, size_t workspace_bytes, int32_t* d_status, dt_stream_t stream) {
  clear_error();
  if (workspace && reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(DT_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  MlpPlan plan;
  std::vector<HostGroup> up_groups, down_groups;
  dt_status st = mlp_build(x, w_gate, w_up, w_down, y, mode, tp_mesh_dim, static_cast<char*>(workspace), &plan,
                           &up_groups, &down_groups);
  if (st != DT_OK) return st;
  if (plan.bytes > 0 && (!workspace || workspace_bytes < plan.bytes))
    return fail(DT_ERR_INVALID_ARG, "workspace of at least %zu bytes (H) needed", plan.bytes);
  // H is empty with no tokens or no ffn columns: then the launches write Y
  // alone (zeros and nothing else when the ffn width is 0), or nothing
  const void* anchor = workspace ? workspace : first_output(down_groups);
  if (!anchor) return DT_OK;
  if ((st = bind_device_of(anchor)) != DT_OK) return st;
  // the split tail's scratch follows H; both launches run in order on the
  // stream, so they share it
  gemm::Workspace split;
  split.ptr = workspace ? static_cast<char*>(workspace) + plan.bytes : nullptr;
  split.bytes = workspace ? workspace_bytes - plan.bytes : 0;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = gemm::run_groups(up_groups, d_status, s, split)) != DT_OK) return st;
  return gemm::run_groups(down_groups, d_status, s, split);
}

}  // namespace

dt_status mlp_hidden_bytes(const dt_dtensor* x, const dt_dtensor* w_gate, size_t* bytes) {
  DTensor X, Wg;
  dt_status st;
  if ((st = parse_dtensor(x, &X, "x")) != DT_OK) return st;
  if ((st = parse_dtensor(w_gate, &Wg, "w_gate")) != DT_OK) return st;
  MlpPlan plan;
  if ((st = mlp_plan(X, Wg, &plan)) != DT_OK) return st;
  *bytes = plan.bytes;
  return DT_OK;
}

}  // namespace dt

extern "C" {

dt_status dt_tp_mlp_workspace_size(const dt_dtensor* x, const dt_dtensor* w_gate, const dt_dtensor* w_up,
                                   const dt_dtensor* w_down, const dt_dtensor* y, int32_t mode, int32_t tp_mesh_dim,
                                   size_t* bytes) {
  clear_error();
  if (!bytes) return fail(DT_ERR_INVALID_ARG, "bytes is NULL");
  // H's place in the workspace only matters through its alignment
  char* const h_base = reinterpret_cast<char*>(uintptr_t(256));
  MlpPlan plan;
  std::vector<HostGroup> up_groups, down_groups;
  dt_status st = mlp_build(x, w_gate, w_up, w_down, y, mode, tp_mesh_dim, h_base, &plan, &up_groups, &down_groups);
  if (st != DT_OK) return st;
  size_t up = 0, down = 0;
  if ((st = gemm::workspace_bytes(up_groups, &up)) != DT_OK) return st;
  if ((st = gemm::workspace_bytes(down_groups, &down)) != DT_OK) return st;
  *bytes = plan.bytes + std::max(up, down);
  return DT_OK;
}

dt_status dt_tp_mlp(const dt_dtensor* x, const dt_dtensor* w_gate, const dt_dtensor* w_up, const dt_dtensor* w_down,
                    const dt_dtensor* y, int32_t mode, int32_t tp_mesh_dim, void* workspace, size_t workspace_bytes,
                    int32_t* d_status, dt_stream_t stream) {
  std::string key(1, 'm');
  const bool keyed = append_plan_key(&key, x) && append_plan_key(&key, w_gate) && append_plan_key(&key, w_up) &&
                     append_plan_key(&key, w_down) && append_plan_key(&key, y);
  append_plan_scalar(&key, mode);
  append_plan_scalar(&key, tp_mesh_dim);
  finish_key(&key, workspace, workspace_bytes, d_status, stream);
  return with_gemm_plan(keyed ? &key : nullptr, stream, [&] {
    return tp_mlp_planned(x, w_gate, w_up, w_down, y, mode, tp_mesh_dim, workspace, workspace_bytes, d_status,
                          stream);
  });
}

}  // extern "C"
