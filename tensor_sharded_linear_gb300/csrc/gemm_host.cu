// Lowering of batched GEMM groups to launches: TMA descriptors (cached on
// the host), the packing of groups into launches, the tile order, the split
// tail (its scratch in the caller's workspace), and the choice between the
// tcgen05 kernel and the CUDA-core kernel (fp32 operands, or bf16 operands
// whose pitches TMA cannot describe).
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "gemm_plan.h"
#include "gemm_sm103.cuh"

namespace dt {
namespace gemm {

// A bf16 matrix copied into the workspace with a row pitch TMA can describe.
struct PitchCopy {
  char* dst;
  const char* src;
  int64_t dst_ld, src_ld, rows, cols;  // elements
  int grid_x, grid_y;
};

// One recorded step of a call: a GEMM launch (kind 0: tcgen05 pair kernel,
// 2: CUDA-core kernel) with its exact parameter block, (kind 3) the zeroing
// of split-tail counters that precedes a split launch, or (kind 4) the copy
// of an operand into a TMA-compatible pitch.
struct GemmLaunch {
  int kind = 0;
  int grid = 0;
  std::shared_ptr<void> params;  // a heap Params (keeps its 128-byte alignment) or SParams
  void* zero_ptr = nullptr;
  size_t zero_bytes = 0;
  PitchCopy pc{};
};
struct GemmRecord {
  std::vector<GemmLaunch> launches;
};

namespace {

// ------------------------------------------------------------ TMA descriptors

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

struct MapKey {
  uintptr_t ptr;
  int64_t rows, cols, ld;
  int32_t box_rows;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && cols == o.cols && ld == o.ld && box_rows == o.box_rows;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    size_t h = std::hash<uintptr_t>()(k.ptr);
    h ^= std::hash<int64_t>()(k.rows) + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    h ^= std::hash<int64_t>()(k.cols) + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    h ^= std::hash<int64_t>()(k.ld) + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
    h ^= std::hash<int32_t>()(k.box_rows) + (h << 6);
    return h;
  }
};

std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;
thread_local GemmRecord* g_grec = nullptr;
std::atomic<uint64_t> g_simt_launches{0};

// 2-D bf16 map over a row-major [rows, cols] matrix with pitch ld elements:
// box of 64 columns (128 bytes, the swizzle width) by box_rows rows, 128-byte
// swizzle, zero fill outside the matrix.
dt_status encode_map(const Mat& m, int box_rows, CUtensorMap* out) {
  MapKey key{reinterpret_cast<uintptr_t>(m.ptr), m.rows, m.cols, m.ld, box_rows};
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *out = it->second;
      return DT_OK;
    }
  }
  auto fn = encode_fn();
  if (!fn) return fail(DT_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  CUtensorMap map;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(m.cols), static_cast<cuuint64_t>(m.rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(m.ld) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, m.ptr, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DT_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_maps.size() > 8192) g_maps.clear();
    g_maps.emplace(key, map);
  }
  *out = map;
  return DT_OK;
}

// The matrix as it lies in memory: rows x cols row-major with pitch ld
// (a K-major weight [K, N] is stored as N rows of K).
Mat stored(const Mat& m) {
  if (!m.kmajor) return m;
  Mat s = m;
  s.rows = m.cols;
  s.cols = m.rows;
  s.kmajor = false;
  return s;
}

bool tma_ok(const Mat& m0) {
  const Mat m = stored(m0);
  return m.dtype == DT_BF16 && m.rows > 0 && m.cols > 0 && (reinterpret_cast<uintptr_t>(m.ptr) % 16) == 0 &&
         (m.ld * 2) % 16 == 0 && m.ld >= m.cols && m.rows < (1ll << 31) && m.cols < (1ll << 31);
}

// ------------------------------------------------------------ CUDA-core kernel

constexpr int S_TILE = 64, S_BK = 16, S_THREADS = 256;

struct SSeg {
  const char* a;
  const char* b;
  int64_t lda, ldb;
  int32_t k, dtype;
  int32_t b_kmajor, pad;
};

struct SGroup {
  int64_t m, n;
  int32_t seg_begin, seg_count, m_tiles, n_tiles, tile_begin, out_dtype, nout, bias_dtype;
  const void* bias;
  int64_t row_begin[MAX_OUT + 1];
  char* out_ptr[MAX_OUT];
  int64_t out_ld[MAX_OUT];
};

struct SParams {
  SSeg segs[MAX_SEGS];
  SGroup groups[MAX_GROUPS];
  int32_t ngroups, total_tiles;
};

__device__ __forceinline__ float load_elem(const char* base, int64_t idx, int dtype) {
  if (dtype == DT_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  return reinterpret_cast<const float*>(base)[idx];
}

// 64 x 64 output tile per block, 4 x 4 per thread; each output sums its
// segments in order, k ascending, with fp32 fused multiply-adds.
__global__ void __launch_bounds__(S_THREADS) simt_gemm_kernel(const __grid_constant__ SParams p) {
  __shared__ float As[S_BK][S_TILE + 4];
  __shared__ float Bs[S_BK][S_TILE + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
    int g = 0;
    while (g + 1 < p.ngroups && p.groups[g + 1].tile_begin <= t) ++g;
    const SGroup& G = p.groups[g];
    const int local = t - G.tile_begin;
    const int64_t m0 = (int64_t)(local / G.n_tiles) * S_TILE;
    const int64_t n0 = (int64_t)(local % G.n_tiles) * S_TILE;
    float acc[4][4] = {};
    for (int si = G.seg_begin; si < G.seg_begin + G.seg_count; ++si) {
      const SSeg& S = p.segs[si];
      for (int k0 = 0; k0 < S.k; k0 += S_BK) {
        for (int e = threadIdx.x; e < S_TILE * S_BK; e += S_THREADS) {
          const int kk = e % S_BK, rr = e / S_BK;
          const int64_t row = m0 + rr, k = k0 + kk;
          As[kk][rr] = (row < G.m && k < S.k) ? load_elem(S.a, row * S.lda + k, S.dtype) : 0.f;
          const int cc = e % S_TILE, kb = e / S_TILE;
          const int64_t col = n0 + cc, kr = k0 + kb;
          Bs[kb][cc] = (col < G.n && kr < S.k)
                           ? load_elem(S.b, S.b_kmajor ? col * S.ldb + kr : kr * S.ldb + col, S.dtype)
                           : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < S_BK; ++kk) {
          float a[4], b[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
          for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = m0 + ty * 4 + i;
      if (r >= G.m) continue;
      int j = 0;
      while (j + 1 < G.nout && G.row_begin[j + 1] <= r) ++j;
      const int esize = G.out_dtype == DT_BF16 ? 2 : 4;
      char* row_ptr = G.out_ptr[j] + (r - G.row_begin[j]) * G.out_ld[j] * esize;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int64_t c = n0 + tx * 4 + jj;
        if (c >= G.n) continue;
        float v = acc[i][jj];
        if (G.bias_dtype >= 0) v += load_elem(static_cast<const char*>(G.bias), c, G.bias_dtype);
        if (G.out_dtype == DT_BF16) reinterpret_cast<__nv_bfloat16*>(row_ptr)[c] = __float2bfloat16_rn(v);
        else reinterpret_cast<float*>(row_ptr)[c] = v;
      }
    }
  }
}

// ------------------------------------------------------------ pitch copies

// Copy a [rows, cols] bf16 matrix (any element-aligned base and pitch) to a
// destination whose base is 16-byte aligned and whose pitch is a multiple of
// 8 elements: thread x of the row grid moves elements [8x, 8x + 8) of rows
// blockIdx.y, blockIdx.y + gridDim.y, ...; reads are element-wise (the
// source may sit at any alignment), writes whole 16-byte vectors.
__global__ void __launch_bounds__(256) pitch_copy_kernel(PitchCopy c) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t c0 = g * 8;
  if (c0 >= c.cols) return;
  const int n = c.cols - c0 < 8 ? static_cast<int>(c.cols - c0) : 8;
  for (int64_t r = blockIdx.y; r < c.rows; r += gridDim.y) {
    const uint16_t* s = reinterpret_cast<const uint16_t*>(c.src) + r * c.src_ld + c0;
    uint16_t* d = reinterpret_cast<uint16_t*>(c.dst) + r * c.dst_ld + c0;
    if (n == 8) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) w[k] = static_cast<uint32_t>(s[2 * k]) | (static_cast<uint32_t>(s[2 * k + 1]) << 16);
      *reinterpret_cast<uint4*>(d) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      for (int k = 0; k < n; ++k) d[k] = s[k];
    }
  }
}

cudaError_t launch_pitch_copy(const PitchCopy& c, cudaStream_t stream) {
  pitch_copy_kernel<<<dim3(c.grid_x, c.grid_y), 256, 0, stream>>>(c);
  return cudaGetLastError();
}

// ------------------------------------------------------------ lowering

// Every output block starts on a 32-byte boundary and its pitch is a
// multiple of 32 bytes: the epilogue may store whole 32-byte sectors.
bool out_vec32_ok(const HostGroup& g) {
  const int esize = g.out_dtype == DT_BF16 ? 2 : 4;
  for (size_t j = 0; j < g.out_ptr.size(); ++j) {
    if (reinterpret_cast<uintptr_t>(g.out_ptr[j]) % 32) return false;
    if ((g.out_ld[j] * esize) % 32) return false;
  }
  return true;
}

bool out_vec_ok(const HostGroup& g) {
  const int esize = g.out_dtype == DT_BF16 ? 2 : 4;
  for (size_t j = 0; j < g.out_ptr.size(); ++j) {
    if (reinterpret_cast<uintptr_t>(g.out_ptr[j]) % 16) return false;
    if ((g.out_ld[j] * esize) % 16) return false;
  }
  return true;
}

// Test hooks, read once from the environment: DT_GEMM_WAIT_LIMIT_MS bounds
// every mbarrier wait (default 2000 ms); DT_GEMM_STARVE=1 makes the TMA
// producers issue no loads, so the MMA waits run out and the kernel reports
// DT_DEV_ERR_TIMEOUT -- it exercises the bounded-wait exit without a fault.
unsigned long long gemm_wait_limit_ns() {
  static unsigned long long v = 0;
  if (!v) {
    const char* e = getenv("DT_GEMM_WAIT_LIMIT_MS");
    const long ms = e ? atol(e) : 0;
    v = (ms > 0 && ms <= 10000) ? (unsigned long long)ms * 1000000ull : WAIT_LIMIT_NS;
  }
  return v;
}

int gemm_starve() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("DT_GEMM_STARVE");
    v = (e && e[0] == '1') ? 1 : 0;
  }
  return v;
}

// What a split tail costs beyond its share of the MMAs, in 64-deep K
// iterations of one 256 x 256 pair tile (~0.33 us each): zeroing the
// counters, writing the pieces' partials, finishing the tiles, and the
// tail's operand traffic squeezed into a fraction of a tile's time.
// Measured on GB300 with the pieces first and the tiles finished from L2,
// forcing the split on 64-iteration launches: fused q/k/v (1536 tiles, a
// 16-tile tail) went from 418-421 to 413-415 us, the o projection (512
// tiles, a 56-tile tail) from 146-147 to 153-154 us.  Both put the cost
// at 35-40 iterations.
constexpr double SPLIT_OVERHEAD_ITERS = 40.0;

// DT_GEMM_SPLIT=0 in the environment turns the split tail off (every tile
// whole), DT_GEMM_SPLIT=2 splits every last wave the finishing can take
// whatever the cost model says, e.g. to compare the schedules.
int split_mode() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("DT_GEMM_SPLIT");
    v = (e && e[0] == '0') ? 0 : (e && e[0] == '2') ? 2 : 1;
  }
  return v;
}

// DT_GEMM_BANDS=m,n fixes the tile order's band height and block width (in
// tiles) of every launch with common M tiles, e.g. to compare orders; unset,
// the host chooses them (choose_bands).
bool bands_override(int* m, int* n) {
  static int vm = -1, vn = -1;
  if (vm < 0) {
    vm = vn = 0;
    const char* e = getenv("DT_GEMM_BANDS");
    int a = 0, b = 0;
    if (e && sscanf(e, "%d,%d", &a, &b) == 2 && a > 0 && b > 0) {
      vm = a;
      vn = b;
    }
  }
  *m = vm;
  *n = vn;
  return vm > 0;
}

// ---- launch packing

MapKey key_of(const Mat& m, int box) { return MapKey{reinterpret_cast<uintptr_t>(m.ptr), m.rows, m.cols, m.ld, box}; }

// Rows of a B descriptor's box: 64 K rows (MN-major B); 128 N rows per CTA
// of a pair (K-major B).
int b_box_rows(const HostGroup& G) { return G.segs.empty() || !G.segs[0].b.kmajor ? BK : 128; }

// Split `groups` into launches: consecutive runs whose groups, K segments
// and distinct TMA descriptors fit one parameter block.
dt_status pack_launches(const std::vector<HostGroup>& groups, std::vector<std::pair<size_t, size_t>>* out) {
  size_t gi = 0;
  while (gi < groups.size()) {
    std::vector<MapKey> keys;
    size_t g_end = gi;
    int nsegs = 0;
    while (g_end < groups.size()) {
      const HostGroup& G = groups[g_end];
      std::vector<MapKey> trial = keys;
      auto add = [&](const MapKey& k) {
        for (const auto& e : trial)
          if (e == k) return;
        trial.push_back(k);
      };
      for (const HostSeg& sg : G.segs) {
        add(key_of(sg.a, BM));
        add(key_of(stored(sg.b), b_box_rows(G)));
        if (G.dual) add(key_of(stored(sg.b2), b_box_rows(G)));
      }
      if ((int)(g_end - gi) + 1 > MAX_GROUPS || nsegs + (int)G.segs.size() > MAX_SEGS || (int)trial.size() > MAX_MAPS)
        break;
      keys.swap(trial);
      nsegs += (int)G.segs.size();
      ++g_end;
    }
    if (g_end == gi) return fail(DT_ERR_CAPACITY, "one GEMM group needs more than %d segments", MAX_SEGS);
    out->push_back({gi, g_end});
    gi = g_end;
  }
  return DT_OK;
}

// ---- the shape of one launch

int group_bn(const HostGroup& G) { return G.dual ? 128 : BN_MAX; }
int group_kiters(const HostGroup& G) {
  int k = 0;
  for (const HostSeg& sg : G.segs) k += (int)((sg.a.cols + BK - 1) / BK);
  return k;
}

struct LaunchShape {
  int tiles = 0;
  int m_tiles = 0;   // > 0: every group has this many M tiles
  int m_blocks = 1;  // row blocks (runs of groups with one N structure)
  int total_n = 0;   // N tiles over the groups of one row block
  int kiters = 0;    // K iterations of every tile when uniform
  bool uniform = true;
  bool dual = false;
};

LaunchShape launch_shape(const std::vector<HostGroup>& groups, size_t b, size_t e) {
  LaunchShape s;
  int common_m = -1;
  for (size_t g = b; g < e; ++g) {
    const HostGroup& G = groups[g];
    const int mt = (int)((G.m + PAIR_TILE_M - 1) / PAIR_TILE_M);
    const int nt = (int)((G.n + group_bn(G) - 1) / group_bn(G));
    s.tiles += mt * nt;
    s.total_n += nt;
    common_m = (common_m == -1 || common_m == mt) ? mt : -2;
    const int k = group_kiters(G);
    if (g == b) s.kiters = k;
    s.uniform = s.uniform && k == s.kiters;
    s.dual = s.dual || G.dual;
  }
  s.m_tiles = common_m > 0 ? common_m : 0;
  // row blocks: equal runs of groups by m_block whose N tiles match
  // position by position; then the M axis is the blocks end to end
  const size_t n = e - b;
  size_t run = 1;
  while (run < n && groups[b + run].m_block == groups[b].m_block) ++run;
  if (s.m_tiles > 0 && run < n && n % run == 0) {
    bool ok = true;
    for (size_t i = run; i < n && ok; ++i) {
      const HostGroup& G = groups[b + i];
      const HostGroup& F = groups[b + i % run];
      const HostGroup& P = groups[b + i - 1];
      ok = G.n == F.n && group_bn(G) == group_bn(F) && G.dual == F.dual &&
           (i % run == 0 ? G.m_block != P.m_block : G.m_block == P.m_block);
    }
    if (ok) {
      s.m_blocks = (int)(n / run);
      s.total_n = 0;
      for (size_t i = 0; i < run; ++i) s.total_n += (int)((groups[b + i].n + group_bn(groups[b + i]) - 1) / group_bn(groups[b + i]));
    }
  }
  return s;
}

// ---- split tail

// When the last wave would leave clusters idle, the remaining tiles' K
// iterations are divided over every cluster, where every tile has the same
// K and a cluster's share plus SPLIT_OVERHEAD_ITERS is shorter than a whole
// tile.  Finishing stages partials in shared memory, which bounds the
// pieces of one tile.
struct SplitPlan {
  int sk_tiles = 0;  // 0: every tile whole
  int kiters = 0;
  int pieces = 0;    // partial accumulators written
  int counters = 0;  // arrival counters (8 per tail tile: 2 CTAs x 4 row quarters)
};

SplitPlan plan_split(const LaunchShape& s, int ctas) {
  SplitPlan sp;
  if (s.tiles <= 0 || ctas <= 0 || !s.uniform || split_mode() == 0) return sp;
  const int rem = s.tiles % ctas;
  const int ki = s.kiters;
  const int64_t share_min = (int64_t)rem * ki / ctas;  // shortest share, in K iterations
  // most pieces one tile can have: the shares it meets
  const int np = share_min > 0 ? (int)((ki + share_min - 1) / share_min) + 1 : 0;
  const double split_cost = (double)rem * ki / ctas + SPLIT_OVERHEAD_ITERS;
  // the warp that finishes a tile reads every piece's partial back
  const bool fits = np <= FIN_MAX_PIECES;
  if (rem > 0 && share_min >= 8 && fits && (split_cost <= ki || split_mode() == 2)) {
    sp.sk_tiles = rem;
    sp.kiters = ki;
    sp.pieces = rem + ctas - 1;  // every cluster boundary inside the tail adds one
    sp.counters = 8 * rem;
  }
  return sp;
}

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }
size_t split_part_bytes(const SplitPlan& sp) { return round256((size_t)sp.pieces * 2 * BM * BN_MAX * sizeof(float)); }
size_t split_bytes(const SplitPlan& sp) {
  return sp.sk_tiles > 0 ? split_part_bytes(sp) + round256((size_t)sp.counters * sizeof(int32_t)) : 0;
}

// ---- tile order

// Band height and block width of a launch with common M tiles: bands whose
// A rows take about a quarter of L2, at least one wave high, each sweeping
// every N tile (band_n = total_n) in snake order; for long K (8192 and more,
// where one tile's A rows or B columns pass 4 MB) blocks of 8 M x 4 N tiles.
// Measured on GB300 with DT_GEMM_BANDS over 13 orders (blocks of 1..32 M
// tiles by 1..48 N tiles): the fused q/k/v ran fastest with 16-tile bands
// and lost 4-10% with 32-tile or 1-tile bands; the o projection gained 2.5%
// with 1-tile bands; the MLP down projection (K = 11008) moved by about 1%
// whatever the order, but 8 x 4 blocks cut its DRAM reads from 520 to 401 MB
// (ncu), so long-K launches take them.  No simple traffic model ranked the
// orders' times correctly.
void choose_bands(const std::vector<HostGroup>& groups, size_t b, size_t e, const LaunchShape& s, int ctas,
                  int* band_m, int* band_n) {
  *band_m = 1;
  *band_n = std::max(1, s.total_n);
  if (s.m_tiles <= 0) return;
  const int m_all = s.m_tiles * s.m_blocks;
  int om, on;
  if (bands_override(&om, &on)) {
    *band_m = std::min(om, m_all);
    *band_n = std::min(on, s.total_n);
    return;
  }
  int64_t max_k = 0;
  for (size_t g = b; g < e; ++g) max_k = std::max<int64_t>(max_k, (int64_t)group_kiters(groups[g]) * BK);
  const int64_t a_tile_bytes = (int64_t)PAIR_TILE_M * std::max<int64_t>(max_k, 1) * 2;
  if (max_k >= 8192) {
    *band_m = std::min(8, m_all);
    *band_n = std::min(4, *band_n);
    return;
  }
  int band = (int)std::max<int64_t>(1, (32ll << 20) / a_tile_bytes);
  band = std::max(band, (ctas + s.total_n - 1) / s.total_n);
  *band_m = std::max(1, std::min(band, m_all));
}

// ---- launches

dt_status run_tcgen05(const std::vector<HostGroup>& groups, int32_t* status, cudaStream_t stream, Workspace ws) {
  static thread_local Params p;
  const int ctas = pair_max_clusters();  // clusters in one wave
  if (ctas <= 0) return fail(DT_ERR_CUDA, "the tcgen05 GEMM cannot be launched on this device");
  std::vector<std::pair<size_t, size_t>> launches;
  dt_status st = pack_launches(groups, &launches);
  if (st != DT_OK) return st;
  for (const auto& range : launches) {
    const size_t gi = range.first, g_end = range.second;
    const LaunchShape shape = launch_shape(groups, gi, g_end);
    int map_i = 0, seg_i = 0, tiles = 0;
    std::vector<MapKey> encoded;
    // index of the descriptor for (matrix, box rows) in this launch, encoding it once
    auto map_index = [&](const Mat& m, int box, int32_t* idx) -> dt_status {
      const MapKey k = key_of(m, box);
      for (size_t i = 0; i < encoded.size(); ++i)
        if (encoded[i] == k) {
          *idx = (int32_t)i;
          return DT_OK;
        }
      if (map_i >= MAX_MAPS) return fail(DT_ERR_CAPACITY, "more than %d TMA descriptors in one launch", MAX_MAPS);
      dt_status e = encode_map(m, box, &p.maps[map_i]);
      if (e != DT_OK) return e;
      encoded.push_back(k);
      *idx = map_i++;
      return DT_OK;
    };
    p.ngroups = 0;
    for (size_t g = gi; g < g_end; ++g) {
      const HostGroup& H = groups[g];
      Group& G = p.groups[p.ngroups++];
      G.m = (int32_t)H.m;
      G.n = (int32_t)H.n;
      G.bn = group_bn(H);
      G.m_tiles = (int32_t)((H.m + PAIR_TILE_M - 1) / PAIR_TILE_M);
      G.n_tiles = (int32_t)((H.n + G.bn - 1) / G.bn);
      G.tile_begin = tiles;
      tiles += G.m_tiles * G.n_tiles;
      G.seg_begin = seg_i;
      G.seg_count = (int32_t)H.segs.size();
      G.dual = H.dual ? 1 : 0;
      G.out_dtype = H.out_dtype;
      G.nout = (int32_t)H.out_ptr.size();
      for (int j = 0; j < G.nout; ++j) {
        G.out_row_begin[j] = H.row_begin[j];
        G.out_ptr[j] = H.out_ptr[j];
        G.out_ld[j] = H.out_ld[j];
      }
      G.out_row_begin[G.nout] = H.m;
      G.bias = H.bias;
      G.bias_dtype = H.bias ? H.bias_dtype : -1;
      G.out_vec = out_vec_ok(H) ? 1 : 0;
      G.out_vec32 = out_vec32_ok(H) ? 1 : 0;
      G.b_kmajor = H.segs.empty() ? 0 : (H.segs[0].b.kmajor ? 1 : 0);
      for (const HostSeg& sg : H.segs) {
        Seg& S = p.segs[seg_i++];
        S.k_tiles = (int32_t)((sg.a.cols + BK - 1) / BK);
        S.last_steps = (int32_t)((sg.a.cols - (int64_t)(S.k_tiles - 1) * BK + 15) / 16);
        if ((st = map_index(sg.a, BM, &S.a_map)) != DT_OK) return st;
        if ((st = map_index(stored(sg.b), b_box_rows(H), &S.b_map)) != DT_OK) return st;
        S.b_map2 = S.b_map;
        if (H.dual && (st = map_index(stored(sg.b2), b_box_rows(H), &S.b_map2)) != DT_OK) return st;
      }
    }
    p.total_tiles = tiles;
    p.nmaps = map_i;
    p.nsegs = seg_i;
    p.status = status;
    p.wait_limit_ns = gemm_wait_limit_ns();
    p.starve = gemm_starve();
    // N tile prefix sums over one row block's groups (all groups when the
    // launch is one block)
    p.m_blocks = shape.m_blocks;
    p.n_tile_begin[0] = 0;
    for (int g = 0; g < p.ngroups / p.m_blocks; ++g) p.n_tile_begin[g + 1] = p.n_tile_begin[g] + p.groups[g].n_tiles;
    p.m_tiles = shape.m_tiles;
    choose_bands(groups, gi, g_end, shape, ctas, &p.band_m, &p.band_n);
    // the split tail, where the caller's workspace holds its scratch
    p.sk_tiles = 0;
    p.sk_kiters = 0;
    p.sk_part = nullptr;
    p.sk_count = nullptr;
    int grid = std::min(tiles, ctas);
    const SplitPlan sp = plan_split(shape, ctas);
    const size_t need = split_bytes(sp);
    int32_t* counters = nullptr;
    if (sp.sk_tiles > 0 && ws.ptr && ws.bytes >= need) {
      p.sk_tiles = sp.sk_tiles;
      p.sk_kiters = sp.kiters;
      p.sk_part = reinterpret_cast<float*>(ws.ptr);
      counters = reinterpret_cast<int32_t*>(ws.ptr + split_part_bytes(sp));
      p.sk_count = counters;
      grid = ctas;
    }
    if (tiles > 0) {
      if (counters) {
        // the counters start at zero in every launch: the workspace's
        // contents are the caller's between calls
        const size_t cbytes = (size_t)sp.counters * sizeof(int32_t);
        cudaError_t e = cudaMemsetAsync(counters, 0, cbytes, stream);
        if (e != cudaSuccess) return fail(DT_ERR_CUDA, "zeroing the split-tail counters: %s", cudaGetErrorString(e));
        if (g_grec) {
          GemmLaunch z;
          z.kind = 3;
          z.zero_ptr = counters;
          z.zero_bytes = cbytes;
          g_grec->launches.push_back(z);
        }
      }
      cudaError_t e = launch_tcgen05_pair(p, grid, stream);
      if (e != cudaSuccess) return fail(DT_ERR_CUDA, "tcgen05 GEMM launch: %s", cudaGetErrorString(e));
      count_launch();
      if (g_grec) {
        GemmLaunch l;
        l.kind = 0;
        l.grid = grid;
        l.params = std::make_shared<Params>(p);
        g_grec->launches.push_back(l);
      }
    }
  }
  return DT_OK;
}

dt_status run_simt(const std::vector<HostGroup>& groups, cudaStream_t stream) {
  static thread_local SParams p;
  const int sms = device_sm_count();
  size_t gi = 0;
  while (gi < groups.size()) {
    size_t g_end = gi;
    int nsegs = 0;
    while (g_end < groups.size() && (int)(g_end - gi) < MAX_GROUPS &&
           nsegs + (int)groups[g_end].segs.size() <= MAX_SEGS) {
      nsegs += (int)groups[g_end].segs.size();
      ++g_end;
    }
    if (g_end == gi) return fail(DT_ERR_CAPACITY, "one GEMM group needs more than %d segments", MAX_SEGS);
    int seg_i = 0, tiles = 0;
    p.ngroups = 0;
    for (size_t g = gi; g < g_end; ++g) {
      const HostGroup& H = groups[g];
      if (H.dual) return fail(DT_ERR_ALIGNMENT, "the gated MLP needs TMA-compatible bf16 operands");
      SGroup& G = p.groups[p.ngroups++];
      G.m = H.m;
      G.n = H.n;
      G.m_tiles = (int32_t)((H.m + S_TILE - 1) / S_TILE);
      G.n_tiles = (int32_t)((H.n + S_TILE - 1) / S_TILE);
      G.tile_begin = tiles;
      tiles += G.m_tiles * G.n_tiles;
      G.seg_begin = seg_i;
      G.seg_count = (int32_t)H.segs.size();
      G.out_dtype = H.out_dtype;
      G.nout = (int32_t)H.out_ptr.size();
      for (int j = 0; j < G.nout; ++j) {
        G.row_begin[j] = H.row_begin[j];
        G.out_ptr[j] = H.out_ptr[j];
        G.out_ld[j] = H.out_ld[j];
      }
      G.row_begin[G.nout] = H.m;
      G.bias = H.bias;
      G.bias_dtype = H.bias ? H.bias_dtype : -1;
      for (const HostSeg& s : H.segs) {
        SSeg& S = p.segs[seg_i++];
        S.a = s.a.ptr;
        S.b = s.b.ptr;
        S.lda = s.a.ld;
        S.ldb = s.b.ld;
        S.k = (int32_t)s.a.cols;
        S.dtype = s.a.dtype;
        S.b_kmajor = s.b.kmajor ? 1 : 0;
      }
    }
    p.total_tiles = tiles;
    if (tiles > 0) {
      const int grid = std::min(tiles, sms * 8);
      simt_gemm_kernel<<<grid, S_THREADS, 0, stream>>>(p);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return fail(DT_ERR_CUDA, "CUDA-core GEMM launch: %s", cudaGetErrorString(e));
      count_launch();
      g_simt_launches.fetch_add(1, std::memory_order_relaxed);
      if (g_grec) {
        GemmLaunch l;
        l.kind = 2;
        l.grid = grid;
        l.params = std::make_shared<SParams>(p);
        g_grec->launches.push_back(l);
      }
    }
    gi = g_end;
  }
  return DT_OK;
}

// Groups with output; a group with no K contributes bias (or zeros).
std::vector<HostGroup> live_groups(std::vector<HostGroup>& groups) {
  std::vector<HostGroup> live;
  live.reserve(groups.size());
  for (auto& g : groups) {
    if (g.m <= 0 || g.n <= 0) continue;
    std::vector<HostSeg> segs;
    for (auto& s : g.segs)
      if (s.a.cols > 0) segs.push_back(s);
    g.segs.swap(segs);
    live.push_back(std::move(g));
  }
  return live;
}

// true: the tcgen05 kernel can run every group (bf16 operands TMA can
// describe, one B major-ness per group)
bool tensor_core_ok(const std::vector<HostGroup>& live) {
  for (const auto& g : live) {
    if (g.segs.empty()) return false;
    for (const auto& s : g.segs) {
      if (!tma_ok(s.a) || !tma_ok(s.b) || (g.dual && !tma_ok(s.b2))) return false;
      if (s.b.kmajor != g.segs[0].b.kmajor || (g.dual && s.b2.kmajor != s.b.kmajor)) return false;
    }
  }
  return true;
}

dt_status check_limits(const std::vector<HostGroup>& live) {
  for (auto& g : live)
    if (g.out_ptr.size() > (size_t)MAX_OUT) return fail(DT_ERR_CAPACITY, "more than %d output row blocks", MAX_OUT);
  // M, N and the TMA and tile coordinates are 32-bit on the device: refuse a
  // dimension that would not fit (an [8, 2^31] bf16 activation is only
  // 32 GB) instead of truncating it
  constexpr int64_t DIM_LIMIT = (1ll << 31) - 512;
  for (const auto& g : live) {
    if (g.m > DIM_LIMIT || g.n > DIM_LIMIT)
      return fail(DT_ERR_CAPACITY, "GEMM output %lld x %lld: each dimension must be below 2^31 - 512", (long long)g.m,
                  (long long)g.n);
    for (const auto& sg : g.segs)
      if (sg.a.rows > DIM_LIMIT || sg.a.cols > DIM_LIMIT || sg.b.rows > DIM_LIMIT || sg.b.cols > DIM_LIMIT)
        return fail(DT_ERR_CAPACITY, "GEMM operand of %lld x %lld / %lld x %lld: each dimension must be below 2^31 - 512",
                    (long long)sg.a.rows, (long long)sg.a.cols, (long long)sg.b.rows, (long long)sg.b.cols);
  }
  return DT_OK;
}

}  // namespace

namespace {

// Operands TMA cannot describe (bf16 with a row pitch that is not a multiple
// of 16 bytes, or a base that is not 16-byte aligned: the shards of a dim
// torch.chunk splits unevenly), each given a copy in the workspace.
struct PadPlan {
  std::vector<PitchCopy> copies;
  size_t bytes = 0;  // the copies' share of the workspace (each 256-byte aligned)
  bool possible = true;  // every group could run on the tensor cores after padding
};

PadPlan plan_padding(std::vector<HostGroup>& live, char* base) {
  PadPlan pp;
  std::vector<std::pair<MapKey, Mat>> done;  // stored matrix -> its padded copy
  auto pad = [&](Mat& m) {
    if (tma_ok(m)) return;
    const Mat st = stored(m);
    if (st.dtype != DT_BF16 || st.rows <= 0 || st.cols <= 0 || st.ld < st.cols) {
      pp.possible = false;
      return;
    }
    const MapKey k = key_of(st, 0);
    for (const auto& e : done)
      if (e.first == k) {
        m.ptr = e.second.ptr;
        m.ld = e.second.ld;
        return;
      }
    PitchCopy c{};
    c.src = st.ptr;
    c.src_ld = st.ld;
    c.rows = st.rows;
    c.cols = st.cols;
    c.dst_ld = (st.cols + 7) & ~int64_t(7);
    c.dst = base + pp.bytes;
    pp.bytes += round256((size_t)c.rows * (size_t)c.dst_ld * 2);
    const int64_t gx = (st.cols + 8 * 256 - 1) / (8 * 256);
    c.grid_x = (int)gx;
    c.grid_y = (int)std::max<int64_t>(1, std::min<int64_t>(st.rows, std::max<int64_t>(1, 4096 / gx)));
    pp.copies.push_back(c);
    Mat padded = m;
    padded.ptr = c.dst;
    padded.ld = c.dst_ld;
    done.push_back({k, padded});
    m.ptr = c.dst;
    m.ld = c.dst_ld;
  };
  for (auto& g : live) {
    for (auto& sg : g.segs) {
      if (sg.a.kmajor) pp.possible = false;
      pad(sg.a);
      pad(sg.b);
      if (g.dual) pad(sg.b2);
      if (sg.b.kmajor != g.segs[0].b.kmajor || (g.dual && sg.b2.kmajor != sg.b.kmajor)) pp.possible = false;
    }
    if (g.segs.empty()) pp.possible = false;
  }
  return pp;
}

}  // namespace

dt_status run_groups(std::vector<HostGroup>& groups, int32_t* d_status, cudaStream_t stream, Workspace ws) {
  std::vector<HostGroup> live = live_groups(groups);
  if (live.empty()) return DT_OK;
  dt_status st = check_limits(live);
  if (st != DT_OK) return st;
  bool tc = tensor_core_ok(live);
  if (!tc && ws.ptr) {
    // bf16 operands with pitches TMA cannot describe: copy them into the
    // workspace with one it can, when the workspace holds the copies
    std::vector<HostGroup> padded = live;
    const PadPlan pp = plan_padding(padded, ws.ptr);
    if (pp.possible && pp.bytes <= ws.bytes && tensor_core_ok(padded)) {
      for (const PitchCopy& c : pp.copies) {
        cudaError_t e = launch_pitch_copy(c, stream);
        if (e != cudaSuccess) return fail(DT_ERR_CUDA, "operand copy: %s", cudaGetErrorString(e));
        count_launch();
        if (g_grec) {
          GemmLaunch l;
          l.kind = 4;
          l.pc = c;
          g_grec->launches.push_back(l);
        }
      }
      live.swap(padded);
      ws.ptr += pp.bytes;
      ws.bytes -= pp.bytes;
      tc = true;
    }
  }
  if (tc) {
    int32_t* status = device_status_word(d_status);
    if (!status) return fail(DT_ERR_CUDA, "no device status word");
    return run_tcgen05(live, status, stream, ws);
  }
  return run_simt(live, stream);
}

dt_status workspace_bytes(std::vector<HostGroup>& groups, size_t* bytes) {
  *bytes = 0;
  std::vector<HostGroup> live = live_groups(groups);
  if (live.empty()) return DT_OK;
  dt_status st = check_limits(live);
  if (st != DT_OK) return st;
  size_t pad_bytes = 0;
  if (!tensor_core_ok(live)) {
    // the padded copies, placed from a 256-aligned base (only their sizes matter here)
    const PadPlan pp = plan_padding(live, reinterpret_cast<char*>(uintptr_t(256)));
    if (!pp.possible || !tensor_core_ok(live)) return DT_OK;  // the CUDA-core kernel needs no workspace
    pad_bytes = pp.bytes;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return fail(DT_ERR_CUDA, "no CUDA device: the split tail's scratch depends on the device's SM count");
  }
  const int ctas = pair_max_clusters();
  if (ctas <= 0) return fail(DT_ERR_CUDA, "the tcgen05 GEMM cannot be launched on device %d", dev);
  std::vector<std::pair<size_t, size_t>> launches;
  if ((st = pack_launches(live, &launches)) != DT_OK) return st;
  size_t split = 0;
  for (const auto& r : launches)  // launches run one after the other: one scratch serves all
    split = std::max(split, split_bytes(plan_split(launch_shape(live, r.first, r.second), ctas)));
  *bytes = pad_bytes + split;
  return DT_OK;
}

uint64_t cuda_core_launches() { return g_simt_launches.load(std::memory_order_relaxed); }

GemmRecordScope::GemmRecordScope(GemmRecord* r) { g_grec = r; }
GemmRecordScope::~GemmRecordScope() { g_grec = nullptr; }
std::shared_ptr<GemmRecord> new_gemm_record() { return std::make_shared<GemmRecord>(); }

dt_status replay_gemm(const GemmRecord& r, cudaStream_t stream) {
  for (const GemmLaunch& l : r.launches) {
    cudaError_t e;
    if (l.kind == 3) {
      e = cudaMemsetAsync(l.zero_ptr, 0, l.zero_bytes, stream);
      if (e != cudaSuccess) return fail(DT_ERR_CUDA, "zeroing the split-tail counters: %s", cudaGetErrorString(e));
      continue;
    }
    if (l.kind == 4) {
      e = launch_pitch_copy(l.pc, stream);
      if (e != cudaSuccess) return fail(DT_ERR_CUDA, "operand copy: %s", cudaGetErrorString(e));
      count_launch();
      continue;
    }
    if (l.kind == 2) {
      simt_gemm_kernel<<<l.grid, S_THREADS, 0, stream>>>(*static_cast<const SParams*>(l.params.get()));
      e = cudaGetLastError();
      g_simt_launches.fetch_add(1, std::memory_order_relaxed);
    } else {
      e = launch_tcgen05_pair(*static_cast<const Params*>(l.params.get()), l.grid, stream);
    }
    if (e != cudaSuccess) return fail(DT_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
    count_launch();
  }
  return DT_OK;
}

}  // namespace gemm
}  // namespace dt

extern "C" dt_status dt_clear_cache(void) {
  {
    std::lock_guard<std::mutex> lk(dt::gemm::g_map_mu);
    dt::gemm::g_maps.clear();
  }
  dt::clear_redistribute_plans();
  dt::clear_gemm_plans();
  return DT_OK;
}

extern "C" uint64_t dt_cuda_core_gemm_count(void) { return dt::gemm::cuda_core_launches(); }
