// Lowering of batched GEMM groups to a launch: TMA descriptors (cached on
// the host), tile counts, and the choice between the tcgen05 kernel and the
// CUDA-core kernel (fp32 operands, or bf16 operands whose pitches TMA
// cannot describe).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <unordered_map>

#include "gemm_plan.h"
#include "gemm_sm103.cuh"

namespace dt {
namespace gemm {

struct GemmLaunch {
  int kind = 0;  // 0 pair kernel, 1 single-CTA kernel, 2 CUDA-core kernel
  int grid = 0;
  std::shared_ptr<void> params;  // a heap Params (kinds 0, 1; keeps its 128-byte alignment) or SParams
};
struct GemmRecord {
  std::vector<GemmLaunch> launches;
};

namespace {

#ifdef DT_GEMM_TRACE
__device__ unsigned long long g_trace[1024 * TRACE_SLOTS];
unsigned long long* trace_ptr() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_trace) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<unsigned long long*>(ptr);
}
#endif

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

// Split-tail scratch, one per (device, stream): the pieces' fp32 partial
// accumulators and the tiles' arrival counters.  Made on the first split
// launch on that stream outside a stream capture (cudaMalloc, then the
// counters zeroed on that stream) and kept until dt_clear_cache.  Every
// launch that completes leaves the counters at zero again.
struct SplitScratch {
  float* part = nullptr;
  int32_t* count = nullptr;
  int pieces = 0, counters = 0;
};
std::mutex g_split_mu;
std::map<std::pair<int, uintptr_t>, SplitScratch> g_split;
thread_local int g_no_alloc = 0;
thread_local GemmRecord* g_grec = nullptr;

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

// ------------------------------------------------------------ lowering

bool out_vec_ok(const HostGroup& g) {
  const int esize = g.out_dtype == DT_BF16 ? 2 : 4;
  for (size_t j = 0; j < g.out_ptr.size(); ++j) {
    if (reinterpret_cast<uintptr_t>(g.out_ptr[j]) % 16) return false;
    if ((g.out_ld[j] * esize) % 16) return false;
  }
  return true;
}

// The CTA-pair kernel (256 x 256 tiles on tcgen05 .cta_group::2) is the
// default; DT_GEMM_PAIR=0 in the environment selects the single-CTA kernel
// (128 x 256 tiles), e.g. to compare the two.
// Test hooks, read once from the environment: DT_GEMM_WAIT_LIMIT_MS bounds
// every mbarrier wait (default 2000 ms); DT_GEMM_STARVE=1 makes the TMA
// producers issue no loads, so the MMA waits run out and the kernels report
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
// iterations of one 256 x 256 pair tile (~0.3 us each): writing the pieces'
// partials, finishing the tiles, and the tail's operand traffic squeezed
// into a fraction of a tile's time.  Measured on GB300 at about 20-25 us
// per launch (the TP MLP down projection gains 15 us; 64-iteration tiles
// lose 7-20 us).
constexpr double SPLIT_OVERHEAD_ITERS = 72.0;

// DT_GEMM_SPLIT=0 in the environment turns the split tail off (every tile
// whole), e.g. to compare the two schedules.
bool use_split_tail() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("DT_GEMM_SPLIT");
    v = (e && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}

// Scratch for `pieces` partial tiles and `counters` counters on this
// device and stream; nullptr inside a NoAllocScope, inside a stream
// capture, once MAX_SPLIT_STREAMS (device, stream) pairs hold one, or when
// the allocation fails (the launch then runs every tile whole).
constexpr size_t MAX_SPLIT_STREAMS = 16;  // ~39 MB each
const SplitScratch* split_scratch(cudaStream_t stream, int pieces, int counters) {
  if (g_no_alloc) return nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(g_split_mu);
  auto key = std::make_pair(dev, reinterpret_cast<uintptr_t>(stream));
  auto it = g_split.find(key);
  if (it != g_split.end() && it->second.pieces >= pieces && it->second.counters >= counters) return &it->second;
  if (it != g_split.end()) return nullptr;  // sized once, for the largest split a launch can make
  if (g_split.size() >= MAX_SPLIT_STREAMS) return nullptr;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return nullptr;  // no allocation inside a capture; a later uncaptured launch makes the scratch
  }
  // the largest split: fewer tail tiles than clusters, so fewer than twice
  // the clusters pieces and eight counters per tail tile
  const int cl = std::max(pair_max_clusters(), 1);
  SplitScratch sc;
  sc.pieces = std::max(pieces, 2 * cl);
  sc.counters = std::max(counters, 8 * cl);
  if (cudaMalloc(&sc.part, (size_t)sc.pieces * 2 * BM * BN_MAX * sizeof(float)) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  // zeroed on the launch's own stream, so it precedes every launch that uses it
  if (cudaMalloc(&sc.count, (size_t)sc.counters * sizeof(int32_t)) != cudaSuccess ||
      cudaMemsetAsync(sc.count, 0, (size_t)sc.counters * sizeof(int32_t), stream) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(sc.part);
    if (sc.count) cudaFree(sc.count);
    return nullptr;
  }
  return &(g_split[key] = sc);
}

bool use_pair_kernel() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("DT_GEMM_PAIR");
    v = (e && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}

dt_status run_tcgen05(std::vector<HostGroup>& groups, int32_t* status, cudaStream_t stream) {
  static thread_local Params p;
  const int sms = device_sm_count();
  const int max_clusters = use_pair_kernel() ? pair_max_clusters() : 0;
  const bool pair = max_clusters > 0;
  const int tile_m = pair ? PAIR_TILE_M : BM;
  const int ctas = pair ? max_clusters : sms;  // CTAs (single) or clusters (pair) in one wave
  size_t gi = 0;
  while (gi < groups.size()) {
    // pack as many groups as fit one parameter block; descriptors of the
    // same matrix and box (e.g. x shared by every column shard) are shared
    auto b_rows = [&](const HostGroup& G) { return G.segs.empty() || !G.segs[0].b.kmajor ? BK : ((pair || G.dual) ? 128 : 256); };
    std::vector<MapKey> keys;
    auto key_of = [](const Mat& m, int box) {
      return MapKey{reinterpret_cast<uintptr_t>(m.ptr), m.rows, m.cols, m.ld, box};
    };
    auto count_new = [&](const HostGroup& G, std::vector<MapKey>* ks) {
      int added = 0;
      auto add = [&](const MapKey& k) {
        for (const auto& e : *ks)
          if (e == k) return;
        ks->push_back(k);
        ++added;
      };
      for (const HostSeg& s : G.segs) {
        add(key_of(s.a, BM));
        add(key_of(stored(s.b), b_rows(G)));
        if (G.dual) add(key_of(stored(s.b2), b_rows(G)));
      }
      return added;
    };
    size_t g_end = gi;
    int nsegs = 0;
    while (g_end < groups.size()) {
      const HostGroup& G = groups[g_end];
      const int need_segs = (int)G.segs.size();
      std::vector<MapKey> trial = keys;
      count_new(G, &trial);
      if ((int)(g_end - gi) + 1 > MAX_GROUPS || nsegs + need_segs > MAX_SEGS || (int)trial.size() > MAX_MAPS) break;
      keys.swap(trial);
      nsegs += need_segs;
      ++g_end;
    }
    if (g_end == gi) return fail(DT_ERR_CAPACITY, "one GEMM group needs more than %d segments", MAX_SEGS);
    // 256-column tiles: one N=256 MMA per 16-deep K step reads each A row
    // once for 256 outputs (128-wide tiles re-read A and halve the MMA work
    // per pipeline stage)
    const int bn = BN_MAX;
    int map_i = 0, seg_i = 0, tiles = 0;
    std::vector<MapKey> encoded;
    // index of the descriptor for (matrix, box rows) in this launch, encoding it once
    auto map_index = [&](const Mat& m, int box, int32_t* idx) -> dt_status {
      const MapKey k{reinterpret_cast<uintptr_t>(m.ptr), m.rows, m.cols, m.ld, box};
      for (size_t i = 0; i < encoded.size(); ++i)
        if (encoded[i] == k) {
          *idx = (int32_t)i;
          return DT_OK;
        }
      if (map_i >= MAX_MAPS) return fail(DT_ERR_CAPACITY, "more than %d TMA descriptors in one launch", MAX_MAPS);
      dt_status st = encode_map(m, box, &p.maps[map_i]);
      if (st != DT_OK) return st;
      encoded.push_back(k);
      *idx = map_i++;
      return DT_OK;
    };
    p.ngroups = 0;
    int common_m = -1;
    int64_t max_k = 0;
    for (size_t g = gi; g < g_end; ++g) {
      const int mt = (int)((groups[g].m + tile_m - 1) / tile_m);
      common_m = (common_m == -1 || common_m == mt) ? mt : -2;
      int64_t k = 0;
      for (const HostSeg& s : groups[g].segs) k += s.a.cols;
      max_k = std::max(max_k, k);
    }
    for (size_t g = gi; g < g_end; ++g) {
      const HostGroup& H = groups[g];
      Group& G = p.groups[p.ngroups++];
      G.m = (int32_t)H.m;
      G.n = (int32_t)H.n;
      G.bn = H.dual ? 128 : bn;
      G.m_tiles = (int32_t)((H.m + tile_m - 1) / tile_m);
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
      G.b_kmajor = H.segs.empty() ? 0 : (H.segs[0].b.kmajor ? 1 : 0);
      // K-major B boxes: 128 N rows per CTA of a pair or per gated-MLP half,
      // 256 for a plain single-CTA tile; MN-major B boxes: 64 K rows
      const int b_box_rows = G.b_kmajor ? ((pair || H.dual) ? 128 : 256) : BK;
      for (const HostSeg& s : H.segs) {
        Seg& S = p.segs[seg_i++];
        S.k_tiles = (int32_t)((s.a.cols + BK - 1) / BK);
        dt_status st;
        if ((st = map_index(s.a, BM, &S.a_map)) != DT_OK) return st;
        if ((st = map_index(stored(s.b), b_box_rows, &S.b_map)) != DT_OK) return st;
        S.b_map2 = S.b_map;
        if (H.dual && (st = map_index(stored(s.b2), b_box_rows, &S.b_map2)) != DT_OK) return st;
      }
    }
    p.total_tiles = tiles;
    p.nmaps = map_i;
    p.nsegs = seg_i;
    p.status = status;
    p.wait_limit_ns = gemm_wait_limit_ns();
    p.starve = gemm_starve();
#ifdef DT_GEMM_TRACE
    p.trace = trace_ptr();
#else
    p.trace = nullptr;
#endif
    p.n_tile_begin[0] = 0;
    for (int g = 0; g < p.ngroups; ++g) p.n_tile_begin[g + 1] = p.n_tile_begin[g] + p.groups[g].n_tiles;
    p.m_tiles = common_m > 0 ? common_m : 0;
    // band height: the band's A rows (band_m x 128 x K bf16) take about a
    // quarter of L2, and a band holds at least one wave of tiles
    {
      const int64_t a_tile_bytes = (int64_t)tile_m * std::max<int64_t>(max_k, 1) * 2;
      int band = (int)std::max<int64_t>(1, (32ll << 20) / a_tile_bytes);
      const int total_n = std::max(1, p.n_tile_begin[p.ngroups]);
      band = std::max(band, (ctas + total_n - 1) / total_n);
      p.band_m = std::max(1, std::min(band, p.m_tiles > 0 ? p.m_tiles : 1));
    }
    // Split tail: when the last wave would leave clusters idle, divide the
    // remaining tiles' K iterations over every cluster, where every tile has
    // the same K and a cluster's share plus SPLIT_OVERHEAD_ITERS is shorter
    // than a whole tile.  The finishing stages partials in shared memory,
    // which bounds the pieces of a tile.
    p.sk_tiles = 0;
    p.sk_kiters = 0;
    p.sk_part = nullptr;
    p.sk_count = nullptr;
    int grid = std::min(tiles, ctas);
    if (pair && tiles > 0 && use_split_tail()) {
      int ki = -1;
      bool uniform = true;
      for (int g = 0; g < p.ngroups; ++g) {
        int k = 0;
        for (int si = p.groups[g].seg_begin; si < p.groups[g].seg_begin + p.groups[g].seg_count; ++si)
          k += p.segs[si].k_tiles;
        if (ki < 0) ki = k;
        uniform = uniform && k == ki;
      }
      bool dual = false;
      for (int g = 0; g < p.ngroups; ++g) dual = dual || p.groups[g].dual;
      const int rem = tiles % ctas;
      const int64_t share_min = (int64_t)rem * ki / ctas;  // shortest share, in K iterations
      // most pieces one tile can have: the shares it meets
      const int np = share_min > 0 ? (int)((ki + share_min - 1) / share_min) + 1 : 0;
      const double split_cost = (double)rem * ki / ctas + SPLIT_OVERHEAD_ITERS;
      // a finishing round stages one 32-column chunk of every piece (gate
      // and up chunks for the gated MLP) in an epilogue warp's half of its
      // shared-memory quarter
      const bool fits = np * (dual ? 2 : 1) <= FIN_MAX_PIECES;
      if (uniform && rem > 0 && share_min >= 8 && fits && split_cost <= ki) {
        const SplitScratch* sc = split_scratch(stream, rem + ctas - 1, 8 * rem);
        if (sc) {
          p.sk_tiles = rem;
          p.sk_kiters = ki;
          p.sk_part = sc->part;
          p.sk_count = sc->count;
          grid = ctas;
        }
      }
    }
    if (tiles > 0) {
      cudaError_t e = pair ? launch_tcgen05_pair(p, grid, stream) : launch_tcgen05(p, grid, stream);
      if (e != cudaSuccess) return fail(DT_ERR_CUDA, "tcgen05 GEMM launch: %s", cudaGetErrorString(e));
      count_launch();
      if (g_grec) g_grec->launches.push_back({pair ? 0 : 1, grid, std::make_shared<Params>(p)});
    }
    gi = g_end;
  }
  return DT_OK;
}

dt_status run_simt(std::vector<HostGroup>& groups, cudaStream_t stream) {
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
      if (g_grec) g_grec->launches.push_back({2, grid, std::make_shared<SParams>(p)});
    }
    gi = g_end;
  }
  return DT_OK;
}

}  // namespace

dt_status run_groups(std::vector<HostGroup>& groups, int32_t* d_status, cudaStream_t stream) {
  // drop groups with no output; a group with no K contributes bias (or zeros)
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
  if (live.empty()) return DT_OK;
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
  bool tc = true;
  for (const auto& g : live) {
    if (g.segs.empty()) tc = false;
    for (const auto& s : g.segs) {
      if (!tma_ok(s.a) || !tma_ok(s.b) || (g.dual && !tma_ok(s.b2))) tc = false;
      // one B major-ness per group (the kernel decides it per tile)
      if (s.b.kmajor != g.segs[0].b.kmajor || (g.dual && s.b2.kmajor != s.b.kmajor)) tc = false;
    }
  }
  if (tc) {
    int32_t* status = device_status_word(d_status);
    if (!status) return fail(DT_ERR_CUDA, "no device status word");
    return run_tcgen05(live, status, stream);
  }
  return run_simt(live, stream);
}

}  // namespace gemm
}  // namespace dt

#ifdef DT_GEMM_TRACE
// Traced builds only: copy (and optionally clear) the per-CTA wait records.
extern "C" __attribute__((visibility("default"))) int dt_gemm_trace_read(unsigned long long* out, int n, int clear) {
  using dt::gemm::g_trace;
  if (n > 1024 * dt::gemm::TRACE_SLOTS) n = 1024 * dt::gemm::TRACE_SLOTS;
  if (cudaMemcpyFromSymbol(out, g_trace, n * sizeof(unsigned long long)) != cudaSuccess) return -1;
  if (clear) {
    static unsigned long long zeros[1024 * dt::gemm::TRACE_SLOTS] = {};
    if (cudaMemcpyToSymbol(g_trace, zeros, sizeof(zeros)) != cudaSuccess) return -1;
  }
  return n;
}
#endif

namespace dt {
namespace gemm {

NoAllocScope::NoAllocScope() { ++g_no_alloc; }
NoAllocScope::~NoAllocScope() { --g_no_alloc; }
bool gemm_no_alloc() { return g_no_alloc > 0; }

GemmRecordScope::GemmRecordScope(GemmRecord* r) { g_grec = r; }
GemmRecordScope::~GemmRecordScope() { g_grec = nullptr; }
std::shared_ptr<GemmRecord> new_gemm_record() { return std::make_shared<GemmRecord>(); }

dt_status replay_gemm(const GemmRecord& r, cudaStream_t stream) {
  for (const GemmLaunch& l : r.launches) {
    cudaError_t e;
    if (l.kind == 2) {
      simt_gemm_kernel<<<l.grid, S_THREADS, 0, stream>>>(*static_cast<const SParams*>(l.params.get()));
      e = cudaGetLastError();
    } else {
      const Params& p = *static_cast<const Params*>(l.params.get());
      e = l.kind == 0 ? launch_tcgen05_pair(p, l.grid, stream) : launch_tcgen05(p, l.grid, stream);
    }
    if (e != cudaSuccess) return fail(DT_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
    count_launch();
  }
  return DT_OK;
}

// After a launch gave up (DT_DEV_ERR_TIMEOUT) its tiles' arrival counters
// may be left part-counted; zero every counter so later launches start clean.
void reset_split_counters() {
  std::lock_guard<std::mutex> lk(g_split_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_split) {
    cudaSetDevice(kv.first.first);
    cudaDeviceSynchronize();  // no launch may still be counting
    cudaMemset(kv.second.count, 0, (size_t)kv.second.counters * sizeof(int32_t));
    cudaDeviceSynchronize();  // zero before any later launch on any stream
  }
  cudaSetDevice(cur);
}

}  // namespace gemm
}  // namespace dt

extern "C" dt_status dt_clear_cache(void) {
  {
    std::lock_guard<std::mutex> lk(dt::gemm::g_map_mu);
    dt::gemm::g_maps.clear();
  }
  dt::clear_redistribute_plans();
  dt::clear_gemm_plans();  // their parameters point into the scratch freed below
  std::lock_guard<std::mutex> lk(dt::gemm::g_split_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : dt::gemm::g_split) {
    cudaSetDevice(kv.first.first);
    cudaFree(kv.second.part);  // waits for the device's work first
    cudaFree(kv.second.count);
  }
  dt::gemm::g_split.clear();
  cudaSetDevice(cur);
  return DT_OK;
}
