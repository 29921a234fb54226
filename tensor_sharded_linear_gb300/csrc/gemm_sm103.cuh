// Device side of the tensor-parallel GEMM for sm_103a: tcgen05 MMA with the
// accumulator in tensor memory (TMEM), operands staged in shared memory by
// TMA, persistent CTA pairs (clusters of two) with warp-specialised roles.
//
// Problem description: a list of GROUPS, each an independent output tile
// grid, and per group a list of K SEGMENTS, each one (A, B) pair of TMA
// descriptors.  A tile accumulates every segment of its group, in order, in
// fp32 in TMEM.  This one shape covers
//   column parallel  (wineandchord "Column parallel", Y_i = X W_i):
//                    one group per shard, one segment each;
//   row parallel     (wineandchord "Row parallel", Y = sum_i X_i W_i):
//                    one group, one segment per shard -- the Partial sum
//                    never leaves the accumulator;
//   gated MLP        two B descriptors per segment (gate, up) whose tiles sit
//                    side by side in smem, so one N=256 MMA fills both halves
//                    of the accumulator and the epilogue forms SiLU(g) * u.
//
// Operand layouts: A is K-major (row-major [M, K] activations), B is
// MN-major (row-major [K, N] weights, the [in, out] convention) or K-major
// (a transposed view of [out, in] storage), all with the 128-byte swizzle
// that TMA writes and the MMA reads.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dt.h"
#include "gemm_plan.h"  // Params and its capacities
#include "ptx_sm103.cuh"

namespace dt {
namespace gemm {

constexpr int BM = 128;                       // accumulator rows = TMEM lanes
constexpr int BN_MAX = 256;                   // accumulator columns per buffer
constexpr int BK = 64;                        // 64 bf16 = one 128-byte swizzle row
constexpr int B_CHUNK_BYTES = 64 * BK * 2;    // 8 KiB: 64 N columns x 64 K rows
constexpr int TMEM_COLS = 512;                // two 256-column accumulators
constexpr int GROUP_M = 8;                    // per-group raster: 8 M tiles per band
constexpr int MAX_OUT = 8;

struct Seg {
  int32_t a_map, b_map, b_map2, k_tiles;
  int32_t last_steps;  // 16-deep MMA steps of the last K tile that hold data (1..4)
};

struct Group {
  int32_t m, n, m_tiles, n_tiles;
  int32_t tile_begin, seg_begin, seg_count, bn;  // bn: output columns per tile
  int32_t dual, out_dtype, nout, bias_dtype;     // bias_dtype < 0: no bias
  int32_t out_vec, b_kmajor, out_vec32, pad2;    // out_vec / out_vec32: 16- / 32-byte stores
                                                 // allowed; b_kmajor: B stored [N, K] (K contiguous)
  const void* bias;
  int64_t out_row_begin[MAX_OUT + 1];  // output row blocks: rows [begin[j], begin[j+1]) -> out j
  char* out_ptr[MAX_OUT];
  int64_t out_ld[MAX_OUT];  // elements
};

// Every launch's description travels in its parameter block.  Its size
// costs launch time, so a launch whose tables fit the compact capacities
// (ParamsSmall, ~8 KB) uses them and only large launches take Params (~25 KB).
template <int NMAPS, int NSEGS, int NGROUPS>
struct ParamsT {  // CUtensorMap carries its own 128-byte alignment
  static constexpr int kMaps = NMAPS, kSegs = NSEGS, kGroups = NGROUPS;
  CUtensorMap maps[NMAPS];
  Seg segs[NSEGS];
  Group groups[NGROUPS];
  int32_t n_tile_begin[NGROUPS + 1];  // prefix sums of the groups' N tiles
  int32_t nmaps, nsegs;               // entries of maps and segs in use
  int32_t ngroups, total_tiles;
  int32_t m_tiles;  // > 0: every group has this many M tiles, rastered together
  int32_t m_blocks; // row blocks: groups [b * ngroups / m_blocks, ...) hold rows block b
  int32_t band_m;   // M tiles per raster band
  int32_t band_n;   // N tiles (across groups) per block of a band
  int32_t starve;   // test hook: producers issue no loads, so every MMA wait runs out
  unsigned long long wait_limit_ns;  // bound of every mbarrier wait
  int32_t* status;
  // Split tail (pair kernel only).  The last sk_tiles tiles are not given to
  // clusters whole: their sk_tiles * sk_kiters K iterations are divided
  // evenly over all clusters, and each (cluster, tile) piece accumulates
  // its K range on its own.  Every piece writes its fp32 accumulator to
  // sk_part; the warp whose arrival completes a tile's count (sk_count,
  // one counter per tile, CTA and 32-row quarter, zeroed before the launch)
  // reads every piece's partial back, adds them in K order and runs the
  // tile's epilogue for its 32 rows.
  int32_t sk_tiles;   // 0: every tile whole
  int32_t sk_kiters;  // K iterations of every tile (uniform when sk_tiles > 0)
  float* sk_part;     // [piece][2 CTAs][128 rows][256 columns]
  int32_t* sk_count;  // [sk_tiles][2 CTAs][4 quarters]
};
using ParamsSmall = ParamsT<24, 32, 16>;
static_assert(sizeof(Params) <= 32000, "GEMM parameter block over the launch limit");

// ---------------------------------------------------------------- tcgen05 helpers

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // version
  d |= 2ull << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: fp32 D, bf16 A and B, A K-major,
// B MN-major ([in, out] weights) or K-major ([out, in] weights), M x N.
__host__ __device__ constexpr uint32_t instr_desc(int m, int n, bool b_kmajor = false) {
  return (1u << 4)                                 // D format: f32
         | (1u << 7)                               // A format: bf16
         | (1u << 10)                              // B format: bf16
         | (0u << 15)                              // A K-major
         | ((b_kmajor ? 0u : 1u) << 16)            // B major-ness
         | (static_cast<uint32_t>(n >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);  // M / 16
}

// ---------------------------------------------------------------- CTA-pair helpers
// A cluster of two CTAs shares one MMA (tcgen05 .cta_group::2): rank 0 issues
// it, each CTA holds half the operands and its half of the accumulator.

constexpr int PAIR_STAGES = 6;
constexpr int PAIR_A_BYTES = BM * BK * 2;           // this CTA's 128 rows of A: 16 KiB
constexpr int PAIR_B_BYTES = 128 * BK * 2;          // this CTA's 128 columns of B: 16 KiB
constexpr int PAIR_STAGE_BYTES = PAIR_A_BYTES + PAIR_B_BYTES;
constexpr int PAIR_BAR_BYTES = 512;  // barriers and flags
constexpr int PAIR_SMEM_BYTES = PAIR_STAGES * PAIR_STAGE_BYTES + 1024 + PAIR_BAR_BYTES;
// Most pieces a split tile may have: the warp that finishes it reads every
// piece's partial from L2, so this bounds the finishing time.
constexpr int FIN_MAX_PIECES = 8;
constexpr int PAIR_TILE_M = 2 * BM;                 // rows of one pair tile
constexpr int PAIR_B_PRODUCER_WARP = 6;             // after warps 0 (A), 1 (MMA), 2..5 (epilogue)
constexpr int PAIR_THREADS = 32 * (PAIR_B_PRODUCER_WARP + 1);

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Address, in the cluster's shared window, of the same object in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t cta_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(cta_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load into this CTA's smem whose completion is counted on an mbarrier
// that may live in the peer CTA (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Issued by one warp in EACH CTA of the pair.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem of both CTAs] (+)= A[smem of both] * B[smem of both]; issued by rank 0.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at this smem offset in every CTA of `mask`
// when all tcgen05 operations issued so far by this thread complete.
__device__ __forceinline__ void mma_commit_pair_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ---------------------------------------------------------------- tile helpers

struct TileCoord {
  int g, m0, n0;
};

// Tile order of a launch whose groups all have the same M tiles (all groups
// of a column-parallel launch share x; a row-parallel launch is one group):
// the groups' N tiles form one axis of total_n tiles.  When x is split into
// row blocks (a token-sharded input: one group per (row block, weight
// shard)), the launch holds m_blocks runs of groups with the same N
// structure, and the M axis is the blocks' M tiles end to end: the tiles
// form the same grid as the one GEMM they are parts of.  Tiles go in bands of
// band_m M tiles; a band is cut into blocks of band_n N tiles, visited in
// order, with M fastest inside a block; odd bands sweep N backwards, so
// consecutive bands start on the B panels the previous one ended on.
// Concurrent clusters then share the A rows and B columns of a compact
// block of tiles.  Returns the M tile and the N tile across groups.
__host__ __device__ __forceinline__ void band_order(int t, int m_tiles, int total_n, int band_m, int band_n, int* mi,
                                                    int* jn) {
  const int span = band_m * total_n;
  const int mb = t / span;
  const int first_m = mb * band_m;
  const int gm = m_tiles - first_m < band_m ? m_tiles - first_m : band_m;
  const int r = t - mb * span;
  const int blk = gm * band_n;
  const int nb = r / blk;
  const int r2 = r - nb * blk;
  int j = nb * band_n + r2 / gm;
  if (mb & 1) j = total_n - 1 - j;
  *mi = first_m + r2 % gm;
  *jn = j;
}

// Tile t of a launch.  With common M tiles, band_order; otherwise each
// group is rastered on its own in bands of GROUP_M M tiles.
template <int TILE_M, class P>
__device__ __forceinline__ TileCoord decode_tile(const P& p, int t) {
  if (p.m_tiles > 0) {
    const int gpb = p.ngroups / p.m_blocks;  // groups per row block
    int mi, jn;
    band_order(t, p.m_tiles * p.m_blocks, p.n_tile_begin[gpb], p.band_m, p.band_n, &mi, &jn);
    const int mb = mi / p.m_tiles;
    // the group holding N tile jn: binary search of the prefix sums (a
    // launch may hold 48 groups, e.g. sequence-parallel q/k/v)
    int lo = 0, hi = gpb - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.n_tile_begin[mid] <= jn) lo = mid;
      else hi = mid - 1;
    }
    const int g = mb * gpb + lo;
    return TileCoord{g, (mi - mb * p.m_tiles) * TILE_M, (jn - p.n_tile_begin[lo]) * p.groups[g].bn};
  }
  int lo = 0, hi = p.ngroups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.groups[mid].tile_begin <= t) lo = mid;
    else hi = mid - 1;
  }
  const int g = lo;
  const Group& G = p.groups[g];
  const int local = t - G.tile_begin;
  const int span = GROUP_M * G.n_tiles;
  const int first_m = (local / span) * GROUP_M;
  const int gm = min(GROUP_M, G.m_tiles - first_m);
  const int r = local % span;
  return TileCoord{g, (first_m + r % gm) * TILE_M, (r / gm) * G.bn};
}

// ---------------------------------------------------------------- work list
// What one cluster does, in order: its share [b(cid), b(cid + 1)) of the
// split tail's K iterations, b(c) = c * I / ncl, I = sk_tiles * sk_kiters,
// then whole tiles cid, cid + ncl, ... below the tail.  The host only
// splits when a share is shorter than a tile, so a share covers the end of
// one tail tile and the start of the next at most: one piece each.  The
// piece of tail tile s done by cluster c has id s + c, unique because both
// grow along the K axis.
struct Work {
  int t;       // tile
  int k0, k1;  // K iterations [k0, k1) of the tile
  int piece;   // < 0: the whole tile, finished directly
  int s;       // tail tile index (pieces only)
};

__device__ __forceinline__ int64_t sk_bound(int c, int64_t total, int ncl) { return (int64_t)c * total / ncl; }

struct WorkIter {
  int cid, ncl, t_dp, dp_end, kiters;
  int64_t it, it_end;
  template <class P>
  __device__ WorkIter(const P& p, int cid_, int ncl_) : cid(cid_), ncl(ncl_) {
    dp_end = p.total_tiles - p.sk_tiles;
    t_dp = cid;
    kiters = p.sk_kiters;
    const int64_t total = (int64_t)p.sk_tiles * p.sk_kiters;
    it = p.sk_tiles > 0 ? sk_bound(cid, total, ncl) : 0;
    it_end = p.sk_tiles > 0 ? sk_bound(cid + 1, total, ncl) : 0;
  }
  // The cluster's pieces of the split tail come first, then its whole
  // tiles: a tail tile is complete early in the launch, and the warp that
  // finishes it does so while its pair's MMAs run the whole tiles.
  __device__ bool next(Work* w) {
    if (it < it_end) {
      const int s = (int)(it / kiters);
      const int k0 = (int)(it - (int64_t)s * kiters);
      const int64_t k1_wide = k0 + (it_end - it);
      const int k1 = k1_wide < kiters ? (int)k1_wide : kiters;
      w->t = dp_end + s;
      w->k0 = k0;
      w->k1 = k1;
      w->piece = s + cid;
      w->s = s;
      it += k1 - k0;
      return true;
    }
    if (t_dp < dp_end) {
      w->t = t_dp;
      w->k0 = 0;
      w->k1 = 1 << 30;
      w->piece = -1;
      w->s = -1;
      t_dp += ncl;
      return true;
    }
    return false;
  }
};

// A piece's fp32 accumulator in sk_part, per (CTA, 32-row quarter): 8
// column chunks x 8 float4 x 32 lanes, so every warp access to it moves
// 512 contiguous bytes (lane = accumulator row within the quarter).
template <class P>
__device__ __forceinline__ float4* sk_slot(const P& p, int piece, uint32_t rank, int quarter) {
  return reinterpret_cast<float4*>(p.sk_part) + ((static_cast<size_t>(piece) * 2 + rank) * 4 + quarter) * (8 * 8 * 32);
}

// Clusters whose shares meet tail tile s: [c_first, c_last].
template <class P>
__device__ __forceinline__ void sk_tile_clusters(const P& p, int ncl, int s, int* c_first, int* c_last) {
  const int64_t total = (int64_t)p.sk_tiles * p.sk_kiters;
  const int64_t lo = (int64_t)s * p.sk_kiters, hi = lo + p.sk_kiters;  // [lo, hi)
  const int64_t c_est = lo * ncl / total;
  int c = c_est < ncl - 1 ? (int)c_est : ncl - 1;
  while (c + 1 < ncl && sk_bound(c + 1, total, ncl) <= lo) ++c;
  while (c > 0 && sk_bound(c, total, ncl) > lo) --c;
  *c_first = c;
  int e = c;
  while (e + 1 < ncl && sk_bound(e + 1, total, ncl) < hi) ++e;
  *c_last = e;
}

// Gated-MLP pair tile: columns of gate (and of up) it holds, a multiple of
// 32 up to 128.  The MMA is 2 * that wide; gate fills accumulator columns
// [0, h) and up [h, 2h), so a shard's short last tile does no wasted work.
__device__ __forceinline__ int pair_dual_half(const Group& G, int n0) {
  const int r = (G.n - n0 + 31) & ~31;
  return r < 128 ? r : 128;
}

__device__ __forceinline__ float bias_at(const Group& G, int col) {
  if (G.bias_dtype == DT_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(G.bias)[col]);
  return reinterpret_cast<const float*>(G.bias)[col];
}

// One 32-byte store (address 32-byte aligned).  A lane's run of 32 output
// columns goes out as two (bf16) or four (fp32) of these, each a whole
// 32-byte sector, where the rows allow it: 16-byte stores wrote every sector
// in two halves from two instructions, and the o projection took 3% longer
// (q/k/v 2%, the MLP 1%).
__device__ __forceinline__ void st_global_v8(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t e,
                                             uint32_t f, uint32_t g, uint32_t h) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d),
               "r"(e), "r"(f), "r"(g), "r"(h)
               : "memory");
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Store the NW words w (a run of 4 * NW bytes, elements of ES bytes) at
// address `a`, which is ES-aligned and H bytes short of a 16-byte boundary:
// the first H bytes element by element, then whole 16-byte vectors shifted
// out of the words, then the remaining elements.  Output rows whose pitch is
// not a multiple of 16 bytes (an uneven shard of a column layer) get 16-byte
// stores this way instead of one store per element.
template <int ES, int NW, int H>
__device__ __forceinline__ void store_words_at(char* a, const uint32_t (&w)[NW]) {
  constexpr int NB = NW * 4;
  constexpr int NV = (NB - H) / 16;
  auto elem = [&](int b) -> uint32_t {  // the element at byte b of the run
    return ES == 4 ? w[b >> 2] : (w[b >> 2] >> ((b & 3) * 8)) & 0xffffu;
  };
#pragma unroll
  for (int b = 0; b < H; b += ES) {
    if (ES == 4) *reinterpret_cast<uint32_t*>(a + b) = elem(b);
    else *reinterpret_cast<uint16_t*>(a + b) = static_cast<uint16_t>(elem(b));
  }
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int b = H + 16 * j;
    const int q = b >> 2, sh = (b & 3) * 8;
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = sh ? __funnelshift_r(w[q + k], w[q + k + 1], sh) : w[q + k];
    *reinterpret_cast<uint4*>(a + b) = make_uint4(o[0], o[1], o[2], o[3]);
  }
#pragma unroll
  for (int b = H + 16 * NV; b < NB; b += ES) {
    if (ES == 4) *reinterpret_cast<uint32_t*>(a + b) = elem(b);
    else *reinterpret_cast<uint16_t*>(a + b) = static_cast<uint16_t>(elem(b));
  }
}

// Store 32 fp32 values of one output row at columns [col0, col0 + 32).
__device__ __forceinline__ void store_row32(const Group& G, char* row_ptr, int col0, const float (&v)[32]) {
  const int valid = min(32, G.n - col0);
  if (valid <= 0) return;
  if (G.out_dtype == DT_BF16) {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(row_ptr) + col0;
    if (valid == 32 && G.out_vec32) {
#pragma unroll
      for (int q = 0; q < 2; ++q)
        st_global_v8(o + 16 * q, pack2(v[16 * q + 0], v[16 * q + 1]), pack2(v[16 * q + 2], v[16 * q + 3]),
                     pack2(v[16 * q + 4], v[16 * q + 5]), pack2(v[16 * q + 6], v[16 * q + 7]),
                     pack2(v[16 * q + 8], v[16 * q + 9]), pack2(v[16 * q + 10], v[16 * q + 11]),
                     pack2(v[16 * q + 12], v[16 * q + 13]), pack2(v[16 * q + 14], v[16 * q + 15]));
    } else if (valid == 32 && G.out_vec) {
      uint4* o4 = reinterpret_cast<uint4*>(o);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        o4[q] = make_uint4(pack2(v[8 * q + 0], v[8 * q + 1]), pack2(v[8 * q + 2], v[8 * q + 3]),
                           pack2(v[8 * q + 4], v[8 * q + 5]), pack2(v[8 * q + 6], v[8 * q + 7]));
    } else if (valid == 32) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = pack2(v[2 * i], v[2 * i + 1]);
      char* a = reinterpret_cast<char*>(o);
      switch ((16 - (reinterpret_cast<uintptr_t>(a) & 15)) & 15) {
        case 0: store_words_at<2, 16, 0>(a, w); break;
        case 2: store_words_at<2, 16, 2>(a, w); break;
        case 4: store_words_at<2, 16, 4>(a, w); break;
        case 6: store_words_at<2, 16, 6>(a, w); break;
        case 8: store_words_at<2, 16, 8>(a, w); break;
        case 10: store_words_at<2, 16, 10>(a, w); break;
        case 12: store_words_at<2, 16, 12>(a, w); break;
        default: store_words_at<2, 16, 14>(a, w); break;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < valid) o[i] = __float2bfloat16_rn(v[i]);
    }
  } else {
    float* o = reinterpret_cast<float*>(row_ptr) + col0;
    if (valid == 32 && G.out_vec32) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_global_v8(o + 8 * q, __float_as_uint(v[8 * q]), __float_as_uint(v[8 * q + 1]), __float_as_uint(v[8 * q + 2]),
                     __float_as_uint(v[8 * q + 3]), __float_as_uint(v[8 * q + 4]), __float_as_uint(v[8 * q + 5]),
                     __float_as_uint(v[8 * q + 6]), __float_as_uint(v[8 * q + 7]));
    } else if (valid == 32 && G.out_vec) {
      float4* o4 = reinterpret_cast<float4*>(o);
#pragma unroll
      for (int q = 0; q < 8; ++q) o4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else if (valid == 32) {
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
      char* a = reinterpret_cast<char*>(o);
      switch ((16 - (reinterpret_cast<uintptr_t>(a) & 15)) & 15) {
        case 0: store_words_at<4, 32, 0>(a, w); break;
        case 4: store_words_at<4, 32, 4>(a, w); break;
        case 8: store_words_at<4, 32, 8>(a, w); break;
        default: store_words_at<4, 32, 12>(a, w); break;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < valid) o[i] = v[i];
    }
  }
}

// Epilogue of 32 accumulator columns of one row: bias, cast, store.
__device__ __forceinline__ void finish_chunk(const Group& G, char* row_ptr, int col0, float (&v)[32]) {
  if (G.bias_dtype >= 0) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int col = col0 + i;
      if (col < G.n) v[i] += bias_at(G, col);
    }
  }
  store_row32(G, row_ptr, col0, v);
}

// Gated-MLP epilogue of 32 columns of one row: SiLU(g) * u in fp32, cast, store.
__device__ __forceinline__ void finish_dual(const Group& G, char* row_ptr, int col0, const float (&g)[32],
                                            const float (&u)[32]) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = g[i] / (1.0f + __expf(-g[i])) * u[i];
  store_row32(G, row_ptr, col0, v);
}

// ---------------------------------------------------------------- split tiles
// A piece's partial in sk_part, as seen by one lane: 8 float4 (32 columns of
// its row) 32 float4 apart; consecutive pieces' partials SK_PIECE_F4 apart.
constexpr size_t SK_PIECE_F4 = 2 * 4 * 8 * 8 * 32;

// v = the sum, in piece (K) order, of np pieces' 32 columns for this lane's
// row, read from L2 (the pieces were written by other SMs) two pieces at a
// time, so 16 loads are in flight per lane.
__device__ __forceinline__ void sum_pieces(const float4* src, int np, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 x = __ldcg(src + i * 32);
    v[4 * i] = x.x;
    v[4 * i + 1] = x.y;
    v[4 * i + 2] = x.z;
    v[4 * i + 3] = x.w;
  }
  for (int q = 1; q < np; q += 2) {
    const float4* a = src + q * SK_PIECE_F4;
    const bool two = q + 1 < np;
    float4 xa[8], xb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) xa[i] = __ldcg(a + i * 32);
    if (two) {
#pragma unroll
      for (int i = 0; i < 8; ++i) xb[i] = __ldcg(a + SK_PIECE_F4 + i * 32);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[4 * i] += xa[i].x;
      v[4 * i + 1] += xa[i].y;
      v[4 * i + 2] += xa[i].z;
      v[4 * i + 3] += xa[i].w;
    }
    if (two) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[4 * i] += xb[i].x;
        v[4 * i + 1] += xb[i].y;
        v[4 * i + 2] += xb[i].z;
        v[4 * i + 3] += xb[i].w;
      }
    }
  }
}

// Finishes split tile tc for one epilogue warp's 32 rows (this lane's row
// at row_ptr, null when past the last row): the np pieces first_piece ...
// are added in K order and the sums take the tile's normal epilogue.
template <class P>
__device__ __noinline__ void finish_split_tile(const P& p, const Group& G, const TileCoord& tc, char* row_ptr,
                                               int first_piece, int np, uint32_t rank, int quarter, int lane) {
  const float4* src = sk_slot(p, first_piece, rank, quarter) + lane;
  if (!G.dual) {
    const int nrounds = min(8, (G.n - tc.n0 + 31) >> 5);
    for (int rd = 0; rd < nrounds; ++rd) {
      float v[32];
      sum_pieces(src + rd * 8 * 32, np, v);
      if (row_ptr) finish_chunk(G, row_ptr, tc.n0 + rd * 32, v);
    }
  } else {
    // gate in accumulator columns [0, hh), up in [hh, 2 hh)
    const int hc = pair_dual_half(G, tc.n0) >> 5;
    for (int rd = 0; rd < hc; ++rd) {
      float g[32], u[32];
      sum_pieces(src + rd * 8 * 32, np, g);
      sum_pieces(src + (rd + hc) * 8 * 32, np, u);
      if (row_ptr) finish_dual(G, row_ptr, tc.n0 + rd * 32, g, u);
    }
  }
}

}  // namespace gemm
}  // namespace dt
