// The tensor-parallel GEMM on CTA pairs: a cluster of two CTAs computes one
// 256 x 256 tile with tcgen05.mma.cta_group::2 (M = 256: each CTA holds its
// 128 rows of A and 128 of the 256 columns of B, and its 128 rows of the
// accumulator in its own TMEM).  Per SM this stages 32 KiB per 64-deep K
// step instead of 48 KiB for a 128 x 256 single-CTA tile, which halves the
// B traffic into each SM and leaves room for 6 pipeline stages.
//
// Roles per CTA (224 threads): warp 0 TMA producer of A, warp 6 TMA producer
// of B, warp 1 MMA issuer (rank 0 only; it owns the pair's MMAs) and TMEM
// allocator, warps 2..5 epilogue (one accumulator row per thread).  The
// producer and MMA warps run their loops with all 32 lanes, waits included,
// and one elected lane issues the copies, MMAs and commits: the same loops
// run by lane 0 alone, inside a branch on the lane, took 5-7% longer (the
// issuing thread's time between stages shows up as tensor-pipe idle time).  Two
// producers because one thread issuing every copy capped the copies alone
// at ~46 B/clk per SM (the issuing thread blocks ~110 cycles per copy);
// split, the copies alone run 16-20% faster and the GEMMs ~1%.
// Barriers:
//   full[s]    in rank 0: 1 arrival (rank 0's A producer, with the byte
//              count of both CTAs' loads) + the loads' bytes.  Every
//              other producer only issues its loads: its bytes are its
//              share.  (A cluster-scope release arrive from rank 1 before
//              each stage would wait for that thread's copies still in
//              flight and serialise rank 1's pipeline.)
//   empty[s]   in each CTA: 1 arrival, rank 0's MMA commit multicast to both
//              (both producers of a CTA wait on it);
//   tfull[b]   in each CTA: 1 arrival, multicast commit after a tile's MMAs;
//   tempty[b]  in rank 0: 8 arrivals, the 4 epilogue warps of each CTA.
// Every wait is bounded (Params::wait_limit_ns); on expiry the role raises
// the CTA's abort flag, the launch reports DT_DEV_ERR_TIMEOUT and unwinds.
// Split tail (Params::sk_tiles > 0): a cluster runs its pieces of the tail
// tiles first, then its whole tiles; a piece's epilogue writes its fp32
// partial to the workspace and counts it, and the warp whose count completes
// a tail tile adds every piece's partial (read from L2, in K order) and runs
// the tile's epilogue, while the pair's MMAs move on.  No wait involves
// another cluster.
#include <algorithm>

#include "gemm_plan.h"
#include "gemm_sm103.cuh"

namespace dt {
namespace gemm {

template <class P>
__global__ void __launch_bounds__(PAIR_THREADS, 1) tcgen05_gemm_pair_kernel(const __grid_constant__ P p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + PAIR_STAGES * PAIR_STAGE_BYTES);
  uint64_t* empty = full + PAIR_STAGES;
  uint64_t* tfull = empty + PAIR_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(nclusters_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < PAIR_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, TMEM_COLS);
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised, TMEM of both allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool leader = elect_one();

  bool aborted = false;

  if (warp == 0 || warp == PAIR_B_PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producers (both CTAs)
    // warp 0 loads this CTA's A rows (and, in rank 0, arms the stage's
    // barrier for every byte of both CTAs); the B producer loads its B
    // columns.  Both walk the same stages and wait on the same `empty`.
    const bool loads_a = warp == 0;
    {
      for (int i = 0; leader && i < p.ngroups; ++i) {
        const Group& G = p.groups[i];
        for (int s = G.seg_begin; s < G.seg_begin + G.seg_count && s < G.seg_begin + 2; ++s)
          prefetch_map(&p.maps[loads_a ? p.segs[s].a_map : p.segs[s].b_map]);
      }
      int stage = 0;
      uint32_t phase = 0;
      WorkIter wi(p, cid, ncl);
      Work w;
      while (!aborted && !p.starve && wi.next(&w)) {
        const TileCoord tc = decode_tile<PAIR_TILE_M>(p, w.t);
        const Group& G = p.groups[tc.g];
        const int a_row = tc.m0 + static_cast<int>(rank) * BM;
        // this CTA's B columns: plain tiles split N in halves; the gated MLP
        // puts gate (rank 0) and up (rank 1) side by side
        const int b_col = G.dual ? tc.n0 : tc.n0 + static_cast<int>(rank) * 128;
        int kbase = 0;  // K iterations of the tile before segment si
        for (int si = G.seg_begin; si < G.seg_begin + G.seg_count && !aborted; ++si) {
          const Seg& S = p.segs[si];
          const CUtensorMap* bmap = &p.maps[(G.dual && rank == 1) ? S.b_map2 : S.b_map];
          const int kt_end = min(S.k_tiles, w.k1 - kbase);
          for (int kt = max(0, w.k0 - kbase); kt < kt_end; ++kt) {
            if (!mbar_wait_warp(&empty[stage], phase ^ 1u, abort_flag, p.wait_limit_ns)) {
              aborted = true;
              *abort_flag = 1;
              break;
            }
            const uint32_t full0 = mapa_shared(smem_u32(&full[stage]), 0);
            uint8_t* a = smem + stage * PAIR_STAGE_BYTES;
            uint8_t* b = a + PAIR_A_BYTES;
            if (leader) {
              if (loads_a) {
                if (rank == 0) mbar_expect_tx(&full[stage], 2 * PAIR_STAGE_BYTES);
                tma_load_2d_pair(a, &p.maps[S.a_map], kt * BK, a_row, full0);
              } else if (G.b_kmajor) {
                tma_load_2d_pair(b, bmap, kt * BK, b_col, full0);  // 128 N rows of 64 K
              } else {
                tma_load_2d_pair(b, bmap, b_col, kt * BK, full0);
                tma_load_2d_pair(b + B_CHUNK_BYTES, bmap, b_col + 64, kt * BK, full0);
              }
            }
            if (++stage == PAIR_STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          kbase += S.k_tiles;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t tphase = 0;
      const uint32_t a_base = smem_u32(smem);
      WorkIter wi(p, cid, ncl);
      Work w;
      while (!aborted && wi.next(&w)) {
        const TileCoord tc = decode_tile<PAIR_TILE_M>(p, w.t);
        const Group& G = p.groups[tc.g];
        const bool bk = G.b_kmajor != 0;
        const uint32_t idesc = instr_desc(PAIR_TILE_M, G.dual ? 2 * pair_dual_half(G, tc.n0) : 256, bk);
        if (!mbar_wait_warp(&tempty[buf], tphase ^ 1u, abort_flag, p.wait_limit_ns)) {
          aborted = true;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN_MAX);
        uint32_t acc = 0;
        int kbase = 0;
        for (int si = G.seg_begin; si < G.seg_begin + G.seg_count && !aborted; ++si) {
          const int kts = p.segs[si].k_tiles;
          const int last_steps = p.segs[si].last_steps;
          const int kt_end = min(kts, w.k1 - kbase);
          for (int kt = max(0, w.k0 - kbase); kt < kt_end; ++kt) {
            if (!mbar_wait_warp(&full[stage], phase, abort_flag, p.wait_limit_ns)) {
              aborted = true;
              *abort_flag = 1;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = a_base + stage * PAIR_STAGE_BYTES;
            const uint32_t b_addr = a_addr + PAIR_A_BYTES;
            const int nsteps = kt == kts - 1 ? last_steps : BK / 16;  // the K tail past the data is zero fill
            if (leader) {
#pragma unroll
              for (int j = 0; j < BK / 16; ++j) {
                if (j >= nsteps) break;
                // 16-deep K steps: A advances 32 bytes inside its 128-byte
                // swizzle rows; an MN-major B half is two 64-column chunks
                // 8 KiB apart, a K-major one advances like A
                const uint64_t adesc = smem_desc(a_addr + j * 32, 16, 1024);
                const uint64_t bdesc =
                    bk ? smem_desc(b_addr + j * 32, 16, 1024) : smem_desc(b_addr + j * 2048, B_CHUNK_BYTES, 1024);
                mma_bf16_pair(d_tmem, adesc, bdesc, idesc, acc | static_cast<uint32_t>(j));
              }
              mma_commit_pair_mc(&empty[stage], 0x3);
            }
            acc = 1;
            if (++stage == PAIR_STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          kbase += kts;
        }
        if (aborted) break;
        if (leader) mma_commit_pair_mc(&tfull[buf], 0x3);
        if (++buf == 2) {
          buf = 0;
          tphase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t tempty0[2] = {mapa_shared(smem_u32(&tempty[0]), 0), mapa_shared(smem_u32(&tempty[1]), 0)};
    int buf = 0;
    uint32_t tphase = 0;
    WorkIter wi(p, cid, ncl);
    Work w;
    while (wi.next(&w)) {
      const TileCoord tc = decode_tile<PAIR_TILE_M>(p, w.t);
      const Group& G = p.groups[tc.g];
      // the whole warp waits: tcgen05.ld below is warp-collective
      if (!mbar_wait_warp(&tfull[buf], tphase, abort_flag, p.wait_limit_ns)) {
        aborted = true;
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int64_t r = tc.m0 + static_cast<int>(rank) * BM + row_in_tile;
      char* row_ptr = nullptr;
      if (r < G.m) {
        int j = 0;
        while (j + 1 < G.nout && G.out_row_begin[j + 1] <= r) ++j;
        const int esize = G.out_dtype == DT_BF16 ? 2 : 4;
        row_ptr = G.out_ptr[j] + (r - G.out_row_begin[j]) * G.out_ld[j] * esize;
      }
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * BN_MAX);
      // accumulator columns that hold outputs (the gated MLP: gate [0, hh), up [hh, 2 hh))
      const int hh = G.dual ? pair_dual_half(G, tc.n0) : 0;
      const int ncols = G.dual ? 2 * hh : min(256, (G.n - tc.n0 + 31) & ~31);
      if (w.piece < 0) {
        if (!G.dual) {
          for (int c = 0; c < ncols; c += 32) {
            uint32_t raw[32];
            tmem_ld32(tbase + c, raw);
            tmem_ld_wait();
            if (row_ptr) {
              float v[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]);
              finish_chunk(G, row_ptr, tc.n0 + c, v);
            }
          }
        } else {
          for (int c = 0; c < hh; c += 32) {
            uint32_t g[32], u[32];
            tmem_ld32(tbase + c, g);
            tmem_ld32(tbase + hh + c, u);
            tmem_ld_wait();
            if (row_ptr) {
              float gv[32], uv[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                gv[i] = __uint_as_float(g[i]);
                uv[i] = __uint_as_float(u[i]);
              }
              finish_dual(G, row_ptr, tc.n0 + c, gv, uv);
            }
          }
        }
      } else {
        // a piece of a split tile: this warp's 32 accumulator rows go to the
        // piece's slot in sk_part (L2 only), then TMEM is released
        float4* mine = sk_slot(p, w.piece, rank, quarter) + lane;
        for (int c = 0; c < ncols; c += 32) {
          uint32_t raw[32];
          tmem_ld32(tbase + c, raw);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            __stcg(mine + ((c >> 5) * 8 + q) * 32,
                   make_float4(__uint_as_float(raw[4 * q]), __uint_as_float(raw[4 * q + 1]),
                               __uint_as_float(raw[4 * q + 2]), __uint_as_float(raw[4 * q + 3])));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0[buf]);
      if (++buf == 2) {
        buf = 0;
        tphase ^= 1u;
      }
      if (w.piece >= 0) {
        // the warp whose arrival completes this tile's count (its CTA and
        // row quarter) finishes the tile now, while the pair's MMAs move on
        __threadfence();  // this lane's partial before the count
        __syncwarp();
        int c_first = 0, c_last = 0, last = 0;
        if (lane == 0) {
          sk_tile_clusters(p, ncl, w.s, &c_first, &c_last);
          int* cnt = p.sk_count + (w.s * 2 + static_cast<int>(rank)) * 4 + quarter;
          last = atomicAdd(cnt, 1) == c_last - c_first ? 1 : 0;
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
          __threadfence();  // every piece's partial after the count
          const int first_piece = w.s + __shfl_sync(0xffffffffu, c_first, 0);
          const int np = __shfl_sync(0xffffffffu, c_last, 0) - __shfl_sync(0xffffffffu, c_first, 0) + 1;
          finish_split_tile(p, G, tc, row_ptr, first_piece, np, rank, quarter, lane);
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  if (aborted && lane == 0) atomicOr(p.status, DT_DEV_ERR_TIMEOUT);
  if ((warp == 0 || warp == PAIR_B_PRODUCER_WARP) && leader && aborted) {
    // copies this CTA issued count on rank 0's barrier; give them a bounded
    // time to land before the pair leaves
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 20000000ull) {
    }
  }
  if (warp == 1 && leader && rank == 0) {
    // every MMA of the pair has completed before either CTA frees TMEM
    mma_commit_pair(drain);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < 100000000ull) {
    }
  }
  tc_fence_before();
  cluster_sync();  // no CTA leaves while its peer may still touch its smem or TMEM
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

namespace {

void pair_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int clusters, cudaStream_t stream) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = dim3(2 * clusters, 1, 1);
  cfg->blockDim = dim3(PAIR_THREADS, 1, 1);
  cfg->dynamicSmemBytes = PAIR_SMEM_BYTES;
  cfg->stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

int g_max_clusters[64] = {};

}  // namespace

// Clusters that can be resident at once.  The kernel is persistent with a
// static tile assignment, so launching more than this would run the extra
// clusters as a second wave; SMs whose TPC partner is fused off cannot host
// a pair, so this can be below SMs / 2.  Both parameter-block sizes get the
// shared-memory opt-in here (same resources, so the same count).
int pair_max_clusters() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!g_max_clusters[dev]) {
    if (cudaFuncSetAttribute(tcgen05_gemm_pair_kernel<Params>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PAIR_SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(tcgen05_gemm_pair_kernel<ParamsSmall>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PAIR_SMEM_BYTES) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    pair_config(&cfg, attr, 1, nullptr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tcgen05_gemm_pair_kernel<Params>, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return 0;
    }
    g_max_clusters[dev] = n;
  }
  return g_max_clusters[dev];
}

cudaError_t launch_tcgen05_pair(const Params& p, int clusters, cudaStream_t stream) {
  if (pair_max_clusters() <= 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pair_config(&cfg, attr, clusters, stream);
  if (p.nmaps <= ParamsSmall::kMaps && p.nsegs <= ParamsSmall::kSegs && p.ngroups <= ParamsSmall::kGroups) {
    static thread_local ParamsSmall ps;
    std::copy(p.maps, p.maps + p.nmaps, ps.maps);
    std::copy(p.segs, p.segs + p.nsegs, ps.segs);
    std::copy(p.groups, p.groups + p.ngroups, ps.groups);
    std::copy(p.n_tile_begin, p.n_tile_begin + p.ngroups + 1, ps.n_tile_begin);
    ps.nmaps = p.nmaps;
    ps.nsegs = p.nsegs;
    ps.ngroups = p.ngroups;
    ps.total_tiles = p.total_tiles;
    ps.m_tiles = p.m_tiles;
    ps.m_blocks = p.m_blocks;
    ps.band_m = p.band_m;
    ps.band_n = p.band_n;
    ps.starve = p.starve;
    ps.wait_limit_ns = p.wait_limit_ns;
    ps.status = p.status;
    ps.sk_tiles = p.sk_tiles;
    ps.sk_kiters = p.sk_kiters;
    ps.sk_part = p.sk_part;
    ps.sk_count = p.sk_count;
    return cudaLaunchKernelEx(&cfg, tcgen05_gemm_pair_kernel<ParamsSmall>, ps);
  }
  return cudaLaunchKernelEx(&cfg, tcgen05_gemm_pair_kernel<Params>, p);
}

}  // namespace gemm
}  // namespace dt
