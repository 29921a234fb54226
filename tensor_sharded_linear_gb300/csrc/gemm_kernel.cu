// Persistent warp-specialised tcgen05 GEMM (see gemm_sm103.cuh for the
// roles and the problem description) and its launcher.
#include "gemm_sm103.cuh"
#include "gemm_plan.h"

namespace dt {
namespace gemm {

__global__ void __launch_bounds__(THREADS, 1) tcgen05_gemm_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
#ifdef DT_GEMM_TRACE
  volatile long long* t_issue = reinterpret_cast<volatile long long*>(drain + 2);   // per stage
  volatile long long* t_commit = t_issue + STAGES;
  for (int i = threadIdx.x; i < 2 * STAGES; i += blockDim.x) t_issue[i] = 0;
#endif

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  bool aborted = false;
#ifdef DT_GEMM_TRACE
  const long long _trace_start = clock64();
#endif
  int8_t issued_parity[STAGES];
#pragma unroll
  for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int i = 0; i < p.ngroups; ++i) {
        const Group& G = p.groups[i];
        for (int s = G.seg_begin; s < G.seg_begin + G.seg_count && s < G.seg_begin + 2; ++s) {
          prefetch_map(&p.maps[p.segs[s].a_map]);
          prefetch_map(&p.maps[p.segs[s].b_map]);
        }
      }
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < p.total_tiles && !aborted && !p.starve; t += gridDim.x) {
        const TileCoord tc = decode_tile<BM>(p, t);
        const Group& G = p.groups[tc.g];
        const int nmma = tile_mma_n(G, tc.n0);
        const int nchunks = (nmma + 63) / 64;
        // K-major B arrives as one 256-row box (two 128-row boxes for the
        // gated MLP); MN-major B as 64-column chunks
        const uint32_t bytes = A_TILE_BYTES + (G.b_kmajor ? B_TILE_BYTES : nchunks * B_CHUNK_BYTES);
        for (int si = G.seg_begin; si < G.seg_begin + G.seg_count && !aborted; ++si) {
          const Seg& S = p.segs[si];
          for (int kt = 0; kt < S.k_tiles; ++kt) {
            bool _ok;
            {
              DT_TRACE_T0();
              _ok = mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.wait_limit_ns);
              DT_TRACE_ADD(TR_PROD_EMPTY);
#ifdef DT_GEMM_TRACE
              if (p.trace && t_commit[stage] != 0)
                atomicAdd(&p.trace[blockIdx.x * TRACE_SLOTS + TR_COMMIT_LAT],
                          (unsigned long long)(clock64() - t_commit[stage]));
              t_issue[stage] = clock64();
#endif
            }
            if (!_ok) {
              aborted = true;
              *abort_flag = 1;
              break;
            }
            mbar_expect_tx(&full[stage], bytes);
            uint8_t* a = smem + stage * STAGE_BYTES;
            uint8_t* b = a + A_TILE_BYTES;
            tma_load_2d(a, &p.maps[S.a_map], kt * BK, tc.m0, &full[stage]);
            if (G.b_kmajor) {
              if (!G.dual) {
                tma_load_2d(b, &p.maps[S.b_map], kt * BK, tc.n0, &full[stage]);
              } else {
                tma_load_2d(b, &p.maps[S.b_map], kt * BK, tc.n0, &full[stage]);
                tma_load_2d(b + B_TILE_BYTES / 2, &p.maps[S.b_map2], kt * BK, tc.n0, &full[stage]);
              }
            } else if (!G.dual) {
              for (int c = 0; c < nchunks; ++c)
                tma_load_2d(b + c * B_CHUNK_BYTES, &p.maps[S.b_map], tc.n0 + 64 * c, kt * BK, &full[stage]);
            } else {
              for (int c = 0; c < 2; ++c) {
                tma_load_2d(b + c * B_CHUNK_BYTES, &p.maps[S.b_map], tc.n0 + 64 * c, kt * BK, &full[stage]);
                tma_load_2d(b + (2 + c) * B_CHUNK_BYTES, &p.maps[S.b_map2], tc.n0 + 64 * c, kt * BK, &full[stage]);
              }
            }
            issued_parity[stage] = static_cast<int8_t>(phase);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t tphase = 0;
      const uint32_t a_base = smem_u32(smem);
      for (int t = blockIdx.x; t < p.total_tiles && !aborted; t += gridDim.x) {
        const TileCoord tc = decode_tile<BM>(p, t);
        const Group& G = p.groups[tc.g];
        const uint32_t idesc = instr_desc(BM, tile_mma_n(G, tc.n0), G.b_kmajor != 0);
        const bool bk = G.b_kmajor != 0;
        bool _ok;
        {
          DT_TRACE_T0();
          _ok = mbar_wait(&tempty[buf], tphase ^ 1u, abort_flag, p.wait_limit_ns);
          DT_TRACE_ADD(TR_MMA_TEMPTY);
        }
        DT_TRACE_COUNT(TR_TILES);
        if (!_ok) {
          aborted = true;
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN_MAX);
        uint32_t acc = 0;
        for (int si = G.seg_begin; si < G.seg_begin + G.seg_count && !aborted; ++si) {
          const int kts = p.segs[si].k_tiles;
          for (int kt = 0; kt < kts; ++kt) {
            bool _okf;
            {
              DT_TRACE_T0();
              _okf = mbar_wait(&full[stage], phase, abort_flag, p.wait_limit_ns);
              DT_TRACE_ADD(TR_MMA_FULL);
#ifdef DT_GEMM_TRACE
              if (p.trace) atomicAdd(&p.trace[blockIdx.x * TRACE_SLOTS + TR_TMA_LAT],
                                     (unsigned long long)(clock64() - t_issue[stage]));
#endif
            }
            DT_TRACE_COUNT(TR_STAGES);
            if (!_okf) {
              aborted = true;
              *abort_flag = 1;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = a_base + stage * STAGE_BYTES;
            const uint32_t b_addr = a_addr + A_TILE_BYTES;
#pragma unroll
            for (int j = 0; j < BK / 16; ++j) {
              // A: K-major, 128 B rows, 8-row groups 1024 B apart; a K step of 16
              //    elements moves 32 B inside the swizzled row.
              // B: MN-major, 64-column chunks 8 KiB apart (LBO), 8-row K groups
              //    1024 B apart (SBO); a K step of 16 rows moves 2 KiB.
              // K-major B is laid out like A: 128-byte rows of K, a K step of
              // 16 moves 32 B.
              const uint64_t adesc = smem_desc(a_addr + j * 32, 16, 1024);
              const uint64_t bdesc =
                  bk ? smem_desc(b_addr + j * 32, 16, 1024) : smem_desc(b_addr + j * 2048, B_CHUNK_BYTES, 1024);
              mma_bf16(d_tmem, adesc, bdesc, idesc, acc);
              acc = 1;
            }
#ifdef DT_GEMM_TRACE
            t_commit[stage] = clock64();
#endif
            mma_commit(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (aborted) break;
        mma_commit(&tfull[buf]);
        if (++buf == 2) {
          buf = 0;
          tphase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int row_in_tile = quarter * 32 + lane;
    int buf = 0;
    uint32_t tphase = 0;
    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      const TileCoord tc = decode_tile<BM>(p, t);
      const Group& G = p.groups[tc.g];
      int ok = 1;
      if (lane == 0) {
        DT_TRACE_T0();
        ok = mbar_wait(&tfull[buf], tphase, abort_flag, p.wait_limit_ns) ? 1 : 0;
        if (warp == 2) DT_TRACE_ADD(TR_EPI_TFULL);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);  // tcgen05.ld below is warp-collective
      if (!ok) {
        aborted = true;
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int64_t r = tc.m0 + row_in_tile;
      char* row_ptr = nullptr;
      if (r < G.m) {
        int j = 0;
        while (j + 1 < G.nout && G.out_row_begin[j + 1] <= r) ++j;
        const int esize = G.out_dtype == DT_BF16 ? 2 : 4;
        row_ptr = G.out_ptr[j] + (r - G.out_row_begin[j]) * G.out_ld[j] * esize;
      }
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(buf * BN_MAX);
      if (!G.dual) {
        const int nmma = tile_mma_n(G, tc.n0);
        for (int c = 0; c < nmma; c += 32) {
          uint32_t raw[32];
          tmem_ld32(tbase + c, raw);
          tmem_ld_wait();
          if (row_ptr) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(raw[i]);
            if (G.bias_dtype >= 0) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int col = tc.n0 + c + i;
                if (col < G.n) v[i] += bias_at(G, col);
              }
            }
            store_row32(G, row_ptr, tc.n0 + c, v);
          }
        }
      } else {
        for (int c = 0; c < 128; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(tbase + c, g);
          tmem_ld32(tbase + 128 + c, u);
          tmem_ld_wait();
          if (row_ptr) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float gv = __uint_as_float(g[i]);
              const float uv = __uint_as_float(u[i]);
              v[i] = gv / (1.0f + __expf(-gv)) * uv;  // SiLU(g) * u in fp32
            }
            store_row32(G, row_ptr, tc.n0 + c, v);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      if (++buf == 2) {
        buf = 0;
        tphase ^= 1u;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();  // lanes 1..31 of warps 0 and 1 wait here for their lane 0
#ifdef DT_GEMM_TRACE
  if (threadIdx.x == 0 && p.trace) atomicAdd(&p.trace[blockIdx.x * TRACE_SLOTS + TR_TOTAL], (unsigned long long)(clock64() - _trace_start));
#endif
  if (aborted && lane == 0) {
    atomicOr(p.status, DT_DEV_ERR_TIMEOUT);
  }
  if (warp == 0 && lane == 0 && aborted) {
    // let copies already in flight land before the CTA's smem is released
    for (int s = 0; s < STAGES; ++s) {
      if (issued_parity[s] < 0) continue;
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(&full[s], static_cast<uint32_t>(issued_parity[s])) && globaltimer() - t0 < 100000000ull) {
      }
    }
  }
  if (warp == 1 && lane == 0) {
    // every MMA this CTA issued has completed before TMEM is freed
    mma_commit(drain);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < 100000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

cudaError_t launch_tcgen05(const Params& p, int grid, cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tcgen05_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  tcgen05_gemm_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gemm
}  // namespace dt
