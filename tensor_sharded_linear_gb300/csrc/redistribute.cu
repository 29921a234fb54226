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
#include <cstdlib>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "dt_internal.h"
#include "ptx_sm103.cuh"

namespace dt {
namespace {

// Tuning (overridable at build time for sweeps): bytes of a row per work
// item, resident CTAs per SM, 16-byte vectors in flight per lane.
#ifndef RD_COPY_SEG
#define RD_COPY_SEG 4096
#endif
#ifndef RD_COPY_CTAS
#define RD_COPY_CTAS 4
#endif
#ifndef RD_COPY_UNROLL
#define RD_COPY_UNROLL 4
#endif
#ifndef RD_REALIGN_UNROLL
#define RD_REALIGN_UNROLL 4
#endif
#ifndef RD_SUM_CTAS
#define RD_SUM_CTAS 2
#endif
#ifndef RD_BULK_DEFAULT
#define RD_BULK_DEFAULT 1
#endif

constexpr int RD_MAX_TASKS = 192;
constexpr int RD_MAX_REFS = 256;
constexpr int RD_MAX_LAUNCH_SLOTS = 128;  // per side, over every tensor of a batch
constexpr int RD_MAX_SRC = 16;  // sources a lane keeps addresses of; more take sum_many
constexpr int RD_MAX_EXTRA_DST = 15;  // further destinations of one copy task
constexpr int RD_THREADS = 256;
constexpr int RD_WARPS = RD_THREADS / 32;
constexpr int COPY_SEG_BYTES = RD_COPY_SEG;  // one warp moves up to this much of a row per work item
constexpr int SUM_SEG_BYTES = 2048;          // of the destination, for Partial sums

struct RdSlot {
  char* ptr;
  int64_t stride[4];  // elements; dims padded at the front
};

// One box: `ext` elements per (padded) dim, taken from `nsrc` sources (rank
// order) and written to one destination slot; nsrc == 0 writes zeros.  The
// box is cut into work items of (row, segment): rows are the outer three
// padded dims, a segment is `seg_elems` consecutive elements of a row.
struct RdTask {
  int64_t ext[4];
  int64_t dst_off;
  int64_t item_begin;
  int32_t seg_elems;
  int32_t segs_per_row;
  int16_t dst_slot;
  int16_t nsrc;
  int16_t ref_begin;  // sources, then (copies) the extra destinations as byte distances
  int8_t dmap[4];     // slot stride used for each padded position (dims merged on the host)
  int8_t nextra;      // copies: further destination slots receiving the same box
  int8_t extra16;     // 1: every further destination is a multiple of 16 bytes from the first
  int16_t rows_per_item;  // bulk copies: whole rows per work item (1: one segment of a row)
};

struct RdRef {
  int64_t off;
  int32_t slot;
  int32_t pad;
};

// Everything a launch needs travels in its parameter block (limit 32 KB).
// The block's size costs launch time (about 1 us per 10 KB measured on
// GB300), so a launch whose tables fit the compact capacities uses the
// compact block and only large batches take the full one.
template <int NSLOT, int NTASK, int NREF>
struct RdParamsT {
  static constexpr int kSlots = NSLOT, kTasks = NTASK, kRefs = NREF;
  RdSlot dst[NSLOT];
  RdSlot src[NSLOT];
  RdTask task[NTASK];
  RdRef ref[NREF];
  int64_t nitems;
  int32_t ntasks;
  int32_t dtype;  // one dtype, element size and reduce op per launch
  int32_t esize;
  int32_t op;
  int32_t* status;  // DT_DEV_* bits (the bulk copy kernel's bounded waits)
  unsigned long long wait_limit_ns;  // bound of the bulk copy kernel's waits
  int32_t starve;                    // test hook: the bulk kernel issues no loads, so its waits run out
};
using RdParams = RdParamsT<RD_MAX_LAUNCH_SLOTS, RD_MAX_TASKS, RD_MAX_REFS>;
using RdParamsSmall = RdParamsT<32, 48, 64>;
static_assert(sizeof(RdParams) <= 32000, "redistribute parameter block over the launch limit");

// ---------------------------------------------------------------- device

__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) { __stcs(p, v); }

// 16-byte vectors, source and destination equally aligned: every lane keeps
// up to 8 loads in flight before storing.
__device__ __forceinline__ void copy_vec_aligned(uint4* dv, const uint4* sv, int64_t nvec, int lane) {
  constexpr int UN = RD_COPY_UNROLL;
  int64_t i = lane;
  for (; i + (UN - 1) * 32 < nvec; i += UN * 32) {
    uint4 v[UN];
#pragma unroll
    for (int u = 0; u < UN; ++u) v[u] = ld_stream(sv + i + 32 * u);
#pragma unroll
    for (int u = 0; u < UN; ++u) st_stream(dv + i + 32 * u, v[u]);
  }
  for (; i < nvec; i += 32) st_stream(dv + i, ld_stream(sv + i));
}

// Bytes [delta, delta + 16) of the 32-byte pair (a, b).
__device__ __forceinline__ uint4 realign(const uint4& a, const uint4& b, int delta) {
  const uint32_t sh = (delta & 3) * 8;
  const uint32_t c0 = a.x, c1 = a.y, c2 = a.z, c3 = a.w, c4 = b.x, c5 = b.y, c6 = b.z, c7 = b.w;
  switch (delta >> 2) {
    case 0:
      return make_uint4(__funnelshift_r(c0, c1, sh), __funnelshift_r(c1, c2, sh), __funnelshift_r(c2, c3, sh),
                        __funnelshift_r(c3, c4, sh));
    case 1:
      return make_uint4(__funnelshift_r(c1, c2, sh), __funnelshift_r(c2, c3, sh), __funnelshift_r(c3, c4, sh),
                        __funnelshift_r(c4, c5, sh));
    case 2:
      return make_uint4(__funnelshift_r(c2, c3, sh), __funnelshift_r(c3, c4, sh), __funnelshift_r(c4, c5, sh),
                        __funnelshift_r(c5, c6, sh));
    default:
      return make_uint4(__funnelshift_r(c3, c4, sh), __funnelshift_r(c4, c5, sh), __funnelshift_r(c5, c6, sh),
                        __funnelshift_r(c6, c7, sh));
  }
}

__device__ __forceinline__ uint4 shfl_lane0_vec(const uint4& v) {
  return make_uint4(__shfl_sync(0xffffffffu, v.x, 0), __shfl_sync(0xffffffffu, v.y, 0),
                    __shfl_sync(0xffffffffu, v.z, 0), __shfl_sync(0xffffffffu, v.w, 0));
}

__device__ __forceinline__ uint4 shfl_down_vec(const uint4& v) {
  return make_uint4(__shfl_down_sync(0xffffffffu, v.x, 1), __shfl_down_sync(0xffffffffu, v.y, 1),
                    __shfl_down_sync(0xffffffffu, v.z, 1), __shfl_down_sync(0xffffffffu, v.w, 1));
}

// 16-byte destination vectors from a source `delta` (1..15) bytes past a
// 16-byte boundary: each lane loads the aligned source vector under its
// destination vector and takes the next one from its neighbour lane, so
// every source byte is loaded once.  Only aligned vectors that hold at least
// one byte of the source span are read.  Lane 31 takes lane 0's vector of the
// next row by a broadcast shuffle, so a pass keeps one vector per row and
// lane, not two: the kernel stays inside its 64 registers without spilling,
// which took single uneven calls from 0.74-0.77 to 0.77-0.83 of the copy
// peak and the batched sweep from 919 to 911 us.
__device__ __forceinline__ void copy_vec_realign(uint4* dv, const char* s, int64_t nvec, int lane) {
  const int delta = static_cast<int>(reinterpret_cast<uintptr_t>(s) & 15);
  const uint4* sa = reinterpret_cast<const uint4*>(s - delta);
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int64_t base = 0; base < nvec; base += RD_REALIGN_UNROLL * 32) {
    uint4 a[RD_REALIGN_UNROLL];
#pragma unroll
    for (int u = 0; u < RD_REALIGN_UNROLL; ++u) {
      const int64_t j = base + 32 * u + lane;
      a[u] = j <= nvec ? ld_stream(sa + j) : z;
    }
    // the vector after the pass's last one, lane 31's neighbour in the last
    // row, loaded with the others: a pass costs one memory round trip
    const int64_t jl = base + 32 * RD_REALIGN_UNROLL;
    const uint4 extra = (lane == 31 && jl <= nvec) ? ld_stream(sa + jl) : z;
#pragma unroll
    for (int u = 0; u < RD_REALIGN_UNROLL; ++u) {
      // lanes 0..30 take their neighbour's vector; lane 31 takes lane 0's
      // vector of the next row (or the extra one after the last row)
      uint4 next = shfl_down_vec(a[u]);
      // (the index is clamped only to keep it in range where the unrolled
      // branch is not taken)
      const uint4 wrap = u + 1 < RD_REALIGN_UNROLL ? shfl_lane0_vec(a[u + 1 < RD_REALIGN_UNROLL ? u + 1 : u]) : extra;
      if (lane == 31) next = wrap;
      const int64_t j = base + 32 * u + lane;
      if (j < nvec) st_stream(dv + j, realign(a[u], next, delta));
    }
  }
}

// Copy n elements with unit strides.  The elements before the first 16-byte
// aligned destination byte (lanes 0..7) and after the last whole vector
// (lanes 16..23) are loaded in the same pass as the vector body, so a
// segment costs one memory round trip whatever its alignment.
__device__ void copy_span(char* d, const char* s, int64_t n, int esize, int lane) {
  const uintptr_t da = reinterpret_cast<uintptr_t>(d);
  const int64_t nbytes = n * esize;
  int64_t head = static_cast<int64_t>((16 - (da & 15)) & 15);
  if (head > nbytes) head = nbytes;
  const int64_t nvec = (nbytes - head) / 16;
  const int64_t tail = nbytes - head - nvec * 16;
  const int head_n = static_cast<int>(head / esize), tail_n = static_cast<int>(tail / esize);
  int64_t edge = -1;  // element index this lane moves outside the vector body
  if (lane < head_n) edge = lane;
  else if (lane >= 16 && lane - 16 < tail_n) edge = (head + nvec * 16) / esize + (lane - 16);
  uint32_t ev = 0;
  if (edge >= 0) ev = esize == 2 ? reinterpret_cast<const uint16_t*>(s)[edge] : reinterpret_cast<const uint32_t*>(s)[edge];
  char* db = d + head;
  const char* sb = s + head;
  if ((reinterpret_cast<uintptr_t>(sb) & 15) == 0)
    copy_vec_aligned(reinterpret_cast<uint4*>(db), reinterpret_cast<const uint4*>(sb), nvec, lane);
  else
    copy_vec_realign(reinterpret_cast<uint4*>(db), sb, nvec, lane);
  if (edge >= 0) {
    if (esize == 2) reinterpret_cast<uint16_t*>(d)[edge] = static_cast<uint16_t>(ev);
    else reinterpret_cast<uint32_t*>(d)[edge] = ev;
  }
}

// copy_span into the first destination d and nx replicas d + x[j].off,
// each a multiple of 16 bytes from d, with d and s equally aligned: every
// source vector is loaded once and stored to every replica.
__device__ __forceinline__ void copy_span_replicas(char* d, const char* s, int64_t n, int esize, int lane,
                                                   const RdRef* x, int nx) {
  const uintptr_t da = reinterpret_cast<uintptr_t>(d);
  const int64_t nbytes = n * esize;
  int64_t head = static_cast<int64_t>((16 - (da & 15)) & 15);
  if (head > nbytes) head = nbytes;
  const int64_t nvec = (nbytes - head) / 16;
  const int64_t tail = nbytes - head - nvec * 16;
  const int head_n = static_cast<int>(head / esize), tail_n = static_cast<int>(tail / esize);
  int64_t edge = -1;
  if (lane < head_n) edge = lane;
  else if (lane >= 16 && lane - 16 < tail_n) edge = (head + nvec * 16) / esize + (lane - 16);
  uint32_t ev = 0;
  if (edge >= 0) ev = esize == 2 ? reinterpret_cast<const uint16_t*>(s)[edge] : reinterpret_cast<const uint32_t*>(s)[edge];
  const uint4* sv = reinterpret_cast<const uint4*>(s + head);
  uint4* dv = reinterpret_cast<uint4*>(d + head);
  constexpr int UN = RD_COPY_UNROLL;
  int64_t i = lane;
  for (; i + (UN - 1) * 32 < nvec; i += UN * 32) {
    uint4 v[UN];
#pragma unroll
    for (int u = 0; u < UN; ++u) v[u] = ld_stream(sv + i + 32 * u);
    for (int j = 0; j <= nx; ++j) {
      uint4* dj = j == 0 ? dv : reinterpret_cast<uint4*>(reinterpret_cast<char*>(dv) + x[j - 1].off);
#pragma unroll
      for (int u = 0; u < UN; ++u) st_stream(dj + i + 32 * u, v[u]);
    }
  }
  for (; i < nvec; i += 32) {
    const uint4 v = ld_stream(sv + i);
    for (int j = 0; j <= nx; ++j) {
      uint4* dj = j == 0 ? dv : reinterpret_cast<uint4*>(reinterpret_cast<char*>(dv) + x[j - 1].off);
      st_stream(dj + i, v);
    }
  }
  if (edge >= 0) {
    for (int j = 0; j <= nx; ++j) {
      char* dj = j == 0 ? d : d + x[j - 1].off;
      if (esize == 2) reinterpret_cast<uint16_t*>(dj)[edge] = static_cast<uint16_t>(ev);
      else reinterpret_cast<uint32_t*>(dj)[edge] = ev;
    }
  }
}

__device__ void copy_span_strided(char* d, const char* s, int64_t n, int64_t dstr, int64_t sstr, int esize, int lane) {
  if (esize == 2) {
    for (int64_t i = lane; i < n; i += 32)
      reinterpret_cast<uint16_t*>(d)[i * dstr] = reinterpret_cast<const uint16_t*>(s)[i * sstr];
  } else {
    for (int64_t i = lane; i < n; i += 32)
      reinterpret_cast<uint32_t*>(d)[i * dstr] = reinterpret_cast<const uint32_t*>(s)[i * sstr];
  }
}

__device__ void zero_span(char* d, int64_t n, int64_t dstr, int esize, int lane) {
  const uintptr_t da = reinterpret_cast<uintptr_t>(d);
  if (dstr == 1) {
    const int64_t nbytes = n * esize;
    int64_t head = static_cast<int64_t>((16 - (da & 15)) & 15);
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

// Reduction step and final step of the Partial ops, in fp32: SUM and AVG
// add with round-to-nearest adds (AVG then divides once by the count), MAX
// keeps the larger value (rank order decides between equal ones).
__device__ __forceinline__ float red_step(float acc, float v, int op) {
  return op == DT_MAX ? (v > acc ? v : acc) : __fadd_rn(acc, v);
}
__device__ __forceinline__ float red_final(float acc, int nsrc, int op) {
  return op == DT_AVG ? __fdiv_rn(acc, static_cast<float>(nsrc)) : acc;
}

// Element-wise Partial reduction, rank order, fp32: the first value as is,
// the others combined by red_step; bf16 rounded once at the end.
__device__ __forceinline__ void sum_elems(char* d, const char* const* s, int nsrc, int64_t lo, int64_t hi, int64_t dstr,
                                          const int64_t* sstr, int dtype, int op, int lane) {
  for (int64_t i = lo + lane; i < hi; i += 32) {
    if (dtype == DT_BF16) {
      float acc = to_f(reinterpret_cast<const uint16_t*>(s[0])[i * sstr[0]]);
      for (int k = 1; k < nsrc; ++k) acc = red_step(acc, to_f(reinterpret_cast<const uint16_t*>(s[k])[i * sstr[k]]), op);
      reinterpret_cast<uint16_t*>(d)[i * dstr] = from_f(red_final(acc, nsrc, op));
    } else {
      float acc = reinterpret_cast<const float*>(s[0])[i * sstr[0]];
      for (int k = 1; k < nsrc; ++k) acc = red_step(acc, reinterpret_cast<const float*>(s[k])[i * sstr[k]], op);
      reinterpret_cast<float*>(d)[i * dstr] = red_final(acc, nsrc, op);
    }
  }
}

// Vector body of the Partial sum with the source count fixed at compile time:
// every lane issues NSRC x VPL 16-byte loads (at most 16) before the first add.
template <int NSRC, int DTYPE>
__device__ __forceinline__ void sum_vec(uint4* dv, const char* const* s, int64_t byte_off, int64_t nvec, int op,
                                        int lane) {
  constexpr int EPV = DTYPE == DT_BF16 ? 8 : 4;                        // elements per vector
  constexpr int VPL = NSRC >= 8 ? 2 : 4;                               // vectors per lane per pass
  const uint4* sv[NSRC];
#pragma unroll
  for (int k = 0; k < NSRC; ++k) sv[k] = reinterpret_cast<const uint4*>(s[k] + byte_off);
  for (int64_t base = 0; base < nvec; base += VPL * 32) {
    uint4 v[NSRC][VPL];
#pragma unroll
    for (int k = 0; k < NSRC; ++k)
#pragma unroll
      for (int u = 0; u < VPL; ++u) {
        const int64_t j = base + 32 * u + lane;
        v[k][u] = j < nvec ? ld_stream(sv[k] + j) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
      const int64_t j = base + 32 * u + lane;
      if (j >= nvec) continue;
      float acc[EPV];
#pragma unroll
      for (int k = 0; k < NSRC; ++k) {
        const uint32_t w[4] = {v[k][u].x, v[k][u].y, v[k][u].z, v[k][u].w};
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const float f = DTYPE == DT_BF16 ? ((e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1])) : __uint_as_float(w[e]);
          acc[e] = k == 0 ? f : red_step(acc[e], f, op);
        }
      }
#pragma unroll
      for (int e = 0; e < EPV; ++e) acc[e] = red_final(acc[e], NSRC, op);
      uint4 o;
      if (DTYPE == DT_BF16)
        o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                       pack_bf16x2(acc[6], acc[7]));
      else
        o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                       __float_as_uint(acc[3]));
      st_stream(dv + j, o);
    }
  }
}

template <int DTYPE>
__device__ __forceinline__ bool sum_vec_dispatch(uint4* dv, const char* const* s, int nsrc, int64_t off, int64_t nvec,
                                                 int op, int lane) {
  switch (nsrc) {
    case 2: sum_vec<2, DTYPE>(dv, s, off, nvec, op, lane); return true;
    case 3: sum_vec<3, DTYPE>(dv, s, off, nvec, op, lane); return true;
    case 4: sum_vec<4, DTYPE>(dv, s, off, nvec, op, lane); return true;
    case 8: sum_vec<8, DTYPE>(dv, s, off, nvec, op, lane); return true;
    default: return false;
  }
}

__device__ void sum_span(char* d, const char* const* s, int nsrc, int64_t n, int64_t dstr, const int64_t* sstr,
                         int dtype, int op, int lane) {
  const uintptr_t da = reinterpret_cast<uintptr_t>(d);
  bool vec = dstr == 1;
  for (int k = 0; k < nsrc; ++k)
    vec = vec && sstr[k] == 1 && ((reinterpret_cast<uintptr_t>(s[k]) ^ da) & 15) == 0;
  if (!vec) {
    sum_elems(d, s, nsrc, 0, n, dstr, sstr, dtype, op, lane);
    return;
  }
  const int esize = dtype == DT_BF16 ? 2 : 4;
  int64_t head = static_cast<int64_t>(((16 - (da & 15)) & 15) / esize);
  if (head > n) head = n;
  const int64_t nvec = (n - head) * esize / 16;
  const int64_t vec_end = head + nvec * (16 / esize);
  // edge elements (lanes 0..7: head, lanes 16..23: tail): loads issued
  // before the vector body's, summed and stored after it
  int64_t edge = -1;
  if (lane < head) edge = lane;
  else if (lane >= 16 && vec_end + (lane - 16) < n) edge = vec_end + (lane - 16);
  float ev[RD_MAX_SRC];
  if (edge >= 0) {
    for (int k = 0; k < nsrc; ++k)
      ev[k] = dtype == DT_BF16 ? to_f(reinterpret_cast<const uint16_t*>(s[k])[edge])
                               : reinterpret_cast<const float*>(s[k])[edge];
  }
  uint4* dv = reinterpret_cast<uint4*>(d + head * esize);
  const bool done = dtype == DT_BF16 ? sum_vec_dispatch<DT_BF16>(dv, s, nsrc, head * esize, nvec, op, lane)
                                     : sum_vec_dispatch<DT_FP32>(dv, s, nsrc, head * esize, nvec, op, lane);
  if (!done) sum_elems(d, s, nsrc, head, vec_end, 1, sstr, dtype, op, lane);
  if (edge >= 0) {
    float acc = ev[0];
    for (int k = 1; k < nsrc; ++k) acc = red_step(acc, ev[k], op);
    acc = red_final(acc, nsrc, op);
    if (dtype == DT_BF16) reinterpret_cast<uint16_t*>(d)[edge] = from_f(acc);
    else reinterpret_cast<float*>(d)[edge] = acc;
  }
}

// More than RD_MAX_SRC partial sources (several Partial mesh dims): one
// element per lane per pass, each source's address formed from the parameter
// block as it is read, in rank order like sum_elems.
template <class P>
__device__ void sum_many(char* d, int64_t dstr, const P& p, const RdTask& T, int64_t i0, int64_t i1, int64_t i2,
                         int64_t e0, int64_t n, int lane) {
  const int m0 = T.dmap[0], m1 = T.dmap[1], m2 = T.dmap[2], m3 = T.dmap[3];
  const int esize = p.esize;
  for (int64_t i = lane; i < n; i += 32) {
    float acc = 0.f;
    for (int k = 0; k < T.nsrc; ++k) {
      const RdRef& R = p.ref[T.ref_begin + k];
      const RdSlot& S = p.src[R.slot];
      const char* sp =
          S.ptr + (R.off + i0 * S.stride[m0] + i1 * S.stride[m1] + i2 * S.stride[m2] + (e0 + i) * S.stride[m3]) * esize;
      const float v = p.dtype == DT_BF16 ? to_f(*reinterpret_cast<const uint16_t*>(sp))
                                         : *reinterpret_cast<const float*>(sp);
      acc = k == 0 ? v : red_step(acc, v, p.op);
    }
    acc = red_final(acc, T.nsrc, p.op);
    if (p.dtype == DT_BF16) reinterpret_cast<uint16_t*>(d)[i * dstr] = from_f(acc);
    else reinterpret_cast<float*>(d)[i * dstr] = acc;
  }
}

// SUM = false: every task copies (nsrc == 1) or zero-fills (nsrc == 0),
// REPL = true: to its destination and its replicas (nextra of them);
// SUM = true: every task adds nsrc >= 2 partial sources.  One instantiation
// per kind keeps the plain copy path's register use low.  Warps take work
// items (row, segment) in a grid-stride loop.
template <bool SUM, bool REPL, class P>
__global__ void __launch_bounds__(RD_THREADS, SUM ? RD_SUM_CTAS : RD_COPY_CTAS) rd_kernel(const __grid_constant__ P p) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * RD_WARPS;
  int t = 0;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * RD_WARPS + (threadIdx.x >> 5); it < p.nitems; it += nw) {
    while (t + 1 < p.ntasks && p.task[t + 1].item_begin <= it) ++t;
    const RdTask& T = p.task[t];
    const int esize = p.esize;
    const int64_t local = it - T.item_begin;
    const int64_t r = local / T.segs_per_row;
    const int64_t e0 = (local - r * T.segs_per_row) * T.seg_elems;
    const int64_t n = min(T.ext[3] - e0, static_cast<int64_t>(T.seg_elems));
    const int64_t i2 = r % T.ext[2];
    const int64_t q = r / T.ext[2];
    const int64_t i1 = q % T.ext[1];
    const int64_t i0 = q / T.ext[1];
    const RdSlot& D = p.dst[T.dst_slot];
    const int m0 = T.dmap[0], m1 = T.dmap[1], m2 = T.dmap[2], m3 = T.dmap[3];
    char* d =
        D.ptr + (T.dst_off + i0 * D.stride[m0] + i1 * D.stride[m1] + i2 * D.stride[m2] + e0 * D.stride[m3]) * esize;
    if (!SUM && T.nsrc == 0) {
      zero_span(d, n, D.stride[m3], esize, lane);
    } else if (!SUM) {
      const RdRef& R = p.ref[T.ref_begin];
      const RdSlot& S = p.src[R.slot];
      const char* s =
          S.ptr + (R.off + i0 * S.stride[m0] + i1 * S.stride[m1] + i2 * S.stride[m2] + e0 * S.stride[m3]) * esize;
      const bool unit = D.stride[m3] == 1 && S.stride[m3] == 1;
      if (!REPL) {
        if (unit) copy_span(d, s, n, esize, lane);
        else copy_span_strided(d, s, n, D.stride[m3], S.stride[m3], esize, lane);
      } else {
        // the replicas of a materialised Replicate layout: each has the first
        // destination's strides and sits a fixed number of bytes from it (the
        // host stores that distance).  Equally aligned replicas take each
        // loaded vector; otherwise the source span is re-read from L1/L2.
        if (unit && T.extra16 && ((reinterpret_cast<uintptr_t>(d) ^ reinterpret_cast<uintptr_t>(s)) & 15) == 0) {
          copy_span_replicas(d, s, n, esize, lane, &p.ref[T.ref_begin + 1], T.nextra);
          continue;
        }
        for (int j = 0; j <= T.nextra; ++j) {
          char* dj = j == 0 ? d
                            : reinterpret_cast<char*>(reinterpret_cast<uintptr_t>(d) +
                                                      static_cast<uintptr_t>(p.ref[T.ref_begin + j].off));
          if (unit) copy_span(dj, s, n, esize, lane);
          else copy_span_strided(dj, s, n, D.stride[m3], S.stride[m3], esize, lane);
        }
      }
    } else if (T.nsrc > RD_MAX_SRC) {
      sum_many(d, D.stride[m3], p, T, i0, i1, i2, e0, n, lane);
    } else {
      const char* sp[RD_MAX_SRC];
      int64_t ss[RD_MAX_SRC];
      for (int k = 0; k < T.nsrc; ++k) {
        const RdRef& R = p.ref[T.ref_begin + k];
        const RdSlot& S = p.src[R.slot];
        sp[k] = S.ptr + (R.off + i0 * S.stride[m0] + i1 * S.stride[m1] + i2 * S.stride[m2] + e0 * S.stride[m3]) * esize;
        ss[k] = S.stride[m3];
      }
      sum_span(d, sp, T.nsrc, n, D.stride[m3], ss, p.dtype, p.op, lane);
    }
  }
}

// ---------------------------------------------------------------- bulk (TMA) copies
//
// Copies whose every row starts on a 16-byte boundary in source and
// destination and is a multiple of 16 bytes long (the aligned shapes:
// Shard <-> Shard / Replicate of [8192, 8192] bf16 and the like) can run
// entirely on the bulk-copy (TMA) engine: global -> shared memory with
// cp.async.bulk, completion counted on an mbarrier, then shared -> global
// with the bulk store, its reads of shared memory tracked by bulk groups.
// No thread touches the data.  Four pipelines per CTA (lane 0 of warps
// 0..3), each with RDT_STAGES stages of RDT_STAGE_BYTES, walk disjoint work
// items: item i of pipeline q of CTA b is q + 4 b + i * 4 G.  A work item is
// a run of whole rows, or one segment of a longer row, of at most one stage.
// Six 8 KiB stages per pipeline, measured against three of 16 KiB in the
// same shared memory: one call per [8192, 8192] transition went from
// 0.80-0.83 to 0.836-0.838 of the copy peak on every aligned transition
// (more stores in flight per pipeline); 4 KiB stages fell to 0.55-0.59
// (one thread per pipeline issues twice the copies per byte).
constexpr int RDT_PIPES = 4;
constexpr int RDT_STAGES = 6;
constexpr int RDT_STAGE_BYTES = 8192;
constexpr int RDT_THREADS = 32 * RDT_PIPES;
constexpr int RDT_SMEM_BYTES = RDT_PIPES * RDT_STAGES * RDT_STAGE_BYTES + RDT_PIPES * RDT_STAGES * 8 + 16;
constexpr int RDT_LAG = 1;  // a stage is stored this many items after it was loaded

// The rows of work item `it`: task t (advanced from the caller's hint), first
// row r0, nrows rows, elements [e0, e0 + n) of each.  Bulk launches keep row
// and item counts below 2^31 (rows of at least 16 bytes in a tensor below
// 32 GB), so the index arithmetic is 32-bit.
template <class P>
__device__ __forceinline__ void rdt_item(const P& p, int64_t it, int* t, uint32_t* r0, int* nrows, int64_t* e0,
                                         int64_t* n) {
  while (*t + 1 < p.ntasks && p.task[*t + 1].item_begin <= it) ++*t;
  const RdTask& T = p.task[*t];
  const uint32_t local = static_cast<uint32_t>(it - T.item_begin);
  if (T.rows_per_item > 1) {
    const uint32_t rows = static_cast<uint32_t>(T.ext[0] * T.ext[1] * T.ext[2]);
    *r0 = local * static_cast<uint32_t>(T.rows_per_item);
    *nrows = static_cast<int>(min(static_cast<uint32_t>(T.rows_per_item), rows - *r0));
    *e0 = 0;
    *n = T.ext[3];
  } else {
    const uint32_t spr = static_cast<uint32_t>(T.segs_per_row);
    *r0 = local / spr;
    *nrows = 1;
    *e0 = static_cast<int64_t>(local - *r0 * spr) * T.seg_elems;
    *n = min(T.ext[3] - *e0, static_cast<int64_t>(T.seg_elems));
  }
}

// Consecutive rows of a task: the (i0, i1, i2) index of the three outer
// (padded) dims, advanced like an odometer, and the row's two addresses.
struct RdtRows {
  uint32_t i0, i1, i2, e1, e2;
  __device__ __forceinline__ RdtRows(const RdTask& T, uint32_t r) {
    e1 = static_cast<uint32_t>(T.ext[1]);
    e2 = static_cast<uint32_t>(T.ext[2]);
    i2 = r % e2;
    const uint32_t q = r / e2;
    i1 = q % e1;
    i0 = q / e1;
  }
  __device__ __forceinline__ void next() {
    if (++i2 == e2) {
      i2 = 0;
      if (++i1 == e1) {
        i1 = 0;
        ++i0;
      }
    }
  }
  template <class P>
  __device__ __forceinline__ void at(const P& p, const RdTask& T, int64_t e0, char** d, const char** s) const {
    const RdSlot& D = p.dst[T.dst_slot];
    const RdRef& R = p.ref[T.ref_begin];
    const RdSlot& S = p.src[R.slot];
    const int m0 = T.dmap[0], m1 = T.dmap[1], m2 = T.dmap[2];
    *d = D.ptr + (T.dst_off + i0 * D.stride[m0] + i1 * D.stride[m1] + i2 * D.stride[m2] + e0) * p.esize;
    *s = S.ptr + (R.off + i0 * S.stride[m0] + i1 * S.stride[m1] + i2 * S.stride[m2] + e0) * p.esize;
  }
};

__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  uint64_t g;
  asm volatile("cvta.to.global.u64 %0, %1;" : "=l"(g) : "l"(gdst));
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(g), "r"(smem_u32(smem_src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <class P>
__global__ void __launch_bounds__(RDT_THREADS, 1) rd_tma_kernel(const __grid_constant__ P p) {
  extern __shared__ __align__(128) uint8_t rdt_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(rdt_smem + RDT_PIPES * RDT_STAGES * RDT_STAGE_BYTES) + warp * RDT_STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(reinterpret_cast<uint64_t*>(
                                 rdt_smem + RDT_PIPES * RDT_STAGES * RDT_STAGE_BYTES) + RDT_PIPES * RDT_STAGES);
  if (lane == 0)
    for (int s = 0; s < RDT_STAGES; ++s) mbar_init(&full[s], 1);
  if (threadIdx.x == 0) *abort_flag = 0;
  fence_mbar_init();
  __syncthreads();
  if (lane != 0) return;
  uint8_t* ring = rdt_smem + warp * RDT_STAGES * RDT_STAGE_BYTES;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * RDT_PIPES + warp;
  const int64_t step = static_cast<int64_t>(gridDim.x) * RDT_PIPES;
  const int64_t count = first < p.nitems ? (p.nitems - 1 - first) / step + 1 : 0;
  int t_load = 0, t_store = 0;
  bool aborted = false;
  // iteration k loads item k (if any) and stores item k - RDT_LAG (if any)
  for (int64_t k = 0; k < count + RDT_LAG && !aborted; ++k) {
    if (k < count) {
      const int stage = static_cast<int>(k % RDT_STAGES);
      // the store that last read this stage (item k - RDT_STAGES) is done reading
      if (k >= RDT_STAGES) bulk_wait_read<RDT_STAGES - 1 - RDT_LAG>();
      uint32_t r0;
      int64_t e0, n;
      int nrows;
      rdt_item(p, first + k * step, &t_load, &r0, &nrows, &e0, &n);
      const RdTask& T = p.task[t_load];
      const uint32_t nbytes = static_cast<uint32_t>(n * p.esize);
      mbar_expect_tx(&full[stage], nbytes * static_cast<uint32_t>(nrows));
      uint8_t* dst = ring + stage * RDT_STAGE_BYTES;
      RdtRows rows(T, r0);
      for (int j = 0; j < nrows; ++j, rows.next(), dst += nbytes) {
        char* d;
        const char* src;
        rows.at(p, T, e0, &d, &src);
        if (!p.starve) bulk_load(dst, src, nbytes, &full[stage]);
      }
    }
    if (k >= RDT_LAG) {
      const int64_t ks = k - RDT_LAG;
      const int stage = static_cast<int>(ks % RDT_STAGES);
      if (!mbar_wait(&full[stage], static_cast<uint32_t>((ks / RDT_STAGES) & 1), abort_flag, p.wait_limit_ns)) {
        aborted = true;
        break;
      }
      uint32_t r0;
      int64_t e0, n;
      int nrows;
      rdt_item(p, first + ks * step, &t_store, &r0, &nrows, &e0, &n);
      const RdTask& T = p.task[t_store];
      const uint32_t nbytes = static_cast<uint32_t>(n * p.esize);
      const uint8_t* src = ring + stage * RDT_STAGE_BYTES;
      RdtRows rows(T, r0);
      for (int j = 0; j < nrows; ++j, rows.next(), src += nbytes) {
        char* d;
        const char* s;
        rows.at(p, T, e0, &d, &s);
        bulk_store(d, src, nbytes);
        // the replicas of a materialised Replicate layout: the same row,
        // stored again from the same stage a fixed byte distance away
        for (int x = 1; x <= T.nextra; ++x) bulk_store(d + p.ref[T.ref_begin + x].off, src, nbytes);
      }
      bulk_commit();
    }
  }
  if (aborted) {
    *abort_flag = 1;
    atomicOr(p.status, DT_DEV_ERR_TIMEOUT);
    // loads issued before the wait gave up: a bounded time to land
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 20000000ull) {
    }
  }
  bulk_wait_all();  // every store has read its stage and written global memory
}

// ---------------------------------------------------------------- host

struct HostTask {
  Box box;  // global box moved
  int dst_slot;
  std::vector<int> src_slots;  // rank order; empty = zero fill
  std::vector<int> extra_dst;  // copies: further destination slots, same box and strides
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
      if (ls.is_partial(m)) {
        if (ls.op[m] != ld.op[m]) return fail(DT_ERR_UNSUPPORTED, "a kept Partial dim cannot change its reduce op");
        kept[m] = true;
      } else if (ls.is_replicate(m)) {
        // SUM: coordinate 0 keeps the value, the others are zero; AVG / MAX:
        // every coordinate keeps it (a plain copy from the replica)
        zeroed[m] = ld.op[m] == DT_SUM;
      } else {
        return fail(DT_ERR_UNSUPPORTED, "Shard -> Partial on mesh dim %d is not defined", m);
      }
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
  if (nsum > RD_MAX_REFS) return fail(DT_ERR_CAPACITY, "%d partial sources per element (max %d)", nsum, RD_MAX_REFS);

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
      tasks->push_back(HostTask{bd, ds, {}, {}});
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

// Collapse the task's box dims that are contiguous in the destination and in
// every source (padded position p-1 folds into p when its stride equals
// ext[p] * stride[p] everywhere), so short rows become long runs; extent-1
// dims fold away.  Fills t->ext (front-padded) and t->dmap.
void merge_dims(const HostTask& ht, const DTensor& D, const DTensor& S, int pad, RdTask* t) {
  int64_t ext[4];
  for (int d = 0; d < 4; ++d) ext[d] = d < pad ? 1 : ht.box.size[d - pad];
  auto stride = [&](const SlotView& v, int p) -> int64_t { return p < pad ? 0 : v.stride[p - pad]; };
  // merged dims from the innermost outwards: (extent, padded position whose stride is used)
  int64_t me[4];
  int mp[4];
  int n = 0;
  me[0] = ext[3];
  mp[0] = 3;
  n = 1;
  for (int p = 2; p >= 0; --p) {
    if (ext[p] == 1) continue;
    const int in = mp[n - 1];
    const int64_t run = me[n - 1];
    bool ok = stride(D.slots[ht.dst_slot], p) == run * stride(D.slots[ht.dst_slot], in);
    for (int k = 0; ok && k < (int)ht.src_slots.size(); ++k)
      ok = stride(S.slots[ht.src_slots[k]], p) == run * stride(S.slots[ht.src_slots[k]], in);
    if (ok && me[n - 1] > 0) {
      me[n - 1] *= ext[p];
    } else {
      me[n] = ext[p];
      mp[n] = p;
      ++n;
    }
  }
  // back to front-padded order, innermost at position 3; dmap holds padded
  // positions, which is how RdSlot::stride is indexed
  for (int q = 0; q < 4; ++q) {
    const int k = 3 - q;  // merged dim for padded position q
    t->ext[q] = k < n ? me[k] : 1;
    t->dmap[q] = (int8_t)(k < n ? mp[k] : 0);
  }
}

void fill_slot(RdSlot* out, const SlotView& v, int ndim) {
  out->ptr = v.ptr;
  // pad dims at the front so the innermost tensor dim is padded dim 3
  const int pad = 4 - ndim;
  for (int d = 0; d < 4; ++d) out->stride[d] = d < pad ? 0 : v.stride[d - pad];
}

// Copies of one source box into several destination slots with the same
// strides (the replicas of a materialised Replicate layout) become one task
// with up to RD_MAX_EXTRA_DST further destinations: the kernel reads the
// source once from DRAM and writes every replica.
void group_replica_copies(const DTensor& D, std::vector<HostTask>* tasks) {
  const int nd = D.layout.ndim;
  auto same_strides = [&](int a, int b) {
    for (int d = 0; d < nd; ++d)
      if (D.slots[a].stride[d] != D.slots[b].stride[d]) return false;
    return true;
  };
  auto same_box = [&](const Box& a, const Box& b) {
    for (int d = 0; d < nd; ++d)
      if (a.off[d] != b.off[d] || a.size[d] != b.size[d]) return false;
    return true;
  };
  // open groups by (source slot, box): indices into `out`
  std::map<std::vector<int64_t>, std::vector<int>> groups;
  std::vector<HostTask> out;
  out.reserve(tasks->size());
  for (HostTask& t : *tasks) {
    if (t.src_slots.size() == 1) {
      std::vector<int64_t> key{t.src_slots[0]};
      for (int d = 0; d < nd; ++d) {
        key.push_back(t.box.off[d]);
        key.push_back(t.box.size[d]);
      }
      std::vector<int>& open = groups[key];
      bool merged = false;
      for (int li : open) {
        HostTask& g = out[li];
        if ((int)g.extra_dst.size() < RD_MAX_EXTRA_DST && same_box(g.box, t.box) &&
            same_strides(g.dst_slot, t.dst_slot)) {
          g.extra_dst.push_back(t.dst_slot);
          merged = true;
          break;
        }
      }
      if (merged) continue;
      open.push_back((int)out.size());
    }
    out.push_back(std::move(t));
  }
  tasks->swap(out);
}

struct PairPlan {
  DTensor S, D;
  std::vector<HostTask> copies, sums, repl;  // repl: copies with replica destinations
};

dt_status plan_pair(const dt_dtensor* src, const dt_dtensor* dst, PairPlan* pp) {
  dt_status st = parse_dtensor(src, &pp->S, "src");
  if (st != DT_OK) return st;
  st = parse_dtensor(dst, &pp->D, "dst");
  if (st != DT_OK) return st;
  const Layout& ls = pp->S.layout;
  const Layout& ld = pp->D.layout;
  if (ls.mesh_ndim != ld.mesh_ndim) return fail(DT_ERR_SHAPE, "src and dst meshes differ");
  for (int m = 0; m < ls.mesh_ndim; ++m)
    if (ls.mesh[m] != ld.mesh[m]) return fail(DT_ERR_SHAPE, "src and dst meshes differ");
  if (ls.ndim != ld.ndim) return fail(DT_ERR_SHAPE, "src and dst ranks differ");
  for (int d = 0; d < ls.ndim; ++d)
    if (ls.gshape[d] != ld.gshape[d]) return fail(DT_ERR_SHAPE, "global shapes differ on dim %d", d);
  if (ls.dtype != ld.dtype) return fail(DT_ERR_INVALID_ARG, "src and dst dtypes differ");
  std::vector<HostTask> tasks;
  if ((st = plan(pp->S, pp->D, &tasks)) != DT_OK) return st;
  group_replica_copies(pp->D, &tasks);
  // reductions (>= 2 sources), copies / zero fills and copies to replicas
  // run in separate kernels
  for (auto& t : tasks)
    (t.src_slots.size() >= 2 ? pp->sums : !t.extra_dst.empty() ? pp->repl : pp->copies).push_back(std::move(t));
  return DT_OK;
}

// Launch every task of `plans` of one kind, packing tasks of all pairs into as
// few launches as the parameter block holds.
enum RdKind { RD_COPY = 0, RD_SUM = 1, RD_COPY_REPL = 2 };

// The bulk copy kernel's shared memory, opted in once per parameter-block size.
template <class P>
bool rdt_ready() {
  static int ok = -1;
  if (ok < 0) {
    ok = cudaFuncSetAttribute(rd_tma_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, RDT_SMEM_BYTES) ==
                 cudaSuccess
             ? 1
             : 0;
    if (!ok) cudaGetLastError();
  }
  return ok == 1;
}

template <class P>
void launch_rd(const P& p, int kind, bool bulk, int grid, cudaStream_t stream) {
  if (kind == RD_SUM)
    rd_kernel<true, false, P><<<grid, RD_THREADS, 0, stream>>>(p);
  else if (bulk)  // copies, to replicas too
    rd_tma_kernel<P><<<grid, RDT_THREADS, RDT_SMEM_BYTES, stream>>>(p);
  else if (kind == RD_COPY_REPL)
    rd_kernel<false, true, P><<<grid, RD_THREADS, 0, stream>>>(p);
  else
    rd_kernel<false, false, P><<<grid, RD_THREADS, 0, stream>>>(p);
}

// DT_RD_BULK=0 / 1 in the environment turns the bulk (TMA) copy kernel off
// or on for the copy launches it can run (every row 16-byte aligned on both
// sides), e.g. to compare the two copy kernels; unset, the default applies.
int bulk_copies() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("DT_RD_BULK");
    v = (e && e[0] == '0') ? 0 : (e && e[0] == '1') ? 1 : RD_BULK_DEFAULT;
  }
  return v;
}

// Test hooks, read once from the environment: DT_RD_WAIT_LIMIT_MS bounds
// the bulk copy kernel's waits (default 2000 ms); DT_RD_STARVE=1 makes it
// issue no loads, so its waits run out and the call reports
// DT_DEV_ERR_TIMEOUT -- the bounded-wait exit, exercised without a fault.
unsigned long long rd_wait_limit_ns() {
  static unsigned long long v = 0;
  if (!v) {
    const char* e = getenv("DT_RD_WAIT_LIMIT_MS");
    const long ms = e ? atol(e) : 0;
    v = (ms > 0 && ms <= 10000) ? (unsigned long long)ms * 1000000ull : WAIT_LIMIT_NS;
  }
  return v;
}

int rd_starve() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("DT_RD_STARVE");
    v = (e && e[0] == '1') ? 1 : 0;
  }
  return v;
}

// Whole rows per bulk work item (1: a long row is cut into segments of one
// stage).
void bulk_partition(RdTask* t, int esize) {
  const int64_t row_bytes = t->ext[3] * esize;
  const int64_t rows = t->ext[0] * t->ext[1] * t->ext[2];
  if (row_bytes <= RDT_STAGE_BYTES / 2) {
    t->rows_per_item = (int16_t)std::min<int64_t>(RDT_STAGE_BYTES / row_bytes, rows);
    t->seg_elems = (int32_t)t->ext[3];
    t->segs_per_row = 1;
  } else {
    t->rows_per_item = 1;
    t->seg_elems = (int32_t)(RDT_STAGE_BYTES / esize);
    t->segs_per_row = (int32_t)((t->ext[3] + t->seg_elems - 1) / t->seg_elems);
  }
}

int64_t bulk_items(const RdTask& t) {
  const int64_t rows = t.ext[0] * t.ext[1] * t.ext[2];
  return t.rows_per_item > 1 ? (rows + t.rows_per_item - 1) / t.rows_per_item : rows * t.segs_per_row;
}

// Every row of the task starts on a 16-byte boundary in both slots and is
// a multiple of 16 bytes long; replicas (if any) sit a multiple of 16 bytes
// from the first destination.
bool bulk_task_ok(const RdTask& t, const RdSlot& D, const RdSlot& S, int64_t src_off, int esize) {
  if (t.nsrc != 1 || (t.nextra != 0 && !t.extra16)) return false;
  if (D.stride[t.dmap[3]] != 1 || S.stride[t.dmap[3]] != 1) return false;
  if ((t.ext[3] * esize) % 16) return false;
  if ((reinterpret_cast<uintptr_t>(D.ptr) + (uintptr_t)(t.dst_off * esize)) % 16) return false;
  if ((reinterpret_cast<uintptr_t>(S.ptr) + (uintptr_t)(src_off * esize)) % 16) return false;
  for (int q = 0; q < 3; ++q)
    if (t.ext[q] > 1 && ((D.stride[t.dmap[q]] * esize) % 16 || (S.stride[t.dmap[q]] * esize) % 16)) return false;
  return t.ext[0] * t.ext[1] * t.ext[2] < (1ll << 31);
}

// A call's launches, recorded as issued (kind, kernel, grid and the exact
// parameter block) so a later call with the same operands can replay them
// without planning again.
struct RecordedLaunch {
  int kind = 0;
  bool small = false;
  bool bulk = false;
  int grid = 0;
  std::vector<uint8_t> params;
};
struct RecordedPlan {
  bool forked = false;
  std::vector<RecordedLaunch> launches;
};
thread_local RecordedPlan* g_recording = nullptr;

dt_status launch_kind(std::vector<PairPlan>& plans, int kind, int32_t* status, cudaStream_t stream) {
  const bool sum = kind == RD_SUM;
  static thread_local RdParams p;  // ~28 KB: off the stack
  static thread_local RdParamsSmall ps;
  const int sms = device_sm_count();
  int nd_slots = 0, ns_slots = 0, nt = 0, nref = 0;
  int64_t items = 0;
  // every copy task so far can run on the bulk copy kernel (rows aligned on
  // both sides, replicas a multiple of 16 bytes apart)
  bool aligned = (kind == RD_COPY || kind == RD_COPY_REPL) && bulk_copies() == 1;
  auto flush = [&]() -> dt_status {
    if (nt == 0) return DT_OK;
    const bool small = nd_slots <= ps.kSlots && ns_slots <= ps.kSlots && nt <= ps.kTasks && nref <= ps.kRefs;
    const bool bulk = aligned && (small ? rdt_ready<RdParamsSmall>() : rdt_ready<RdParams>());
    int grid;
    if (bulk) {  // the bulk kernel's work items: whole rows or row segments of one stage
      items = 0;
      for (int i = 0; i < nt; ++i) {
        bulk_partition(&p.task[i], p.esize);
        p.task[i].item_begin = items;
        items += bulk_items(p.task[i]);
      }
      // one CTA (four pipelines) per SM
      grid = (int)std::min<int64_t>((items + RDT_PIPES - 1) / RDT_PIPES, (int64_t)sms);
    } else {
      // one wave of resident CTAs, grid-stride over items
      const int64_t blocks = (items + RD_WARPS - 1) / RD_WARPS;
      grid = (int)std::min<int64_t>(blocks, (int64_t)sms * (sum ? RD_SUM_CTAS : RD_COPY_CTAS));
    }
    p.ntasks = nt;
    p.nitems = items;
    p.status = status;
    p.wait_limit_ns = rd_wait_limit_ns();
    p.starve = rd_starve();
    if (grid > 0) {
      if (small) {
        std::copy(p.dst, p.dst + nd_slots, ps.dst);
        std::copy(p.src, p.src + ns_slots, ps.src);
        std::copy(p.task, p.task + nt, ps.task);
        std::copy(p.ref, p.ref + nref, ps.ref);
        ps.nitems = p.nitems;
        ps.ntasks = p.ntasks;
        ps.dtype = p.dtype;
        ps.esize = p.esize;
        ps.op = p.op;
        ps.status = p.status;
        ps.wait_limit_ns = p.wait_limit_ns;
        ps.starve = p.starve;
        launch_rd(ps, kind, bulk, grid, stream);
        if (g_recording) {
          const uint8_t* b = reinterpret_cast<const uint8_t*>(&ps);
          g_recording->launches.push_back({kind, true, bulk, grid, std::vector<uint8_t>(b, b + sizeof(ps))});
        }
      } else {
        launch_rd(p, kind, bulk, grid, stream);
        if (g_recording) {
          const uint8_t* b = reinterpret_cast<const uint8_t*>(&p);
          g_recording->launches.push_back({kind, false, bulk, grid, std::vector<uint8_t>(b, b + sizeof(p))});
        }
      }
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return fail(DT_ERR_CUDA, "redistribute launch: %s", cudaGetErrorString(e));
      count_launch();
    }
    nd_slots = ns_slots = nt = nref = 0;
    items = 0;
    aligned = kind == RD_COPY && bulk_copies() == 1;
    return DT_OK;
  };
  dt_status st;
  // pairs of one dtype and reduce op share launches: visit them grouped
  std::vector<int> order(plans.size());
  for (size_t i = 0; i < plans.size(); ++i) order[i] = (int)i;
  auto key = [&](int i) { return plans[i].S.layout.dtype * 8 + (sum ? plans[i].S.layout.partial_op() : 0); };
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return key(a) < key(b); });
  for (int pi : order) {
    PairPlan& pp = plans[pi];
    const std::vector<HostTask>& tasks = kind == RD_SUM ? pp.sums : kind == RD_COPY ? pp.copies : pp.repl;
    if (tasks.empty()) continue;
    const Layout& ls = pp.S.layout;
    const int nd = ls.ndim;
    const int pad = 4 - nd;
    const int op = sum ? ls.partial_op() : DT_SUM;
    if (nt > 0 && (p.dtype != ls.dtype || p.op != op))
      if ((st = flush()) != DT_OK) return st;
    p.dtype = ls.dtype;
    p.esize = ls.esize;
    p.op = op;
    int dbase = -1, sbase = -1;
    for (const HostTask& ht : tasks) {
      const bool need_slots = dbase < 0;
      const int task_refs = (int)(ht.src_slots.size() + ht.extra_dst.size());
      const bool fits = nt < RD_MAX_TASKS && nref + task_refs <= RD_MAX_REFS &&
                        (!need_slots || (nd_slots + pp.D.layout.nslots <= RD_MAX_LAUNCH_SLOTS &&
                                         ns_slots + ls.nslots <= RD_MAX_LAUNCH_SLOTS));
      if (!fits) {
        if ((st = flush()) != DT_OK) return st;
        dbase = sbase = -1;
      }
      if (dbase < 0) {
        dbase = nd_slots;
        sbase = ns_slots;
        for (int s = 0; s < pp.D.layout.nslots; ++s) fill_slot(&p.dst[nd_slots++], pp.D.slots[s], nd);
        for (int s = 0; s < ls.nslots; ++s) fill_slot(&p.src[ns_slots++], pp.S.slots[s], nd);
      }
      RdTask& t = p.task[nt];
      merge_dims(ht, pp.D, pp.S, pad, &t);
      t.dst_slot = (int16_t)(dbase + ht.dst_slot);
      t.dst_off = local_offset(pp.D.slots[ht.dst_slot], ht.box, nd);
      t.nsrc = (int16_t)ht.src_slots.size();
      t.ref_begin = (int16_t)nref;
      for (int k = 0; k < t.nsrc; ++k) {
        p.ref[nref].slot = sbase + ht.src_slots[k];
        p.ref[nref].off = local_offset(pp.S.slots[ht.src_slots[k]], ht.box, nd);
        ++nref;
      }
      t.nextra = (int8_t)ht.extra_dst.size();
      t.extra16 = 1;
      const uintptr_t first = reinterpret_cast<uintptr_t>(pp.D.slots[ht.dst_slot].ptr) + (uintptr_t)(t.dst_off * ls.esize);
      for (int x : ht.extra_dst) {  // replica x: byte distance from the first destination
        const uintptr_t at =
            reinterpret_cast<uintptr_t>(pp.D.slots[x].ptr) + (uintptr_t)(local_offset(pp.D.slots[x], ht.box, nd) * ls.esize);
        p.ref[nref].slot = dbase + x;
        p.ref[nref].off = static_cast<int64_t>(at - first);
        if (p.ref[nref].off % 16 != 0) t.extra16 = 0;
        ++nref;
      }
      // segments are whole 16-byte multiples so every segment of a row
      // keeps the row's alignment
      const int64_t seg_bytes = sum ? SUM_SEG_BYTES : COPY_SEG_BYTES;
      t.seg_elems = (int32_t)(seg_bytes / ls.esize);
      const int64_t spr = std::max<int64_t>(1, (t.ext[3] + t.seg_elems - 1) / t.seg_elems);
      if (spr > (1ll << 30)) return fail(DT_ERR_CAPACITY, "row of %lld elements", (long long)t.ext[3]);
      t.segs_per_row = (int32_t)spr;
      t.item_begin = items;
      t.rows_per_item = 1;
      items += t.ext[0] * t.ext[1] * t.ext[2] * spr;
      if (aligned)
        aligned = t.nsrc == 1 && bulk_task_ok(t, p.dst[t.dst_slot], p.src[p.ref[t.ref_begin].slot],
                                              p.ref[t.ref_begin].off, ls.esize);
      ++nt;
    }
  }
  return flush();
}

// The copies and the Partial reductions of one call are independent (no
// output overlaps an input), so the reductions run on an auxiliary stream
// forked from the caller's and joined back before the call returns: one
// launch's ramp and tail overlap the other's.  One auxiliary stream and
// event pair per device, made on first use and kept; the mutex keeps
// concurrent callers' fork/join pairs apart.
struct AuxStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool failed = false;
};
std::mutex g_aux_mu;
AuxStream g_aux[64];

template <class Launch>  // Launch: dt_status(int kind, cudaStream_t)
dt_status launch_forked(Launch&& launch, cudaStream_t s) {
  int dev = 0;
  cudaGetDevice(&dev);
  std::unique_lock<std::mutex> lk(g_aux_mu);
  AuxStream* a = (dev >= 0 && dev < 64) ? &g_aux[dev] : nullptr;
  if (a && !a->s && !a->failed) {
    if (cudaStreamCreateWithFlags(&a->s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&a->fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&a->join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      a->failed = true;
    }
  }
  dt_status st;
  if (!a || a->failed || cudaEventRecord(a->fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(a->s, a->fork, 0) != cudaSuccess) {
    cudaGetLastError();
    lk.unlock();
    for (int k : {RD_COPY, RD_COPY_REPL, RD_SUM})  // one stream, one after the other
      if ((st = launch(k, s)) != DT_OK) return st;
    return DT_OK;
  }
  st = launch(RD_SUM, a->s);
  if (st == DT_OK) st = launch(RD_COPY, s);
  if (st == DT_OK) st = launch(RD_COPY_REPL, s);
  // join even after a failed launch, so the caller's stream never runs ahead of the auxiliary one
  cudaError_t e = cudaEventRecord(a->join, a->s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, a->join, 0);
  if (e != cudaSuccess && st == DT_OK) st = fail(DT_ERR_CUDA, "redistribute join: %s", cudaGetErrorString(e));
  return st;
}

dt_status redistribute_planned(int32_t n, const dt_dtensor* src, const dt_dtensor* dst, int32_t* status,
                               cudaStream_t s, RecordedPlan* rec);

template <class P>
dt_status replay_one(const RecordedLaunch& r, cudaStream_t s) {
  launch_rd(*reinterpret_cast<const P*>(r.params.data()), r.kind, r.bulk, r.grid, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(DT_ERR_CUDA, "redistribute launch: %s", cudaGetErrorString(e));
  count_launch();
  return DT_OK;
}

dt_status replay_kind(const RecordedPlan& rp, int kind, cudaStream_t s) {
  for (const RecordedLaunch& r : rp.launches) {
    if (r.kind != kind) continue;
    dt_status st = r.small ? replay_one<RdParamsSmall>(r, s) : replay_one<RdParams>(r, s);
    if (st != DT_OK) return st;
  }
  return DT_OK;
}

// Plans by operands: the bytes of every pair's layouts, slot pointers and
// strides decide the launches completely (never the data), so equal keys
// replay equal launches.  Bounded; dropped whole when full.
std::mutex g_plan_mu;
std::unordered_map<std::string, std::shared_ptr<const RecordedPlan>> g_plans;
constexpr size_t RD_PLAN_CACHE = 128;

dt_status replay(const RecordedPlan& rp, cudaStream_t s) {
  auto launch = [&](int kind, cudaStream_t st) { return replay_kind(rp, kind, st); };
  if (rp.forked) return launch_forked(launch, s);
  dt_status st;
  for (int k : {RD_COPY, RD_COPY_REPL, RD_SUM})
    if ((st = launch(k, s)) != DT_OK) return st;
  return DT_OK;
}

dt_status redistribute_many(int32_t n, const dt_dtensor* src, const dt_dtensor* dst, int32_t* d_status,
                            dt_stream_t stream) {
  clear_error();
  if (n < 0 || (n > 0 && (!src || !dst))) return fail(DT_ERR_INVALID_ARG, "need n >= 0 and src/dst arrays");
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  std::string key;
  bool keyed = true;
  for (int i = 0; i < n && keyed; ++i) keyed = append_plan_key(&key, &src[i]) && append_plan_key(&key, &dst[i]);
  append_plan_scalar(&key, d_status);  // the recorded parameters hold the status word
  if (keyed && n > 0) {
    std::shared_ptr<const RecordedPlan> hit;
    {
      std::lock_guard<std::mutex> lk(g_plan_mu);
      auto it = g_plans.find(key);
      if (it != g_plans.end()) hit = it->second;
    }
    if (hit) {
      if (hit->launches.empty()) return DT_OK;
      // the device of the first destination slot with data, as when planned
      const void* any = nullptr;
      for (int i = 0; i < n && !any; ++i)
        for (int sl = 0; sl < dst[i].nslots && !any; ++sl)
          if (dst[i].slots[sl]) any = dst[i].slots[sl];
      dt_status st = bind_device_of(any);
      if (st != DT_OK) return st;
      return replay(*hit, cs);
    }
  }
  auto rec = std::make_shared<RecordedPlan>();
  dt_status st = redistribute_planned(n, src, dst, d_status, cs, rec.get());
  if (st == DT_OK && keyed && n > 0) {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    if (g_plans.size() >= RD_PLAN_CACHE) g_plans.clear();
    g_plans[key] = rec;
  }
  return st;
}

dt_status redistribute_planned(int32_t n, const dt_dtensor* src, const dt_dtensor* dst, int32_t* d_status,
                               cudaStream_t s, RecordedPlan* rec) {
  std::vector<PairPlan> plans(n);
  const void* any = nullptr;
  dt_status st;
  for (int i = 0; i < n; ++i) {
    if ((st = plan_pair(&src[i], &dst[i], &plans[i])) != DT_OK) {
      if (n == 1) return st;
      std::string inner = dt_last_error();
      return fail(st, "pair %d: %s", i, inner.c_str());
    }
    for (auto& v : plans[i].D.slots)
      if (!any && v.numel) any = v.ptr;
  }
  if (!any) return DT_OK;
  if ((st = bind_device_of(any)) != DT_OK) return st;
  bool copies = false, sums = false;
  for (const PairPlan& pp : plans) {
    copies = copies || !pp.copies.empty() || !pp.repl.empty();
    sums = sums || !pp.sums.empty();
  }
  struct Recording {  // record the launches this call makes (and stop on return)
    explicit Recording(RecordedPlan* r) { g_recording = r; }
    ~Recording() { g_recording = nullptr; }
  } recording(rec);
  rec->forked = copies && sums;
  int32_t* status = device_status_word(d_status);
  if (!status) return fail(DT_ERR_CUDA, "no device status word");
  auto launch = [&](int kind, cudaStream_t stream) { return launch_kind(plans, kind, status, stream); };
  if (rec->forked) return launch_forked(launch, s);
  for (int k : {RD_COPY, RD_COPY_REPL, RD_SUM})
    if ((st = launch(k, s)) != DT_OK) return st;
  return DT_OK;
}

}  // namespace

void clear_redistribute_plans() {
  std::lock_guard<std::mutex> lk(g_plan_mu);
  g_plans.clear();
}

}  // namespace dt

extern "C" dt_status dt_redistribute(const dt_dtensor* src, const dt_dtensor* dst, int32_t* d_status,
                                     dt_stream_t stream) {
  return dt::redistribute_many(1, src, dst, d_status, stream);
}

extern "C" dt_status dt_redistribute_batch(int32_t n, const dt_dtensor* src, const dt_dtensor* dst,
                                           int32_t* d_status, dt_stream_t stream) {
  return dt::redistribute_many(n, src, dst, d_status, stream);
}
