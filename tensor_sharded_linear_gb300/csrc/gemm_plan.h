// Host-side description of one batched GEMM call: independent output groups,
// each summing a list of (A, B) K segments in order.  Built by the linear
// entry points, lowered either to the tcgen05 kernel or to the CUDA-core
// kernel.
#pragma once

#include <cuda_runtime.h>

#include <memory>
#include <vector>

#include "dt_internal.h"

namespace dt {
namespace gemm {

// Matrix view of rows x cols.  Row-major: element (r, c) at
// ptr + (r * ld + c) * esize.  kmajor (weights only, rows = K): element
// (k, n) at ptr + (n * ld + k) * esize -- the [out, in] storage of a weight,
// passed as a transposed view.
struct Mat {
  char* ptr = nullptr;
  int64_t rows = 0, cols = 0, ld = 0;
  int dtype = DT_BF16;
  bool kmajor = false;
};

struct HostSeg {
  Mat a;   // [M, K_s]
  Mat b;   // [K_s, N]
  Mat b2;  // [K_s, N], gated MLP "up" operand (dual groups only)
};

struct HostGroup {
  int64_t m = 0, n = 0;
  std::vector<HostSeg> segs;
  bool dual = false;  // out = SiLU(A B) * (A B2)
  int out_dtype = DT_BF16;
  // rows [row_begin[j], row_begin[j+1]) go to out_ptr[j] with leading dim out_ld[j]
  std::vector<int64_t> row_begin;
  std::vector<char*> out_ptr;
  std::vector<int64_t> out_ld;
  const void* bias = nullptr;  // [n], added before the cast
  int bias_dtype = -1;
  // row block of x the group reads, when x is split by rows into several
  // slots (token shards); groups come ordered by it
  int m_block = 0;
};

// Caller-owned device memory a call may use for the split tail's scratch
// (256-byte aligned; null or too small: every tile runs whole).
struct Workspace {
  char* ptr = nullptr;
  size_t bytes = 0;
};

// Run every group; returns a host-detected error or DT_OK.  Launches run one
// after another on `stream`, so they share the workspace.
dt_status run_groups(std::vector<HostGroup>& groups, int32_t* d_status, cudaStream_t stream, Workspace ws);

// Workspace bytes with which run_groups on the current device splits every
// launch's last wave that it would split (0 when none would).
dt_status workspace_bytes(std::vector<HostGroup>& groups, size_t* bytes);

// CUDA-core GEMM launches so far (operands TMA cannot describe, or fp32).
uint64_t cuda_core_launches();

// Capacities of one launch's parameter block (the device code's ParamsT).
constexpr int MAX_MAPS = 48;
constexpr int MAX_SEGS = 96;
constexpr int MAX_GROUPS = 64;
template <int NMAPS, int NSEGS, int NGROUPS>
struct ParamsT;
using Params = ParamsT<MAX_MAPS, MAX_SEGS, MAX_GROUPS>;
cudaError_t launch_tcgen05_pair(const Params& p, int clusters, cudaStream_t stream);
int pair_max_clusters();  // co-resident clusters of the pair kernel (0: unavailable)

// The launches one call made, recorded as issued so a later call with the
// same operands replays them without planning.
struct GemmRecord;
struct GemmRecordScope {  // while alive, run_groups on this thread records into r
  explicit GemmRecordScope(GemmRecord* r);
  ~GemmRecordScope();
};
std::shared_ptr<GemmRecord> new_gemm_record();
dt_status replay_gemm(const GemmRecord& r, cudaStream_t stream);

}  // namespace gemm
}  // namespace dt
