// Allreduce fused with RMSNorm: launch arguments and limits.
#pragma once

#include "internal.h"

namespace tccl {

constexpr int kRmsMaxThreads = 256;
constexpr int kRmsClusterThreads = 256;  // cluster path: threads per CTA (4 vectors each)
constexpr int kRmsCluster = 8;           // cluster path: CTAs sharing a row
constexpr int kRmsMaxVectors = 8;  // 16-byte vectors of a row per thread

struct RmsArgs {
  BasePtrs<kMaxRanks> p;
  const void* gamma;  // hidden elements, the output type
  uint32_t* sm_mask;
  uint64_t rows;
  uint32_t hidden;
  float eps;
  int nranks;
  // rmsnorm_kernel with more rows than CTAs: two words, zero between
  // launches, the next-row counter and the count of finished CTAs; null:
  // each CTA takes every gridDim-th row
  unsigned long long* claim;
};

// `vectors`: 16-byte vectors of a row per thread (4 or 8); gamma is staged in
// hidden * element-size bytes of dynamic shared memory.
// early: programmatic dependent launch (uncapped calls only)
int launch_rmsnorm(int dtype, const RmsArgs& a, int grid, int threads, int vectors, bool early,
                   void* stream);
// CTAs of launch_rmsnorm's kernel resident on one SM with this shape (0 if
// the occupancy query fails)
int rmsnorm_ctas_per_sm(int dtype, int threads, int vectors, size_t smem);
// Few rows: `clusters` clusters of `cluster_size` CTAs, each cluster one row at a time.
int launch_rmsnorm_cluster(int dtype, const RmsArgs& a, int clusters, int cluster_size,
                           bool early, void* stream);

}  // namespace tccl
